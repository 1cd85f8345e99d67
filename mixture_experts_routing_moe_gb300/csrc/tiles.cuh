// Ragged per-expert tiling shared by the expert GEMM kernels.
//
// Expert e owns dispatched rows offsets[e] .. offsets[e+1]-1; with BM-row tiles it has
// mt_e = ceil(n_e / BM) m-tiles.  pref[e] = sum_{e' < e} mt_e' (pref[E] = total m-tiles) is
// built in shared memory from the device-side offsets, so no host round trip is needed.
#pragma once

#include <stdint.h>

namespace moe {

// One warp fills pref[0..E] with the exclusive prefix of count(n_e), n_e = rows of expert e.
template <class Count>
__device__ inline void build_expert_prefix(const int32_t* __restrict__ offsets, int E, Count count,
                                           int* pref, int lane) {
  int carry = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    const int v = e < E ? count(offsets[e + 1] - offsets[e]) : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (e < E) pref[e] = carry + x - v;
    carry += __shfl_sync(0xFFFFFFFFu, x, 31);
  }
  if (lane == 0) pref[E] = carry;
}

// m-tiles: count(n) = ceil(n / BM).  E <= 1024.
__device__ inline void build_mtile_prefix(const int32_t* __restrict__ offsets, int E, int BM,
                                          int* pref, int lane) {
  build_expert_prefix(offsets, E, [BM](int n) { return (n + BM - 1) / BM; }, pref, lane);
}

// The expert owning tile j (0 <= j < pref[E]): the largest e < E with pref[e] <= j.
__device__ inline int find_expert(const int* pref, int E, int j) {
  int lo = 0, hi = E;  // invariant: pref[lo] <= j < pref[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= j) lo = mid;
    else hi = mid;
  }
  return lo;
}

}  // namespace moe
