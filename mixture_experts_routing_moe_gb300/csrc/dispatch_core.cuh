// Dispatch of a short batch by one block (ruDNN user guide, §5 "Expertengewichte und
// Verteilung"): count, scan and stable scatter of R <= a few thousand slots with the histograms in
// shared memory.  Warp w of `nwarps` owns the contiguous slot chunk [w*CH, w*CH + CH) (CH a
// multiple of 32, nwarps * CH >= R); inside a chunk, lanes with the same expert are merged and
// ranked with match.any.  Rows of expert e keep ascending slot order s = t*k + j, whatever nwarps
// is.  Shared by the dispatch kernel for short batches and the fused decode kernel.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace moe {

// hist: shared [nwarps * E]; off: shared [E + 1], left holding the offsets.  offsets_out and
// row_of_slot may be null (not written); token_of_row may point to shared or global memory.
// COHERENT reads idx through L2 only (it was written earlier in the same launch).  Expert ids
// >= E are not dispatched: their row_of_slot is kInvalidRow and the status word gets the index bit.
template <bool COHERENT>
__device__ __forceinline__ void dispatch_block(const uint32_t* __restrict__ idx, int64_t R, int E,
                                               int k, int nwarps, int CH, int32_t* hist,
                                               int32_t* off, int32_t* offsets_out,
                                               uint32_t* token_of_row, uint32_t* row_of_slot,
                                               unsigned* status) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < nwarps * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t s0 = (int64_t)warp * CH, s1 = (R < s0 + CH) ? R : s0 + CH;
  int32_t* h = hist + warp * E;
  bool bad = false;
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t s = base + lane;
    const bool act = s < s1;
    const uint32_t e = act ? ld_elem<COHERENT>(idx + s) : 0xFFFFFFFFu;
    const bool valid = act && e < (uint32_t)E;
    bad |= act && !valid;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : 0xFFFFFFFFu);
    if (valid && lane == __ffs(peers) - 1) h[e] += __popc(peers);
    __syncwarp();
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && status) atomicOr(status, kStatusIndex);
  __syncthreads();
  // per expert: exclusive prefix over the chunks, and the expert's total
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int32_t c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    off[e] = run;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the totals -> offsets
    int32_t carry = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int32_t c = e < E ? off[e] : 0;
      int32_t x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      if (e < E) {
        off[e] = carry + x - c;
        if (offsets_out) offsets_out[e] = carry + x - c;
      }
      carry += __shfl_sync(0xFFFFFFFFu, x, 31);
    }
    if (lane == 0) {
      off[E] = carry;
      if (offsets_out) offsets_out[E] = carry;
    }
  }
  __syncthreads();
  if (warp < nwarps) {
    for (int e = lane; e < E; e += 32) h[e] += off[e];  // running row of each expert in this chunk
  }
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t s = base + lane;
    const bool act = s < s1;
    const uint32_t e = act ? ld_elem<COHERENT>(idx + s) : 0xFFFFFFFFu;
    const bool valid = act && e < (uint32_t)E;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : 0xFFFFFFFFu);
    if (valid) {
      const uint32_t row = (uint32_t)(h[e] + __popc(peers & lt));
      if (row_of_slot) row_of_slot[s] = row;
      token_of_row[row] = (uint32_t)(s / k);
    } else if (act && row_of_slot) {
      row_of_slot[s] = kInvalidRow;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) h[e] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace moe
