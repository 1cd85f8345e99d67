// Route kernel: route(logits, RoutingOptions) of the ruDNN user guide, §4 "Routing-Vertrag".
//
// One row of logits is owned by L consecutive lanes of a warp (L = 1..32); lane i of the group
// holds the contiguous elements [i*C, i*C + C) of the row, read with 16-byte loads when the row
// pitch allows.  The softmax runs in FP32 over all E experts (max and sum reduced with xor
// shuffles inside the group).  The top-k is k rounds of a group argmax over 64-bit keys
//     key = monotone_bits(logit) << 32 | (0xFFFFFFFF - id)
// so a larger key is a larger logit, and equal logits prefer the lower id; the winner of each
// round is removed by its owner.  Selected ids and their exp(l - max) are staged in shared memory
// and written out coalesced.  Rows holding a NaN or +inf, or only -inf, get NaN weights and ids
// 0..k-1.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t monotone_bits(float v) {
  uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_monotone_bits(uint32_t m) {
  uint32_t u = (m & 0x80000000u) ? (m & 0x7FFFFFFFu) : ~m;
  return __uint_as_float(u);
}

template <int L, typename V>
__device__ __forceinline__ V group_max(V v) {
#pragma unroll
  for (int o = L / 2; o > 0; o >>= 1) {
    V w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  return v;
}
template <int L>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = L / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
template <int L>
__device__ __forceinline__ uint32_t group_or(uint32_t v) {
#pragma unroll
  for (int o = L / 2; o > 0; o >>= 1) v |= __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

constexpr int kRouteWarps = 8;

template <typename T, int L, int C, bool VEC>
__global__ void __launch_bounds__(kRouteWarps * 32)
    moe_route_kernel(const T* __restrict__ logits, int64_t T_, int E, int k, int renorm,
                     uint32_t* __restrict__ idx_out, T* __restrict__ w_out) {
  extern __shared__ uint8_t route_smem[];
  constexpr int RPW = 32 / L;  // rows per warp
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane / L, gl = lane % L;  // row group inside the warp, lane inside the group
  const int row_local = warp * RPW + g;
  const int64_t row = (int64_t)blockIdx.x * (kRouteWarps * RPW) + row_local;
  const bool row_ok = row < T_;
  uint32_t* s_id = reinterpret_cast<uint32_t*>(route_smem) + (size_t)row_local * k;
  float* s_e = reinterpret_cast<float*>(route_smem + (size_t)kRouteWarps * RPW * k * 4) +
               (size_t)row_local * k;

  float v[C];
  const int e0 = gl * C;
  const T* src = logits + (row_ok ? row : 0) * (int64_t)E;
  if (VEC) {
    constexpr int VW = 16 / sizeof(T);
#pragma unroll
    for (int c = 0; c < C / VW; ++c) {
      Vec16<T> q;
      if (row_ok && e0 + c * VW < E) q.u = ld_nc_v4(src + e0 + c * VW);
      else q.u = make_uint4(0, 0, 0, 0);
      q.to_float(v + c * VW);
    }
  } else {
#pragma unroll
    for (int c = 0; c < C; ++c) v[c] = (row_ok && e0 + c < E) ? Dt<T>::to_f(src[e0 + c]) : 0.f;
  }

  // poison flags: bit0 = NaN or +inf seen, bit1 = a value other than -inf seen
  uint32_t flags = 0;
  float m = -INFINITY;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    if (e0 + c < E) {
      const float x = v[c];
      if (x != x || x == INFINITY) flags |= 1u;
      if (x != -INFINITY) flags |= 2u;
      m = fmaxf(m, x);
    }
  }
  flags = group_or<L>(flags);
  m = group_max<L>(m);
  const bool poisoned = (flags & 1u) || !(flags & 2u);

  // Every lane runs the whole selection (shuffles need the full warp); poisoned rows and rows
  // past T compute throw-away values and are written differently below.
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < C; ++c)
    if (e0 + c < E) s += __expf(v[c] - m);
  s = group_sum<L>(s);

  uint64_t key[C];
#pragma unroll
  for (int c = 0; c < C; ++c)
    key[c] = (e0 + c < E)
                 ? ((uint64_t)monotone_bits(v[c]) << 32) | (0xFFFFFFFFu - (uint32_t)(e0 + c))
                 : 0ull;
  float sel = 0.f;
  for (int r = 0; r < k; ++r) {
    uint64_t best = key[0];
#pragma unroll
    for (int c = 1; c < C; ++c) best = key[c] > best ? key[c] : best;
    best = group_max<L>(best);
    const uint32_t id = 0xFFFFFFFFu - (uint32_t)best;
    const float ex = __expf(from_monotone_bits((uint32_t)(best >> 32)) - m);
    sel += ex;
#pragma unroll
    for (int c = 0; c < C; ++c)
      if (key[c] == best) key[c] = 0ull;
    if (gl == 0) {
      s_id[r] = id;
      s_e[r] = ex;
    }
  }
  __syncwarp();
  if (row_ok) {
    const float denom = renorm ? sel : s;
    for (int j = gl; j < k; j += L) {
      if (poisoned) {
        idx_out[row * k + j] = (uint32_t)j;
        w_out[row * k + j] = Dt<T>::from_f(__int_as_float(0x7FC00000));
      } else {
        idx_out[row * k + j] = s_id[j];
        w_out[row * k + j] = Dt<T>::from_f(s_e[j] / denom);
      }
    }
  }
}

template <typename T, int L, int C>
cudaError_t launch_route_lc(const void* logits, int64_t T_, int E, int k, int renorm,
                            uint32_t* idx, void* w, cudaStream_t s) {
  constexpr int RPB = kRouteWarps * (32 / L);
  const size_t smem = (size_t)RPB * k * 8;
  const int64_t blocks = (T_ + RPB - 1) / RPB;
  const bool vec = (((uintptr_t)logits) % 16 == 0) && ((E * sizeof(T)) % 16 == 0);
  if (smem > 48 * 1024) {
    cudaError_t err;
    err = cudaFuncSetAttribute(moe_route_kernel<T, L, C, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(moe_route_kernel<T, L, C, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  if (vec)
    moe_route_kernel<T, L, C, true><<<(unsigned)blocks, kRouteWarps * 32, smem, s>>>(
        (const T*)logits, T_, E, k, renorm, idx, (T*)w);
  else
    moe_route_kernel<T, L, C, false><<<(unsigned)blocks, kRouteWarps * 32, smem, s>>>(
        (const T*)logits, T_, E, k, renorm, idx, (T*)w);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_route_t(const void* logits, int64_t T_, int E, int k, int renorm, uint32_t* idx,
                           void* w, cudaStream_t s) {
  constexpr int VW = 16 / sizeof(T);
  // choose lanes-per-row L and elements-per-lane C (a multiple of the vector width) with L*C >= E
  if (E <= 1 * VW) return launch_route_lc<T, 1, VW>(logits, T_, E, k, renorm, idx, w, s);
  if (E <= 2 * VW) return launch_route_lc<T, 2, VW>(logits, T_, E, k, renorm, idx, w, s);
  if (E <= 4 * VW) return launch_route_lc<T, 4, VW>(logits, T_, E, k, renorm, idx, w, s);
  if (E <= 8 * VW) return launch_route_lc<T, 8, VW>(logits, T_, E, k, renorm, idx, w, s);
  if (E <= 16 * VW) return launch_route_lc<T, 16, VW>(logits, T_, E, k, renorm, idx, w, s);
  if (E <= 32 * VW) return launch_route_lc<T, 32, VW>(logits, T_, E, k, renorm, idx, w, s);
  if (E <= 64 * VW) return launch_route_lc<T, 32, 2 * VW>(logits, T_, E, k, renorm, idx, w, s);
  if (E <= 128 * VW) return launch_route_lc<T, 32, 4 * VW>(logits, T_, E, k, renorm, idx, w, s);
  if (E <= 256 * VW) return launch_route_lc<T, 32, 8 * VW>(logits, T_, E, k, renorm, idx, w, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_route(const void* logits, int ldt, int64_t T_, int E, int k, int renorm,
                         uint32_t* idx, void* w, cudaStream_t s) {
  switch (ldt) {
    case MOE_F32: return launch_route_t<float>(logits, T_, E, k, renorm, idx, w, s);
    case MOE_F16: return launch_route_t<__half>(logits, T_, E, k, renorm, idx, w, s);
    case MOE_BF16: return launch_route_t<__nv_bfloat16>(logits, T_, E, k, renorm, idx, w, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
