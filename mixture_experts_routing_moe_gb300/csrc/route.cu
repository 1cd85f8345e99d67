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
#include "route_core.cuh"

namespace moe {
namespace {

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
  uint32_t* s_id = reinterpret_cast<uint32_t*>(route_smem) + (size_t)row_local * k;
  float* s_e = reinterpret_cast<float*>(route_smem + (size_t)kRouteWarps * RPW * k * 4) +
               (size_t)row_local * k;
  route_row<T, L, C, VEC>(logits, row, row < T_, E, k, renorm, gl, s_id, s_e, idx_out, w_out);
}

// ------------------------------------------------------------------------------------------
// Fast path for 16-bit logits with E <= 64 (E % 8 == 0, 16-byte aligned rows) and top_k <= 8:
// one row per thread.  Keys are 32-bit: monotone 16-bit value bits << 16 | (0xFFFF - id), so a
// larger key is a larger logit and equal logits prefer the lower id.  Each 16-byte vector (8
// experts) is sorted by an 8-input sorting network and merged into the running sorted top 8 with
// a bitonic merge (elementwise max against the reversed list, then a half-cleaner).  The softmax
// denominator is accumulated online over the vectors (rescaled when the running max grows);
// with renormalisation only the selected experts' exponentials are needed.
__device__ __forceinline__ void ce_desc(uint32_t& a, uint32_t& b) {
  const uint32_t hi = max(a, b), lo = min(a, b);
  a = hi;
  b = lo;
}
__device__ __forceinline__ void sort8_desc(uint32_t (&k)[8]) {
  ce_desc(k[0], k[1]); ce_desc(k[2], k[3]); ce_desc(k[4], k[5]); ce_desc(k[6], k[7]);
  ce_desc(k[0], k[2]); ce_desc(k[1], k[3]); ce_desc(k[4], k[6]); ce_desc(k[5], k[7]);
  ce_desc(k[1], k[2]); ce_desc(k[5], k[6]);
  ce_desc(k[0], k[4]); ce_desc(k[1], k[5]); ce_desc(k[2], k[6]); ce_desc(k[3], k[7]);
  ce_desc(k[2], k[4]); ce_desc(k[3], k[5]);
  ce_desc(k[1], k[2]); ce_desc(k[3], k[4]); ce_desc(k[5], k[6]);
}
// top: sorted descending; g: sorted descending.  Leaves the 8 largest of both in `top`, sorted.
__device__ __forceinline__ void merge_top8(uint32_t (&top)[8], const uint32_t (&g)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) top[i] = max(top[i], g[7 - i]);  // bitonic, holds the top 8
  ce_desc(top[0], top[4]); ce_desc(top[1], top[5]); ce_desc(top[2], top[6]); ce_desc(top[3], top[7]);
  ce_desc(top[0], top[2]); ce_desc(top[1], top[3]); ce_desc(top[4], top[6]); ce_desc(top[5], top[7]);
  ce_desc(top[0], top[1]); ce_desc(top[2], top[3]); ce_desc(top[4], top[5]); ce_desc(top[6], top[7]);
}
template <typename T>
__device__ __forceinline__ float bits16_to_float(uint32_t b) {
  if constexpr (sizeof(T) == 2 && Dt<T>::code == MOE_BF16) {
    return __uint_as_float(b << 16);
  } else {
    return __half2float(__ushort_as_half((unsigned short)b));
  }
}

template <typename T, int NV, bool RENORM>
__global__ void __launch_bounds__(256)
    moe_route16_small(const uint4* __restrict__ logits, int64_t T_, int k,
                      uint32_t* __restrict__ idx_out, T* __restrict__ w_out) {
  constexpr uint32_t EXPMASK = Dt<T>::code == MOE_BF16 ? 0x7F80u : 0x7C00u;
  const int64_t row0 = (int64_t)blockIdx.x * 256;
  const int64_t row = row0 + threadIdx.x;
  // E = 64: the block's 256 rows (32 KB, contiguous) are read with coalesced 16-byte loads into
  // shared memory, vector v of row r stored at slot v ^ (r & 7) so that the row-per-thread reads
  // below hit 8 different bank groups per 8 lanes.
  constexpr bool STAGED = NV == 8;
  __shared__ uint4 tile[STAGED ? 256 * 8 : 1];
  if (STAGED) {
    const int64_t left = T_ - row0;
    const int n = (int)((left < 256 ? left : 256) * 8);
    const uint4* bsrc = logits + row0 * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = threadIdx.x + i * 256;
      if (c < n) tile[(c & ~7) | ((c & 7) ^ ((c >> 3) & 7))] = ld_nc_v4(bsrc + c);
    }
    __syncthreads();
  }
  if (row >= T_) return;
  const uint4* src = logits + row * NV;
  uint32_t top[8];
  uint32_t rawmax = 0u;  // per-half unsigned max of the raw bits: above -inf only for a negative NaN
  float m = -INFINITY, s = 0.f;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const uint4 q = STAGED ? tile[threadIdx.x * 8 + (v ^ (threadIdx.x & 7))] : ld_nc_v4(src + v);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t g[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // monotone map of both 16-bit halves: negative -> all bits flipped, else sign bit set.
      // prmt with selector 0xBB99 replicates each half's sign bit over the half (0xFFFF / 0).
      uint32_t sm;
      asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(sm) : "r"(w[i]));
      const uint32_t t = w[i] ^ (sm | 0x80008000u);
      rawmax = __vmaxu2(rawmax, w[i]);
      const uint32_t e0 = v * 8 + i * 2;
      g[2 * i] = (t << 16) | (0xFFFFu - e0);
      g[2 * i + 1] = (t & 0xFFFF0000u) | (0xFFFFu - (e0 + 1));
    }
    if (!RENORM) {  // online softmax denominator
      float x[8], gm = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = bits16_to_float<T>(w[i] & 0xFFFFu);
        x[2 * i + 1] = bits16_to_float<T>(w[i] >> 16);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) gm = fmaxf(gm, x[i]);
      const float mn = fmaxf(m, gm);
      const float ref = mn == -INFINITY ? 0.f : mn;  // all -inf so far: every term is 0
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc += __expf(x[i] - ref);
      s = (m == -INFINITY ? 0.f : s * __expf(m - mn)) + acc;
      m = mn;
    }
    sort8_desc(g);
    if (v == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) top[i] = g[i];
    } else {
      merge_top8(top, g);
    }
  }
  // poisoned: largest value NaN / +inf / -inf (the last means every value is -inf), or a
  // negative NaN anywhere (its raw bits exceed those of -inf)
  const uint32_t tb = top[0] >> 16;
  const uint32_t vb0 = (tb & 0x8000u) ? (tb & 0x7FFFu) : (~tb & 0xFFFFu);
  const uint32_t rmax = max(rawmax & 0xFFFFu, rawmax >> 16);  // negative NaN: above 0x8000|EXPMASK
  const bool poisoned = (vb0 & 0x7FFFu) >= EXPMASK || rmax > (0x8000u | EXPMASK);
  const float x0 = bits16_to_float<T>(vb0);
  float ex[8], sel = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t b = top[j] >> 16;
    const uint32_t vb = (b & 0x8000u) ? (b & 0x7FFFu) : (~b & 0xFFFFu);
    ex[j] = __expf(bits16_to_float<T>(vb) - x0);
    if (j < k) sel += ex[j];
  }
  const float denom = RENORM ? sel : s * __expf(m - x0);
  uint32_t* io = idx_out + row * k;
  T* wo = w_out + row * k;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      io[j] = poisoned ? (uint32_t)j : 0xFFFFu - (top[j] & 0xFFFFu);
      wo[j] = Dt<T>::from_f(poisoned ? __int_as_float(0x7FC00000) : ex[j] / denom);
    }
  }
}

template <typename T>
cudaError_t launch_route16_small(const void* logits, int64_t T_, int E, int k, int renorm,
                                 uint32_t* idx, void* w, cudaStream_t s) {
  const unsigned blocks = (unsigned)((T_ + 255) / 256);
  const uint4* l = (const uint4*)logits;
#define MOE_R16(NV)                                                                             \
  case NV:                                                                                      \
    if (renorm)                                                                                 \
      moe_route16_small<T, NV, true><<<blocks, 256, 0, s>>>(l, T_, k, idx, (T*)w);              \
    else                                                                                        \
      moe_route16_small<T, NV, false><<<blocks, 256, 0, s>>>(l, T_, k, idx, (T*)w);             \
    break;
  switch (E / 8) {
    MOE_R16(1) MOE_R16(2) MOE_R16(3) MOE_R16(4) MOE_R16(5) MOE_R16(6) MOE_R16(7) MOE_R16(8)
    default: return cudaErrorInvalidValue;
  }
#undef MOE_R16
  return cudaGetLastError();
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
  if constexpr (sizeof(T) == 2) {
    if (E <= 64 && E % 8 == 0 && k <= 8 && ((uintptr_t)logits) % 16 == 0)
      return launch_route16_small<T>(logits, T_, E, k, renorm, idx, w, s);
  }
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
