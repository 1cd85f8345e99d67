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
// one row per thread.
//
// Ranking.  A larger logit ranks first, equal logits prefer the lower id.  Most rows are decided
// on half-width keys: with m the row's largest value,
//     key16 = d << 6 | id,   d = min(number of 16-bit codes from the value up to m, 1023),
// smaller first.  The 1023 codes below m keep their exact order and every lower value is squashed
// into d = 1023.  d comes straight from the storage bits: when m is positive (bits >= 1023 as a
// signed 16-bit integer) the non-negative values in the window are ordered like their bits, and a
// signed packed max against m - 1023 clamps everything lower (every negative value included); when
// m is negative every value is, and flipping all bits turns them into the same case.  Two keys
// share a register (even expert in the low half, odd in the high half) and the packed min / max
// (min.u16x2) runs the sorting networks on both halves at once: each 8-word group is two
// independent 8-input sorts, the groups merge into two sorted top-8 lists (elementwise min against
// the reversed list, then a half-cleaner), and a last merge of the low half against the high half
// leaves the row's top 8.  When the 8th key has d < 1023, every chosen key lies in the window,
// where the order is exact, and every key not chosen is below it.  Otherwise (the top 8 span more
// than 1023 codes, e.g. -inf among them), and for rows whose largest value is a zero or tiny, the
// row is decided again on exact 32-bit keys: monotone code << 16 | (0xFFFF - id), larger first.
__device__ __forceinline__ uint32_t vmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t vmin2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t vmax2s(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// packed floating-point max of both halves; a NaN in either operand gives NaN
template <typename T>
__device__ __forceinline__ uint32_t fmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (Dt<T>::code == MOE_BF16) {
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  } else {
    asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  }
  return d;
}
// compare-exchange: ASC = smaller first on packed 16-bit halves, else larger first on 32-bit keys
template <bool ASC>
__device__ __forceinline__ void cx(uint32_t& a, uint32_t& b) {
  const uint32_t f = ASC ? vmin2(a, b) : max(a, b), s = ASC ? vmax2(a, b) : min(a, b);
  a = f;
  b = s;
}
template <bool ASC>
__device__ __forceinline__ void sort8(uint32_t (&k)[8]) {
  cx<ASC>(k[0], k[1]); cx<ASC>(k[2], k[3]); cx<ASC>(k[4], k[5]); cx<ASC>(k[6], k[7]);
  cx<ASC>(k[0], k[2]); cx<ASC>(k[1], k[3]); cx<ASC>(k[4], k[6]); cx<ASC>(k[5], k[7]);
  cx<ASC>(k[1], k[2]); cx<ASC>(k[5], k[6]);
  cx<ASC>(k[0], k[4]); cx<ASC>(k[1], k[5]); cx<ASC>(k[2], k[6]); cx<ASC>(k[3], k[7]);
  cx<ASC>(k[2], k[4]); cx<ASC>(k[3], k[5]);
  cx<ASC>(k[1], k[2]); cx<ASC>(k[3], k[4]); cx<ASC>(k[5], k[6]);
}
// bitonic sequence of 8 -> sorted
template <bool ASC>
__device__ __forceinline__ void clean8(uint32_t (&t)[8]) {
  cx<ASC>(t[0], t[4]); cx<ASC>(t[1], t[5]); cx<ASC>(t[2], t[6]); cx<ASC>(t[3], t[7]);
  cx<ASC>(t[0], t[2]); cx<ASC>(t[1], t[3]); cx<ASC>(t[4], t[6]); cx<ASC>(t[5], t[7]);
  cx<ASC>(t[0], t[1]); cx<ASC>(t[2], t[3]); cx<ASC>(t[4], t[5]); cx<ASC>(t[6], t[7]);
}
// top, g: sorted.  Leaves the 8 best of both in `top`, sorted.
template <bool ASC>
__device__ __forceinline__ void merge8(uint32_t (&top)[8], const uint32_t (&g)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) top[i] = ASC ? vmin2(top[i], g[7 - i]) : max(top[i], g[7 - i]);
  clean8<ASC>(top);
}
template <typename T>
__device__ __forceinline__ float bits16_to_float(uint32_t b) {
  if constexpr (sizeof(T) == 2 && Dt<T>::code == MOE_BF16) {
    return __uint_as_float(b << 16);
  } else {
    return __half2float(__ushort_as_half((unsigned short)b));
  }
}
constexpr float kLog2e = 1.4426950408889634f;
// 2^y (PTX ex2.approx, subnormal results flushed to zero)
__device__ __forceinline__ float ex2_ftz(float y) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}

// Two FP32 lanes in one 64-bit register, low lane first, and the packed FP32 operations of
// sm_100 and later (one instruction for both lanes, each lane rounded as its scalar form).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float lo_f32(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f32(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// Softmax denominator of one row over all E experts against its maximum x0: sum of exp(x - x0)
// = 2^((x - x0) log2 e), read again from the row's vectors (rowv[v ^ sw]), both logits of a
// 32-bit word in the two lanes of packed FP32 operations.  Terms below 2^-126 are flushed to
// zero, which leaves the sum (>= 1, the maximum's own term) unchanged.  For |x0| <= 64 the
// exponent is one FMA, x log2 e - x0 log2 e, whose rounding of x0 log2 e costs at most
// 2^-24 * 93 < 6e-6 in the exponent; larger maxima subtract first.
template <typename T, int NV, bool SMALL>
__device__ __forceinline__ float row_denominator_t(const uint4* rowv, int sw, float x0) {
  const uint64_t l2 = f32x2(kLog2e, kLog2e);
  const uint64_t c2 = SMALL ? f32x2(-x0 * kLog2e, -x0 * kLog2e) : f32x2(-x0, -x0);
  uint64_t acc = 0ull;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const uint4 q = rowv[v ^ sw];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t x = f32x2(bits16_to_float<T>(w[i] & 0xFFFFu), bits16_to_float<T>(w[i] >> 16));
      const uint64_t y = SMALL ? fma_f32x2(x, l2, c2) : mul_f32x2(add_f32x2(x, c2), l2);
      acc = add_f32x2(acc, f32x2(ex2_ftz(lo_f32(y)), ex2_ftz(hi_f32(y))));
    }
  }
  return lo_f32(acc) + hi_f32(acc);
}
template <typename T, int NV>
__device__ __forceinline__ float row_denominator(const uint4* rowv, int sw, float x0) {
  return fabsf(x0) <= 64.f ? row_denominator_t<T, NV, true>(rowv, sw, x0)
                           : row_denominator_t<T, NV, false>(rowv, sw, x0);
}

// Weights of the chosen experts (ids, logits) and the stores of one row.
template <typename T, int NV, bool RENORM>
__device__ __forceinline__ void emit_row(uint32_t (&id)[8], const float (&x)[8], bool poisoned,
                                         float x0, const uint4* rowv, int sw, int k,
                                         int vec_store, uint32_t* __restrict__ idx_out,
                                         T* __restrict__ w_out, int64_t row) {
  // exp(x - x0) of the chosen logits as (2^((x - x0) log2 e / 2))^2, two per packed operation:
  // the half power stays normal down to (x - x0) log2 e = -252, and the square (an IEEE multiply)
  // rounds into the subnormal range where the result lies there
  uint64_t ex[4];
  float sel = 0.f;
  const uint64_t nx0 = f32x2(-x0, -x0), hl2 = f32x2(0.5f * kLog2e, 0.5f * kLog2e);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t y = mul_f32x2(add_f32x2(f32x2(x[2 * j], x[2 * j + 1]), nx0), hl2);
    const uint64_t h = f32x2(ex2_ftz(lo_f32(y)), ex2_ftz(hi_f32(y)));
    ex[j] = mul_f32x2(h, h);
    if (2 * j < k) sel += lo_f32(ex[j]);
    if (2 * j + 1 < k) sel += hi_f32(ex[j]);
  }
  const float inv = 1.f / (RENORM || poisoned ? sel : row_denominator<T, NV>(rowv, sw, x0));
  float wt[8];
  const uint64_t inv2 = f32x2(inv, inv);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t q = mul_f32x2(ex[j], inv2);
    wt[2 * j] = poisoned ? __int_as_float(0x7FC00000) : lo_f32(q);
    wt[2 * j + 1] = poisoned ? __int_as_float(0x7FC00000) : hi_f32(q);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) id[j] = poisoned ? (uint32_t)j : id[j];
  if (vec_store) {  // k == 8, 16-byte aligned outputs
    uint4* io = reinterpret_cast<uint4*>(idx_out + row * 8);
    io[0] = make_uint4(id[0], id[1], id[2], id[3]);
    io[1] = make_uint4(id[4], id[5], id[6], id[7]);
    uint32_t p[4];  // two weights per word, each rounded to nearest even, the first in the low half
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if constexpr (Dt<T>::code == MOE_BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(wt[2 * j], wt[2 * j + 1]);
        p[j] = *reinterpret_cast<const uint32_t*>(&h);
      } else {
        const __half2 h = __floats2half2_rn(wt[2 * j], wt[2 * j + 1]);
        p[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
    *reinterpret_cast<uint4*>(w_out + row * 8) = make_uint4(p[0], p[1], p[2], p[3]);
  } else {
    uint32_t* io = idx_out + row * k;
    T* wo = w_out + row * k;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        io[j] = id[j];
        wo[j] = Dt<T>::from_f(wt[j]);
      }
    }
  }
}

// A row decided on exact 32-bit keys (monotone code << 16 | (0xFFFF - id), larger first): every
// f16 row, and the bf16 rows whose top 8 reach below the half-width window or whose largest value
// is a zero or tiny (for those it is called out of line, so that the common path holds no
// registers for it).  Vector v of the row is rowv[v ^ sw] (shared or global memory).
template <typename T, int NV, bool RENORM>
__device__ __forceinline__ void exact_row(const uint4* rowv, int sw, float x0, int k,
                                          int vec_store, uint32_t* idx_out, T* w_out,
                                          int64_t row) {
  uint32_t top[8];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const uint4 q = rowv[v ^ sw];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t g[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // monotone code of both halves: negative -> all bits flipped, else sign bit set; prmt
      // with selector 0xBB99 replicates each half's sign bit over the half.  A -0 half is
      // first made +0 (equal logits share a code, and the lower id goes first).
      const uint32_t wz = w[i] & ~__vcmpeq2(w[i], 0x80008000u);
      uint32_t sm;
      asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(sm) : "r"(wz));
      const uint32_t m = wz ^ (sm | 0x80008000u);
      const uint32_t e0 = v * 8 + i * 2;
      g[2 * i] = (m << 16) | (0xFFFFu - e0);
      g[2 * i + 1] = (m & 0xFFFF0000u) | (0xFFFFu - (e0 + 1));
    }
    sort8<false>(g);
    if (v == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) top[i] = g[i];
    } else {
      merge8<false>(top, g);
    }
  }
  uint32_t id[8];
  float x[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t t = top[j] >> 16;
    id[j] = 0xFFFFu - (top[j] & 0xFFFFu);
    x[j] = bits16_to_float<T>((t & 0x8000u) ? (t & 0x7FFFu) : (~t & 0xFFFFu));
  }
  emit_row<T, NV, RENORM>(id, x, false, x0, rowv, sw, k, vec_store, idx_out, w_out, row);
}
template <typename T, int NV, bool RENORM>
__device__ __noinline__ void exact_row_outlined(const uint4* rowv, int sw, float x0, int k,
                                                int vec_store, uint32_t* idx_out, T* w_out,
                                                int64_t row) {
  exact_row<T, NV, RENORM>(rowv, sw, x0, k, vec_store, idx_out, w_out, row);
}

template <typename T, int NV, bool RENORM>
__global__ void __launch_bounds__(256, (RENORM || Dt<T>::code == MOE_BF16) ? 5 : 4)
    moe_route16_small(const uint4* __restrict__ logits, int64_t T_, int k, int vec_store,
                      uint32_t* __restrict__ idx_out, T* __restrict__ w_out) {
  constexpr uint32_t EXPMASK = Dt<T>::code == MOE_BF16 ? 0x7F80u : 0x7C00u;
  constexpr int NG = (NV + 1) / 2;  // groups of 8 words (16 experts)
  // half-width keys for bf16 only: f16's 10-bit mantissa puts a single binade in the window
  constexpr bool HALF = Dt<T>::code == MOE_BF16;
  const int tid = threadIdx.x;
  const int64_t row0 = (int64_t)blockIdx.x * 256;
  const int64_t row = row0 + tid;
  // E = 64: the block's 256 rows (32 KB, contiguous) are read with coalesced 16-byte loads into
  // shared memory, vector v of row r stored at slot v ^ (r & 7) so that the row-per-thread reads
  // below hit 8 different bank groups per 8 lanes.  Chunk c = tid + 256 i belongs to row c / 8,
  // whose low three bits are those of tid / 8, so its slot is c ^ ((tid / 8) & 7).
  constexpr bool STAGED = NV == 8;
  __shared__ uint4 tile[STAGED ? 256 * 8 : 1];
  if (STAGED) {
    const int64_t left = T_ - row0;
    const int n = (int)((left < 256 ? left : 256) * 8);
    const uint4* bsrc = logits + row0 * 8 + tid;
    uint4* dst = tile + (tid ^ ((tid >> 3) & 7));
    if (n == 2048) {
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i * 256] = ld_nc_v4(bsrc + i * 256);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (tid + i * 256 < n) dst[i * 256] = ld_nc_v4(bsrc + i * 256);
    }
    __syncthreads();
  }
  if (row >= T_) return;
  const uint4* src = logits + row * NV;
  auto load = [&](int v) -> uint4 {
    return STAGED ? tile[tid * 8 + (v ^ (tid & 7))] : ld_nc_v4(src + v);
  };

  // pass 1: the row maximum, NaN-propagating
  uint32_t wv[NG * 8];
  uint32_t fm = 0u;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const uint4 q = load(v);
    wv[4 * v] = q.x; wv[4 * v + 1] = q.y; wv[4 * v + 2] = q.z; wv[4 * v + 3] = q.w;
#pragma unroll
    for (int i = 0; i < 4; ++i) fm = v == 0 && i == 0 ? wv[0] : fmax2_nan<T>(fm, wv[4 * v + i]);
  }
  const uint32_t mb = fmax2_nan<T>(fm, fm >> 16) & 0xFFFFu;  // storage bits of the maximum
  // poisoned: the maximum is NaN (a NaN anywhere) or +inf, or -inf (every value is -inf)
  const bool poisoned = (mb & 0x7FFFu) >= EXPMASK;
  const bool pos = mb >= 1023u && mb < 0x8000u;          // positive maximum, window all >= 0
  const bool neg = mb > 0x8000u && mb <= 0xFC00u;        // negative maximum, so is every value
  const float x0 = bits16_to_float<T>(mb);

  const uint4* rowv = STAGED ? tile + tid * 8 : src;
  const int sw = STAGED ? (tid & 7) : 0;
  if (poisoned) {
    uint32_t id[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    emit_row<T, NV, RENORM>(id, x, true, x0, rowv, sw, k, vec_store, idx_out, w_out, row);
    return;
  }
  if constexpr (!HALF) {
    exact_row<T, NV, RENORM>(rowv, sw, x0, k, vec_store, idx_out, w_out, row);
    return;
  }
  if (!(pos || neg)) {
    exact_row_outlined<T, NV, RENORM>(rowv, sw, x0, k, vec_store, idx_out, w_out, row);
    return;
  }

  // pass 2: half-width keys d << 6 | id, two per register
  if (neg) {
#pragma unroll
    for (int j = 0; j < NV * 4; ++j) wv[j] = ~wv[j];
  }
  const uint32_t mf = neg ? (mb ^ 0xFFFFu) : mb;  // maximum in the (flipped) bit order
  const uint32_t floor2 = (mf - 1023u) * 0x10001u, m2 = mf * 0x10001u;
#pragma unroll
  for (int j = 0; j < NV * 4; ++j)
    wv[j] = (m2 - vmax2s(wv[j], floor2)) * 64u + ((uint32_t)(2 * j + 1) << 16 | (uint32_t)(2 * j));
#pragma unroll
  for (int j = NV * 4; j < NG * 8; ++j) wv[j] = 0xFFFFFFFFu;  // padding after every real key
  uint32_t top[8];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    uint32_t g[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = wv[8 * gi + i];
    sort8<true>(g);
    if (gi == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) top[i] = g[i];
    } else {
      merge8<true>(top, g);
    }
  }
  {  // low half (even experts) against the reversed high half (odd experts)
    uint32_t r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) asm("prmt.b32 %0, %1, 0, 0x1032;" : "=r"(r[i]) : "r"(top[7 - i]));
#pragma unroll
    for (int i = 0; i < 8; ++i) top[i] = vmin2(top[i], r[i]);
    clean8<true>(top);
  }
  if ((top[7] & 0xFFFFu) >= 1023u * 64u) {  // the 8th key squashed: decide again exactly
    exact_row_outlined<T, NV, RENORM>(rowv, sw, x0, k, vec_store, idx_out, w_out, row);
    return;
  }
  // chosen ids, and their logits: bf16 bits ((mf - d) ^ flip) << 16 = (mf << 16) - (d << 16)
  // ^ (flip << 16), with d << 16 = (key & 0xFFC0) << 10
  uint32_t id[8];
  float x[8];
  const uint32_t m16 = mf << 16, fl16 = neg ? 0xFFFF0000u : 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    id[j] = top[j] & 63u;
    x[j] = __uint_as_float((m16 - (top[j] & 0xFFC0u) * 1024u) ^ fl16);
  }
  emit_row<T, NV, RENORM>(id, x, false, x0, rowv, sw, k, vec_store, idx_out, w_out, row);
}

template <typename T>
cudaError_t launch_route16_small(const void* logits, int64_t T_, int E, int k, int renorm,
                                 uint32_t* idx, void* w, cudaStream_t s) {
  const unsigned blocks = (unsigned)((T_ + 255) / 256);
  const uint4* l = (const uint4*)logits;
  const int vst = k == 8 && ((uintptr_t)idx % 16) == 0 && ((uintptr_t)w % 16) == 0;
#define MOE_R16(NV)                                                                             \
  case NV:                                                                                      \
    if (renorm)                                                                                 \
      moe_route16_small<T, NV, true><<<blocks, 256, 0, s>>>(l, T_, k, vst, idx, (T*)w);         \
    else                                                                                        \
      moe_route16_small<T, NV, false><<<blocks, 256, 0, s>>>(l, T_, k, vst, idx, (T*)w);        \
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
