// Softmax top-k routing of one row of logits (ruDNN user guide, §4 "Routing-Vertrag"), shared by
// the route kernel and the fused decode kernel.
//
// The row is owned by L consecutive lanes of a warp (L = 1..32); lane gl of the group holds the
// contiguous elements [gl*C, gl*C + C), read with 16-byte loads when VEC.  The softmax runs in FP32
// over all E experts (max and sum reduced with xor shuffles inside the group).  The top-k is k
// rounds of a group argmax over 64-bit keys
//     key = monotone_bits(logit) << 32 | (0xFFFFFFFF - id)
// (32-bit keys, the 16-bit code and 0xFFFF - id, for 16-bit logits), so a larger key is a larger
// logit, and equal logits prefer the lower id; the winner of each round is removed by its owner.  Rows holding a NaN or +inf, or only -inf, get NaN weights and
// ids 0..k-1.  Lanes past E hold nothing and add exact zeros to the sums, so a wider group than
// needed gives the same bits.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint32_t monotone_bits(float v) {
  uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_monotone_bits(uint32_t m) {
  uint32_t u = (m & 0x80000000u) ? (m & 0x7FFFFFFFu) : ~m;
  return __uint_as_float(u);
}

// Storage bits of a float that holds a 16-bit (bf16 / f16) number, exact, and back.
template <typename T>
__device__ __forceinline__ uint32_t bits16_of(float v) {
  if constexpr (Dt<T>::code == MOE_BF16) return __float_as_uint(v) >> 16;
  else return __half_as_ushort(__float2half_rn(v));
}
template <typename T>
__device__ __forceinline__ float float_of_bits16(uint32_t b) {
  if constexpr (Dt<T>::code == MOE_BF16) return __uint_as_float(b << 16);
  else return __half2float(__ushort_as_half((unsigned short)b));
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

// Route `row` (only written when row_ok; every lane of the warp must call this together).
// s_id / s_e: k entries of shared memory for this row's selection.
template <typename T, int L, int C, bool VEC>
__device__ __forceinline__ void route_row(const T* __restrict__ logits, int64_t row, bool row_ok,
                                          int E, int k, int renorm, int gl, uint32_t* s_id,
                                          float* s_e, uint32_t* __restrict__ idx_out,
                                          T* __restrict__ w_out) {
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

  float sel = 0.f;
  if constexpr (sizeof(T) == 2) {
    // 16-bit logits: 32-bit keys monotone16(storage bits) << 16 | (0xFFFF - id) order exactly as
    // the 64-bit ones (E <= 65535), at a quarter of the integer work per compare and shuffle
    uint32_t key[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      uint32_t b = bits16_of<T>(v[c]);
      if (b == 0x8000u) b = 0u;  // -0 and +0 are equal logits: the same key, lower id first
      const uint32_t m16 = (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
      key[c] = (e0 + c < E) ? (m16 << 16) | (0xFFFFu - (uint32_t)(e0 + c)) : 0u;
    }
    for (int r = 0; r < k; ++r) {
      uint32_t best = key[0];
#pragma unroll
      for (int c = 1; c < C; ++c) best = max(best, key[c]);
      best = group_max<L>(best);
      const uint32_t id = 0xFFFFu - (best & 0xFFFFu), mb = best >> 16;
      const float ex = __expf(float_of_bits16<T>((mb & 0x8000u) ? (mb & 0x7FFFu) : (~mb & 0xFFFFu)) - m);
      sel += ex;
#pragma unroll
      for (int c = 0; c < C; ++c) key[c] = key[c] == best ? 0u : key[c];
      if (gl == 0) {
        s_id[r] = id;
        s_e[r] = ex;
      }
    }
  } else {
    uint64_t key[C];
#pragma unroll
    for (int c = 0; c < C; ++c)
      key[c] = (e0 + c < E)  // (v == 0 for both zeros: -0 takes +0's key)
                   ? ((uint64_t)monotone_bits(v[c] == 0.f ? 0.f : v[c]) << 32) |
                         (0xFFFFFFFFu - (uint32_t)(e0 + c))
                   : 0ull;
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

}  // namespace moe
