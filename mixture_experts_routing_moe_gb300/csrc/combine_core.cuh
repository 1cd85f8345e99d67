// One warp's share of the combine (ruDNN user guide, §3 "MoE-Workflow" / §6 "MoE aufrufen"):
// columns [32 c0 VW, 32 c0 VW + 32 VW) of out[t] = sum_j w[t, j] * y[row_of_slot[t*k + j]],
// FP32 accumulation in the fixed slot order j = 0..k-1, one rounding to the output dtype.  A
// slot without a row (poisoned routing) makes the token's output NaN.  With w == nullptr every
// weight is 1 (fmaf(1, v, acc) rounds as acc + v): the slot sum of dispatch_backward.  COHERENT reads y, the map
// and the weights through L2 only (they were written earlier in the same launch).
#pragma once

#include "common.cuh"

namespace moe {

// BATCH: slots whose loads are issued before their FMAs (8 where few warps are in flight, as in
// the fused kernel; 2 in the stage kernel, whose many warps hide most of the load latency: on the
// skewed layer 2 measured 3 % faster than 1, 4 and 8 slower).
template <typename TY, typename TW, bool VEC, bool COHERENT, int BATCH>
__device__ __forceinline__ void combine_warp(const TY* __restrict__ y,
                                             const uint32_t* __restrict__ row_of_slot,
                                             const TW* __restrict__ w, int64_t t, int64_t H, int k,
                                             int64_t c0, TY* __restrict__ out, int lane) {
  constexpr int VW = VEC ? 16 / (int)sizeof(TY) : 1;
  const int64_t chunks = H / VW;
  const int64_t c = c0 * 32 + lane;  // this lane's column chunk
  float acc[VW];
#pragma unroll
  for (int i = 0; i < VW; ++i) acc[i] = 0.f;
  bool poisoned = false;
  for (int jb = 0; jb < k; jb += 32) {
    uint32_t my_row = kInvalidRow;
    float my_w = 0.f;
    if (jb + lane < k) {
      if constexpr (COHERENT) {
        my_row = ld_elem<true>(row_of_slot + t * k + jb + lane);
        my_w = w ? Dt<TW>::to_f(ld_elem<true>(w + t * k + jb + lane)) : 1.f;
      } else {
        my_row = row_of_slot[t * k + jb + lane];
        my_w = w ? Dt<TW>::to_f(w[t * k + jb + lane]) : 1.f;  // no weights: the plain sum
      }
    }
    const int nj = min(32, k - jb);
    if constexpr (BATCH == 1) {  // one slot at a time: load, then FMA
      for (int jj = 0; jj < nj; ++jj) {
        const uint32_t r = __shfl_sync(0xFFFFFFFFu, my_row, jj);
        const float wj = __shfl_sync(0xFFFFFFFFu, my_w, jj);
        if (r == kInvalidRow) {
          poisoned = true;
          continue;
        }
        if (c < chunks) {
          if (VEC) {
            Vec16<TY> q;
            q.u = ld_v4<COHERENT>(y + (int64_t)r * H + c * VW);
            float f[VW];
            q.to_float(f);
#pragma unroll
            for (int i = 0; i < VW; ++i) acc[i] = fmaf(wj, f[i], acc[i]);
          } else {
            acc[0] = fmaf(wj, Dt<TY>::to_f(ld_elem<COHERENT>(y + (int64_t)r * H + c)), acc[0]);
          }
        }
      }
      continue;
    }
    // groups of kBatch slots: all loads of a group are issued before its FMAs, which still run
    // in slot order
    constexpr int kBatch = BATCH;
    for (int j0 = 0; j0 < nj; j0 += kBatch) {
      uint32_t r[kBatch];
      float wj[kBatch];
      uint4 v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int jj = min(j0 + b, nj - 1);
        r[b] = __shfl_sync(0xFFFFFFFFu, my_row, jj);
        wj[b] = __shfl_sync(0xFFFFFFFFu, my_w, jj);
        const bool live = j0 + b < nj && r[b] != kInvalidRow && c < chunks;
        if (VEC) {
          v[b] = live ? ld_v4<COHERENT>(y + (int64_t)r[b] * H + c * VW) : make_uint4(0, 0, 0, 0);
        } else {
          const float f = live ? Dt<TY>::to_f(ld_elem<COHERENT>(y + (int64_t)r[b] * H + c)) : 0.f;
          v[b].x = __float_as_uint(f);
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (j0 + b >= nj) break;
        if (r[b] == kInvalidRow) {
          poisoned = true;
          continue;
        }
        if (c < chunks) {
          if (VEC) {
            Vec16<TY> q;
            q.u = v[b];
            float f[VW];
            q.to_float(f);
#pragma unroll
            for (int i = 0; i < VW; ++i) acc[i] = fmaf(wj[b], f[i], acc[i]);
          } else {
            acc[0] = fmaf(wj[b], __uint_as_float(v[b].x), acc[0]);
          }
        }
      }
    }
  }
  if (c < chunks) {
    if (poisoned) {
#pragma unroll
      for (int i = 0; i < VW; ++i) acc[i] = __int_as_float(0x7FC00000);
    }
    if (VEC) {
      Vec16<TY> q;
      q.from_float(acc);
      st_v4(out + t * H + c * VW, q.u);
    } else {
      out[t * H + c] = Dt<TY>::from_f(acc[0]);
    }
  }
}

}  // namespace moe
