// Group-limited sigmoid routing of one row of logits (ruDNN user guide, §10
// "Gruppenbeschränktes Sigmoid-MoE-Routing"), shared by the sigmoid route kernel and the fused
// short-batch kernel.  The method and the float64 decision are described in route_sigmoid.cu.
#pragma once

#include "common.cuh"

namespace moe {

// warp argmax of (v, id): larger v wins, equal v -> smaller id; returns the winner in all lanes
__device__ __forceinline__ void warp_argmax(double& v, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, id, o);
    if (ov > v || (ov == v && oi < id)) {
      v = ov;
      id = oi;
    }
  }
}

// float argmax over (v, id) with the same rule; all lanes get the winner
__device__ __forceinline__ void warp_argmax_f(float& v, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, id, o);
    if (ov > v || (ov == v && oi < id)) {
      v = ov;
      id = oi;
    }
  }
}

// The FP32 attempt at one row (see the file comment).  Returns true when it wrote the row's ids
// and weights; false leaves the row to the float64 path.  sm: per-warp scratch of at least
// E + 2 G floats.  Every lane of the warp calls it and gets the same answer.
template <typename T, int C>
__device__ __forceinline__ bool sigmoid_row_fp32(const T* __restrict__ src,
                                                 const float* __restrict__ bias, int64_t row, int E,
                                                 int k, int G, int SG, int top_two, int renorm,
                                                 float scale, float* sm, int lane,
                                                 uint32_t* __restrict__ idx_out,
                                                 T* __restrict__ w_out) {
  if (k > 32) return false;  // slot r's expert is kept in lane r
  const int gs = E / G;
  float c[C];
  float amax = 0.f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float x = Dt<T>::to_f(src[e]);
      const float sg = 1.0f / (1.0f + expf(-x));
      c[i] = sg + (bias ? bias[e] : 0.f);
      finite &= isfinite(c[i]);
      amax = fmaxf(amax, fabsf(c[i]));
      sm[e] = c[i];
    } else {
      c[i] = 0.f;
    }
  }
  if (!__all_sync(0xFFFFFFFFu, finite)) return false;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const float ec = 5e-7f + 1.2e-7f * amax;                       // bound on |c32 - c64|
  const float eg = (top_two ? 2.f * ec : ec) + 2.4e-7f * amax;    // bound on a group score
  __syncwarp();
  float* gsc = sm + E;  // [G]
  for (int g = lane; g < G; g += 32) {
    float b1 = -INFINITY, b2 = -INFINITY;
    for (int j = 0; j < gs; ++j) {
      const float v = sm[g * gs + j];
      if (v > b1) {
        b2 = b1;
        b1 = v;
      } else if (v > b2) {
        b2 = v;
      }
    }
    gsc[g] = top_two ? b1 + b2 : b1;
  }
  __syncwarp();
  // SG groups, then (when SG < G) the best other group: its margin to the last chosen one
  unsigned long long chosen_lo = 0, chosen_hi = 0;
  float last = 0.f;
  for (int r = 0; r < SG + (SG < G ? 1 : 0); ++r) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int g = lane; g < G; g += 32) {
      const bool taken = g < 64 ? (chosen_lo >> g) & 1ull : (chosen_hi >> (g - 64)) & 1ull;
      const float v = gsc[g];
      if (!taken && (bi == 0x7FFFFFFF || v > bv || (v == bv && g < bi))) {
        bv = v;
        bi = g;
      }
    }
    warp_argmax_f(bv, bi);
    if (r == SG) {
      if (!(last - bv > 2.f * eg)) return false;
      break;
    }
    last = bv;
    if (bi < 64) chosen_lo |= 1ull << bi;
    else chosen_hi |= 1ull << (bi - 64);
  }
  // top_k experts of the chosen groups, then the best unchosen one; all margins must clear 2 ec
  const int cand = SG * gs;
  unsigned avail = 0;  // this lane's elements that are candidates and not taken yet
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const int g = e / gs;
      if (g < 64 ? (chosen_lo >> g) & 1ull : (chosen_hi >> (g - 64)) & 1ull) avail |= 1u << i;
    }
  }
  float prev = 0.f, px = 0.f, pb = 0.f;
  int my_id = -1;
  for (int r = 0; r < k + (k < cand ? 1 : 0); ++r) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const int e = lane + 32 * i;
      if (((avail >> i) & 1u) && (bi == 0x7FFFFFFF || c[i] > bv || (c[i] == bv && e < bi))) {
        bv = c[i];
        bi = e;
      }
    }
    warp_argmax_f(bv, bi);
    // the previous winner beats this one by the margin, or the two have the same logit and the
    // same correction (then the same score in any precision: the lower id, taken first, wins)
    const float wx = Dt<T>::to_f(src[bi]), wb = bias ? bias[bi] : 0.f;
    if (r > 0 && !(prev - bv > 2.f * ec) && !(bv == prev && wx == px && wb == pb)) return false;
    if (r == k) break;
    prev = bv;
    px = wx;
    pb = wb;
    if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
    if (lane == r) my_id = bi;  // slot r's expert lives in lane r (k <= 32 here)
  }
  // Weights.  16-bit outputs: w in FP32 (relative error below kWeightErr); when w (1 - err) and
  // w (1 + err) round to the same 16-bit value, that value is the rounding of the float64 weight.
  // Otherwise, and for f32 outputs, the float64 path's arithmetic: sigmoids of the chosen experts
  // in float64, summed in slot order.
  float w32 = 0.f;
  if (lane < k) w32 = 1.0f / (1.0f + expf(-Dt<T>::to_f(src[my_id])));
  float sel32 = 0.f;
  for (int j = 0; j < k; ++j) sel32 += __shfl_sync(0xFFFFFFFFu, w32, j);
  bool exact = sizeof(T) == 2;
  T wout = Dt<T>::from_f(0.f);
  if (exact && lane < k) {
    constexpr float kWeightErr = 4e-6f;  // s: 4e-7 each; the sum of <= 32: 32 x 4e-7; / and *: 1e-7
    const float w = (renorm ? w32 / sel32 : w32) * scale;
    wout = Dt<T>::from_f(w);
    const T lo = Dt<T>::from_f(w * (1.f - kWeightErr)), hi = Dt<T>::from_f(w * (1.f + kWeightErr));
    exact = Dt<T>::to_f(lo) == Dt<T>::to_f(wout) && Dt<T>::to_f(hi) == Dt<T>::to_f(wout);
  }
  if (!__all_sync(0xFFFFFFFFu, exact)) {
    double sv = 0.0;
    if (lane < k) {
      const double x = (double)Dt<T>::to_f(src[my_id]);
      sv = 1.0 / (1.0 + exp(-x));
    }
    double sel = 0.0;
    for (int j = 0; j < k; ++j) sel += __shfl_sync(0xFFFFFFFFu, sv, j);
    double w = sv;
    if (renorm) w = w / sel;
    w *= (double)scale;
    wout = Dt<T>::from_f((float)w);
  }
  if (lane < k) {
    idx_out[row * k + lane] = (uint32_t)my_id;
    w_out[row * k + lane] = wout;
  }
  return true;
}

// Route one row (every lane of the warp calls this together): the FP32 attempt, and the float64
// decision when the attempt cannot prove its choice.  cs: per-warp shared scratch of
// E + 128 + 64 + 32 doubles.
template <typename T, int C>
__device__ __forceinline__ void sigmoid_route_row(const T* __restrict__ src,
                                                  const float* __restrict__ bias, int64_t row,
                                                  int E, int k, int G, int SG, int top_two,
                                                  int renorm, float scale, double* cs, int lane,
                                                  uint32_t* __restrict__ idx_out,
                                                  T* __restrict__ w_out) {
  const int gs = E / G;
  double* gsc = cs + E;
  if (sigmoid_row_fp32<T, C>(src, bias, row, E, k, G, SG, top_two, renorm, scale,
                             reinterpret_cast<float*>(cs), lane, idx_out, w_out))
    return;

  double s[C], c[C];
  bool nan_seen = false;
#pragma unroll
  for (int i = 0; i < C; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const double x = (double)Dt<T>::to_f(src[e]);
      s[i] = 1.0 / (1.0 + exp(-x));
      c[i] = s[i] + (bias ? (double)bias[e] : 0.0);
      nan_seen |= c[i] != c[i];
      cs[e] = c[i];
    } else {
      s[i] = c[i] = 0.0;
    }
  }
  const bool poisoned = __any_sync(0xFFFFFFFFu, nan_seen);
  __syncwarp();

  // group scores: lane g handles groups g, g + 32, ...
  for (int g = lane; g < G; g += 32) {
    double b1 = -INFINITY, b2 = -INFINITY;
    for (int j = 0; j < gs; ++j) {
      const double v = cs[g * gs + j];
      if (v > b1) {
        b2 = b1;
        b1 = v;
      } else if (v > b2) {
        b2 = v;
      }
    }
    gsc[g] = top_two ? b1 + b2 : b1;
  }
  __syncwarp();

  // choose SG groups, best first; chosen groups are remembered in a 128-bit mask
  unsigned long long chosen_lo = 0, chosen_hi = 0;  // bitmap of chosen groups (G <= 128)
  for (int r = 0; r < SG; ++r) {
    double bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int g = lane; g < G; g += 32) {
      const bool taken = g < 64 ? (chosen_lo >> g) & 1ull : (chosen_hi >> (g - 64)) & 1ull;
      const double v = gsc[g];
      if (!taken && (bi == 0x7FFFFFFF || v > bv || (v == bv && g < bi))) {
        bv = v;
        bi = g;
      }
    }
    warp_argmax(bv, bi);
    if (bi < 64) chosen_lo |= 1ull << bi;
    else chosen_hi |= 1ull << (bi - 64);
  }

  // top_k experts inside the chosen groups; `used` marks experts already taken
  double* sel_s = gsc + 128;                                  // [64] chosen sigmoid values
  int* sel_id = reinterpret_cast<int*>(sel_s + 64);           // [64] chosen ids
  unsigned used = 0;
  double sel = 0.0;
  for (int r = 0; r < k; ++r) {
    double bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < C; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((used >> i) & 1u)) {
        const int g = e / gs;
        const bool ok = g < 64 ? (chosen_lo >> g) & 1ull : (chosen_hi >> (g - 64)) & 1ull;
        if (ok && (bi == 0x7FFFFFFF || c[i] > bv || (c[i] == bv && e < bi))) {
          bv = c[i];
          bi = e;
        }
      }
    }
    warp_argmax(bv, bi);
    const int owner = bi & 31, slot = bi >> 5;
    double sv = 0.0;
#pragma unroll
    for (int i = 0; i < C; ++i)
      if (lane == owner && i == slot) {
        used |= 1u << i;
        sv = s[i];
      }
    sv = __shfl_sync(0xFFFFFFFFu, sv, owner);
    sel += sv;
    if (lane == 0) {
      sel_s[r] = sv;
      sel_id[r] = bi;
    }
  }
  __syncwarp();
  for (int j = lane; j < k; j += 32) {
    double w = sel_s[j];
    if (renorm) w = w / sel;
    w *= (double)scale;
    idx_out[row * k + j] = poisoned ? (uint32_t)j : (uint32_t)sel_id[j];
    w_out[row * k + j] = Dt<T>::from_f(poisoned ? __int_as_float(0x7FC00000) : (float)w);
  }
}

}  // namespace moe
