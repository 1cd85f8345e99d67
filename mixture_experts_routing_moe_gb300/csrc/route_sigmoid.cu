// Group-limited sigmoid routing: route_sigmoid_grouped of the ruDNN user guide, §10
// "Gruppenbeschränktes Sigmoid-MoE-Routing".
//
// s = sigmoid(logit); c = s + bias (bias optional, FP32, selection only).  Experts form `groups`
// contiguous groups of gs = E / groups; a group scores its largest c, or the sum of its two largest
// with group_top_two.  The `selected_groups` best groups (ties: lower group id) are kept, then the
// top_k experts inside them by c (ties: lower id), slots in that order.  Weights are s of the
// chosen experts, divided by their sum when renormalising, times scale, rounded to the logits
// dtype.  Rows whose corrected scores hold a NaN get NaN weights and ids 0..k-1.
//
// The selection (sigmoid, correction, group scores, ranking) is computed in float64 so that it is
// the same decision as the float64 reference.  One warp owns a row: lane i holds experts
// i, i + 32, ...; s and c are staged in shared memory for the group scores; the group and expert
// choices are rounds of warp argmax over (score, -id) pairs.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int kSigWarps = 4;

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

template <typename T, int C>
__global__ void __launch_bounds__(kSigWarps * 32)
    moe_route_sigmoid_kernel(const T* __restrict__ logits, const float* __restrict__ bias,
                             int64_t T_, int E, int k, int G, int SG, int top_two, int renorm,
                             float scale, uint32_t* __restrict__ idx_out, T* __restrict__ w_out) {
  extern __shared__ double sig_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * kSigWarps + warp;
  if (row >= T_) return;  // whole warp leaves together
  // per warp: corrected scores [E], group scores [128], chosen sigmoids [64], chosen ids [64]
  double* cs = sig_smem + (size_t)warp * (E + 128 + 64 + 32);
  double* gsc = cs + E;
  const int gs = E / G;
  const T* src = logits + row * (int64_t)E;

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

template <typename T, int C>
cudaError_t launch_sig_c(const void* logits, const float* bias, int64_t T_, int E, int k, int G,
                         int SG, int top_two, int renorm, float scale, uint32_t* idx, void* w,
                         cudaStream_t s) {
  const size_t smem = (size_t)kSigWarps * (E + 128 + 64 + 32) * sizeof(double);
  cudaError_t err = cudaFuncSetAttribute(moe_route_sigmoid_kernel<T, C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const unsigned blocks = (unsigned)((T_ + kSigWarps - 1) / kSigWarps);
  moe_route_sigmoid_kernel<T, C><<<blocks, kSigWarps * 32, smem, s>>>(
      (const T*)logits, bias, T_, E, k, G, SG, top_two, renorm, scale, idx, (T*)w);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_sig_t(const void* logits, const float* bias, int64_t T_, int E, int k, int G,
                         int SG, int top_two, int renorm, float scale, uint32_t* idx, void* w,
                         cudaStream_t s) {
#define MOE_SIG(CC)                                                                        \
  if (E <= 32 * CC)                                                                        \
    return launch_sig_c<T, CC>(logits, bias, T_, E, k, G, SG, top_two, renorm, scale, idx, \
                               w, s);
  MOE_SIG(1) MOE_SIG(2) MOE_SIG(4) MOE_SIG(8) MOE_SIG(16) MOE_SIG(32)
#undef MOE_SIG
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_route_sigmoid(const void* logits, int ldt, const float* bias, int64_t T_, int E,
                                 int k, int G, int SG, int top_two, int renorm, float scale,
                                 uint32_t* idx, void* w, cudaStream_t s) {
  switch (ldt) {
    case MOE_F32:
      return launch_sig_t<float>(logits, bias, T_, E, k, G, SG, top_two, renorm, scale, idx, w, s);
    case MOE_F16:
      return launch_sig_t<__half>(logits, bias, T_, E, k, G, SG, top_two, renorm, scale, idx, w, s);
    case MOE_BF16:
      return launch_sig_t<__nv_bfloat16>(logits, bias, T_, E, k, G, SG, top_two, renorm, scale,
                                         idx, w, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
