// Router weights of a fixed selection and their logits gradient: selected_router_weights /
// selected_router_backward of the ruDNN user guide, §12 "MoE-Training erster Ordnung".
//
// For row t and slot j with expert i_j: q_j = p[i_j], where p is the softmax over all E experts
// (FP32) or the sigmoid of the logit.  w_j = scale * q_j, or scale * q_j / Z with Z = sum_j q_j
// when renormalising.  Repeated indices gather the same q; an index outside [0, E) makes the
// whole row NaN and is never dereferenced.  The backward maps dL/dw [T, k] (FP32) to dL/dlogits
// [T, E] in the logits dtype, differentiating the continuous weights of the fixed selection:
//   softmax, plain : dl_e = scale * p_e * (G_e - sum_j g_j q_j)
//   softmax, renorm: dl_e = scale * (GR_e - n_e * (p_e / Z) * sum_j g_j q_j / Z)
//   sigmoid, plain : dl_e = scale * s_e (1 - s_e) * G_e
//   sigmoid, renorm: dl_e = scale * s_e (1 - s_e) / Z * (G_e - n_e * sum_j g_j q_j / Z)
// with G_e = sum of g_j over slots holding e, GR_e the same sum of g_j q_j / Z, n_e their count.
// One warp per row; the per-expert slot sums are accumulated in shared memory by one lane in
// slot order, so the result does not depend on thread timing.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int kRtWarps = 4;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ int64_t load_index(const void* idx, int idt, int64_t pos) {
  switch (idt) {
    case MOE_IDX_U32: return (int64_t)((const uint32_t*)idx)[pos];
    case MOE_IDX_I32: return (int64_t)((const int32_t*)idx)[pos];
    default: return ((const int64_t*)idx)[pos];
  }
}

// Per-row state shared by the forward and the backward.
struct RowScores {
  float m, S;       // softmax max and sum over all experts (softmax scoring)
  bool poisoned;    // softmax: NaN / +inf / only -inf in the row
};

template <typename T>
__device__ RowScores softmax_stats(const T* row, int E, int lane) {
  float m = -INFINITY;
  bool bad = false, finite_seen = false;
  for (int e = lane; e < E; e += 32) {
    const float x = Dt<T>::to_f(row[e]);
    bad |= (x != x) || x == INFINITY;
    finite_seen |= x != -INFINITY;
    m = fmaxf(m, x);
  }
  m = warp_max(m);
  bad = __any_sync(0xFFFFFFFFu, bad) || !__any_sync(0xFFFFFFFFu, finite_seen);
  float S = 0.f;
  if (!bad)
    for (int e = lane; e < E; e += 32) S += expf(Dt<T>::to_f(row[e]) - m);
  S = warp_sum(S);
  return {m, S, bad};
}

template <typename T>
__device__ __forceinline__ float score(const T* row, int e, int sigmoid_scoring, const RowScores& rs) {
  const float x = Dt<T>::to_f(row[e]);
  return sigmoid_scoring ? 1.f / (1.f + expf(-x)) : expf(x - rs.m) / rs.S;
}

template <typename T, bool BACKWARD>
__global__ void __launch_bounds__(kRtWarps * 32)
    moe_router_train_kernel(const T* __restrict__ logits, const void* __restrict__ idx, int idt,
                            const float* __restrict__ grad_w, int64_t T_, int E, int k,
                            int sigmoid_scoring, int renorm, float scale, float* __restrict__ w_out,
                            T* __restrict__ grad_out) {
  extern __shared__ float rt_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t t = (int64_t)blockIdx.x * kRtWarps + warp;
  if (t >= T_) return;  // whole warp
  const T* row = logits + t * (int64_t)E;

  // slots j = lane and lane + 32 (k <= 64)
  int64_t id[2];
  bool invalid = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = lane + 32 * h;
    id[h] = j < k ? load_index(idx, idt, t * k + j) : 0;
    if (j < k && (id[h] < 0 || id[h] >= E)) invalid = true;
  }
  invalid = __any_sync(0xFFFFFFFFu, invalid);
  RowScores rs{0.f, 1.f, false};
  if (!sigmoid_scoring) rs = softmax_stats(row, E, lane);
  const bool nan_row = invalid || rs.poisoned;

  float q[2] = {0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (lane + 32 * h < k && !nan_row) q[h] = score(row, (int)id[h], sigmoid_scoring, rs);
  const float Z = warp_sum(q[0] + q[1]);

  if (!BACKWARD) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = lane + 32 * h;
      if (j < k)
        w_out[t * k + j] = nan_row ? __int_as_float(0x7FC00000)
                                   : (renorm ? q[h] / Z : q[h]) * scale;
    }
    return;
  }

  T* gout = grad_out + t * (int64_t)E;
  if (nan_row) {
    for (int e = lane; e < E; e += 32) gout[e] = Dt<T>::from_f(__int_as_float(0x7FC00000));
    return;
  }
  float g[2] = {0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (lane + 32 * h < k) g[h] = grad_w[t * k + lane + 32 * h];
  const float A = warp_sum(g[0] * q[0] + g[1] * q[1]);  // sum_j g_j q_j

  // per-expert slot sums: acc[e] = sum over slots holding e of g_j (or g_j q_j / Z), cnt[e]
  float* acc = rt_smem + (size_t)warp * 2 * E;
  float* cnt = acc + E;
  for (int e = lane; e < E; e += 32) {
    acc[e] = 0.f;
    cnt[e] = 0.f;
  }
  __syncwarp();
  const bool weighted = renorm && !sigmoid_scoring;
  for (int j = 0; j < k; ++j) {  // slot order, one lane: deterministic sums
    const int h = j >> 5, src = j & 31;
    const float gj = __shfl_sync(0xFFFFFFFFu, h ? g[1] : g[0], src);
    const float qj = __shfl_sync(0xFFFFFFFFu, h ? q[1] : q[0], src);
    const int ej = (int)__shfl_sync(0xFFFFFFFFu, (int)(h ? id[1] : id[0]), src);
    if (lane == 0) {
      acc[ej] += weighted ? gj * qj / Z : gj;
      cnt[ej] += 1.f;
    }
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) {
    const float x = Dt<T>::to_f(row[e]);
    float d;
    if (!sigmoid_scoring) {
      const float p = expf(x - rs.m) / rs.S;
      d = renorm ? acc[e] - cnt[e] * (p / Z) * (A / Z) : p * (acc[e] - A);
    } else {
      const float s = 1.f / (1.f + expf(-x));
      const float ds = s * (1.f - s);
      d = renorm ? ds / Z * (acc[e] - cnt[e] * A / Z) : ds * acc[e];
    }
    gout[e] = Dt<T>::from_f(d * scale);
  }
}

template <typename T>
cudaError_t launch_rt(const void* logits, const void* idx, int idt, const float* grad_w,
                      int64_t T_, int E, int k, int scoring, int renorm, float scale, float* w,
                      void* grad, cudaStream_t s) {
  const unsigned blocks = (unsigned)((T_ + kRtWarps - 1) / kRtWarps);
  if (grad_w == nullptr) {
    moe_router_train_kernel<T, false><<<blocks, kRtWarps * 32, 0, s>>>(
        (const T*)logits, idx, idt, nullptr, T_, E, k, scoring, renorm, scale, w, nullptr);
  } else {
    const size_t smem = (size_t)kRtWarps * 2 * E * sizeof(float);
    moe_router_train_kernel<T, true><<<blocks, kRtWarps * 32, smem, s>>>(
        (const T*)logits, idx, idt, grad_w, T_, E, k, scoring, renorm, scale, nullptr, (T*)grad);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_train(const void* logits, int ldt, const void* idx, int idt,
                                const float* grad_w, int64_t T_, int E, int k, int scoring,
                                int renorm, float scale, float* w, void* grad, cudaStream_t s) {
  switch (ldt) {
    case MOE_F32:
      return launch_rt<float>(logits, idx, idt, grad_w, T_, E, k, scoring, renorm, scale, w, grad, s);
    case MOE_F16:
      return launch_rt<__half>(logits, idx, idt, grad_w, T_, E, k, scoring, renorm, scale, w, grad, s);
    case MOE_BF16:
      return launch_rt<__nv_bfloat16>(logits, idx, idt, grad_w, T_, E, k, scoring, renorm, scale,
                                      w, grad, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
