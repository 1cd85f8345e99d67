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
// The selection (sigmoid, correction, group scores, ranking) is the decision float64 arithmetic
// makes, as in the float64 reference.  One warp owns a row: lane i holds experts i, i + 32, ...;
// the group and expert choices are rounds of warp argmax over (score, -id) pairs.  Each row is
// first decided in FP32 (accurate expf, IEEE division): with the FP32 error of every corrected
// score bounded by E_c = 5e-7 + 1.2e-7 max|c| (expf within 2 ulp, the division and the additions
// rounded once each), the FP32 choice is the float64 choice whenever every margin it rests on --
// last chosen group vs the best other group, each chosen expert vs the next one, the k-th vs the
// best unchosen candidate -- exceeds twice the bound on the two scores compared.  Those rows take
// their k weights from float64 sigmoids of the chosen experts; every other row (a near or exact
// tie, a NaN or infinite score) is decided again entirely in float64.  Either way the indices
// and weights are the float64 path's.
#include "common.cuh"
#include "launch.h"
#include "route_sigmoid_core.cuh"

namespace moe {
namespace {

constexpr int kSigWarps = 4;

template <typename T, int C>
__global__ void __launch_bounds__(kSigWarps * 32)
    moe_route_sigmoid_kernel(const T* __restrict__ logits, const float* __restrict__ bias,
                             int64_t T_, int E, int k, int G, int SG, int top_two, int renorm,
                             float scale, uint32_t* __restrict__ idx_out, T* __restrict__ w_out) {
  extern __shared__ double sig_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * kSigWarps + warp;
  if (row >= T_) return;  // whole warp leaves together
  sigmoid_route_row<T, C>(logits + row * (int64_t)E, bias, row, E, k, G, SG, top_two, renorm,
                          scale, sig_smem + (size_t)warp * (E + 128 + 64 + 32), lane, idx_out,
                          w_out);
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
