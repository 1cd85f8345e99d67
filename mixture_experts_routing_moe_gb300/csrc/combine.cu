// Combine: DispatchedTokens::combine of the ruDNN user guide, §3 "MoE-Workflow" / §6 "MoE aufrufen".
//
// out[t] = sum_{j=0..k-1} w[t, j] * y[row_of_slot[t*k + j]], FP32 accumulation in the fixed slot
// order j = 0..k-1 (no atomics: the result is the same bits on every run), rounded once to the
// output dtype.  A token is spread over ceil(H / (32 * 16-byte chunk)) warps, one 16-byte column
// chunk per lane, so short batches still fill the GPU; each warp loads the token's k
// (row, weight) pairs through its lanes and broadcasts them with shuffles.
#include "combine_core.cuh"
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int kCombWarps = 8;

template <typename TY, typename TW, bool VEC>
__global__ void __launch_bounds__(kCombWarps * 32)
    moe_combine_kernel(const TY* __restrict__ y, const uint32_t* __restrict__ row_of_slot,
                       const TW* __restrict__ w, int64_t T, int64_t H, int k,
                       int64_t warps_per_token, TY* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * kCombWarps + (threadIdx.x >> 5);
  const int64_t t = gw / warps_per_token;
  if (t >= T) return;
  combine_warp<TY, TW, VEC, false, 2>(y, row_of_slot, w, t, H, k, gw - t * warps_per_token, out,
                                      lane);
}

template <typename TY, typename TW>
cudaError_t launch_combine_t(const void* y, const uint32_t* ros, const void* w, int64_t T,
                             int64_t H, int k, void* out, cudaStream_t s) {
  const bool vec = ((uintptr_t)y % 16 == 0) && ((uintptr_t)out % 16 == 0) &&
                   ((H * (int64_t)sizeof(TY)) % 16 == 0);
  const int64_t chunks = vec ? H * (int64_t)sizeof(TY) / 16 : H;
  const int64_t wpt = (chunks + 31) / 32;  // warps per token: one column chunk per lane
  const unsigned blocks = (unsigned)((T * wpt + kCombWarps - 1) / kCombWarps);
  if (vec)
    moe_combine_kernel<TY, TW, true><<<blocks, kCombWarps * 32, 0, s>>>(
        (const TY*)y, ros, (const TW*)w, T, H, k, wpt, (TY*)out);
  else
    moe_combine_kernel<TY, TW, false><<<blocks, kCombWarps * 32, 0, s>>>(
        (const TY*)y, ros, (const TW*)w, T, H, k, wpt, (TY*)out);
  return cudaGetLastError();
}

template <typename TY>
cudaError_t launch_combine_y(const void* y, const uint32_t* ros, const void* w, int wdt,
                             int64_t T, int64_t H, int k, void* out, cudaStream_t s) {
  switch (wdt) {
    case MOE_F32: return launch_combine_t<TY, float>(y, ros, w, T, H, k, out, s);
    case MOE_F16: return launch_combine_t<TY, __half>(y, ros, w, T, H, k, out, s);
    case MOE_BF16: return launch_combine_t<TY, __nv_bfloat16>(y, ros, w, T, H, k, out, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_combine(const void* y, int ydt, const uint32_t* row_of_slot, const void* w,
                           int wdt, int64_t T, int64_t H, int k, void* out, cudaStream_t s) {
  switch (ydt) {
    case MOE_F32: return launch_combine_y<float>(y, row_of_slot, w, wdt, T, H, k, out, s);
    case MOE_F16: return launch_combine_y<__half>(y, row_of_slot, w, wdt, T, H, k, out, s);
    case MOE_BF16:
      return launch_combine_y<__nv_bfloat16>(y, row_of_slot, w, wdt, T, H, k, out, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
