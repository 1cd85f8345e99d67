// Internal launchers of libmoe (not part of the C ABI).  Each returns the CUDA error of its
// launches; arguments are validated by the entry points in api.cu before these run.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

// Capacity of moe_dispatch_static()'s file-scope scratch: 256-byte status header + histograms.
constexpr size_t kStaticDispatchScratchBytes = 256 + (1u << 20);

namespace moe {

// status word bits (device side), reported by moe_device_status()
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusIndex = 2u;

cudaError_t launch_route(const void* logits, int ldt, int64_t T, int E, int k, int renorm,
                         uint32_t* idx, void* w, cudaStream_t s);

// Group-limited sigmoid routing (float64 selection); bias may be null.
cudaError_t launch_route_sigmoid(const void* logits, int ldt, const float* bias, int64_t T, int E,
                                 int k, int G, int SG, int top_two, int renorm, float scale,
                                 uint32_t* idx, void* w, cudaStream_t s);

// Fixed-selection router weights (grad_w == nullptr) or their logits gradient.
cudaError_t launch_router_train(const void* logits, int ldt, const void* idx, int idt,
                                const float* grad_w, int64_t T, int E, int k, int scoring,
                                int renorm, float scale, float* w, void* grad, cudaStream_t s);

// Backward chain (FP32 CUDA-core GEMMs for the experts).
size_t experts_backward_scratch_bytes(int64_t rows, int64_t I);
cudaError_t launch_experts_backward(const void* x_d, const int32_t* offsets, int64_t rows,
                                    const void* gate, const void* up, const void* down, int wdt,
                                    int E, int H, int I, const void* dy, void* dinput,
                                    float* dgate, float* dup, float* ddown, float* scratch,
                                    cudaStream_t s);
// bf16 / f16 expert backward on tensor cores (H % 8 == 0, I % 64 == 0, 16-byte aligned operands);
// scratch of experts_backward_tc_scratch_bytes(rows, I) bytes, 256-byte aligned.
size_t experts_backward_tc_scratch_bytes(int64_t rows, int64_t I);
cudaError_t launch_experts_backward_tc(const void* x_d, const int32_t* offsets, int64_t rows,
                                       const void* gate, const void* up, const void* down,
                                       int wdt, int E, int H, int I, const void* dy, void* dinput,
                                       float* dgate, float* dup, float* ddown, void* scratch,
                                       unsigned* status, cudaStream_t s);
cudaError_t launch_combine_backward(const void* y, int ydt, const uint32_t* ros, const void* w,
                                    int wdt, const void* dout, int64_t T, int64_t H, int k,
                                    void* dexpert, float* dweights, cudaStream_t s);
cudaError_t launch_dispatch_backward(const void* dinput, int dt, const uint32_t* ros, int64_t T,
                                     int64_t H, int k, void* dx, cudaStream_t s);

// Dispatch splits the R = T*k slots into W contiguous chunks of CH slots, one per warp.
struct DispatchPlan {
  int W;   // chunks (warps)
  int CH;  // slots per chunk, a multiple of 32
};
DispatchPlan dispatch_plan(int64_t R);
size_t dispatch_scratch_bytes(int64_t R, int E);  // per-chunk histograms
cudaError_t launch_dispatch(const void* x, int xdt, int64_t T, int64_t H, const uint32_t* idx,
                            int E, int k, void* x_d, int32_t* offsets, uint32_t* token_of_row,
                            uint32_t* row_of_slot, int32_t* hist, unsigned* status,
                            cudaStream_t s);

// One bounded mbarrier wait that nothing completes: sets kStatusTimeout in *status after ~1 s.
cudaError_t launch_wait_selftest(unsigned* status, cudaStream_t s);

// Device address of that scratch on the current device (looked up on first use per device).
cudaError_t static_dispatch_scratch(void** ptr);

// The id of the calling thread's current CUDA context, unique for the life of the process (0 when
// none is current or the driver entry points are unavailable).
unsigned long long current_context_id();

cudaError_t launch_combine(const void* y, int ydt, const uint32_t* row_of_slot, const void* w,
                           int wdt, int64_t T, int64_t H, int k, void* out, cudaStream_t s);

// f32 experts on CUDA cores; `a` is an [rows, I] f32 scratch buffer.
cudaError_t launch_experts_simt(const float* x_d, const int32_t* offsets, int64_t rows,
                                const float* gate, const float* up, const float* down, int E,
                                int H, int I, float* y, float* a, cudaStream_t s,
                                cudaEvent_t between = nullptr);

// Fused forward of short batches (route, dispatch, gate/up, down, combine in one cooperative
// launch).  fused_decode_supported() says whether moe_forward takes it for a shape; pointer
// alignment (16 bytes) is checked by the caller.  grid_count must be zero at launch.
constexpr int kFusedDecodeMaxExperts = 256;
constexpr int64_t kFusedDecodeMaxRows = 4096;
struct FusedDecodeArgs {
  const void* logits;
  const void* x;
  const void* gate;
  const void* up;
  const void* down;
  int64_t T;
  int E, H, I, k, renorm;
  // group-limited sigmoid routing instead of the softmax (bias may be null)
  int sigmoid;
  const float* bias;
  int G, SG, top_two;
  float scale;
  uint32_t* idx;
  void* w;
  uint32_t* row_of_slot;
  int32_t* offsets;
  void* x_d;
  void* a;
  void* out;
  unsigned* status;
  unsigned* grid_count;   // zero at launch
  unsigned* tile_count;   // zeroed by the kernel
  unsigned* mtile_ready;  // (ceil(T k / 128) + E + 1) x (1 + ceil(H / 256)) counters, zeroed by
                          // the kernel
};
bool fused_decode_supported(int64_t T, int E, int64_t H, int64_t I, int k, int ldt, int wdt);
cudaError_t launch_decode_fused(const FusedDecodeArgs& f, int ldt, int wdt, cudaStream_t s);

// bf16 / f16 experts on tcgen05 tensor cores; `a` is an [rows, I] scratch buffer of dtype wdt.
// Steps 1-3 of the tensor-core expert backward on CTA pairs (256-row tiles, cta_group::2): da =
// dy down_e (FP32), g and u recomputed with the SwiGLU gradient (dg | du and a in the layer dtype),
// dinput = [dg du] [gate_e; up_e].  For experts averaging at least 128 rows; I % 64 == 0.
cudaError_t launch_experts_bwd_pair(const void* x_d, const int32_t* offsets, int64_t rows,
                                    const void* gate, const void* up, const void* down, int wdt,
                                    int E, int H, int I, const void* dy, float* da, void* dgdu,
                                    void* a, void* dinput, unsigned* status, cudaStream_t s);
cudaError_t launch_experts_tc(const void* x_d, const int32_t* offsets, int64_t rows,
                              const void* gate, const void* up, const void* down, int wdt, int E,
                              int H, int I, void* y, void* a, unsigned* status, cudaStream_t s,
                              cudaEvent_t between = nullptr);

}  // namespace moe
