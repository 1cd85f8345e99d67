// C-ABI entry points of libmoe (declared in include/moe.h): host-side validation, workspace
// layout and the launch sequence.  No entry point allocates, frees or synchronises, except
// moe_device_status, whose job is to read the device status word back.
#include <atomic>
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "launch.h"

using namespace moe;

namespace {

constexpr int kMaxE = 1024;
constexpr int64_t kMaxRows = (int64_t)1 << 31;

size_t dtype_size(int dt) { return dt == MOE_F32 ? 4 : (dt == MOE_F16 || dt == MOE_BF16) ? 2 : 0; }
bool valid_dtype(int dt) { return dtype_size(dt) != 0; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

struct Cursor {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  }
};

struct FwdLayout {
  size_t idx, w, ros, tor, offsets, hist, ready, xd, a, total;
};
// counters of the fused short-batch launch: per m-tile (gate/up stored), per (m-tile, down
// n-tile) (y stored), per m-tile (x_d rows gathered), then one flag (row_of_slot written)
size_t ready_bytes(int64_t R, int64_t E, int64_t H) {
  return ((size_t)((R + 127) / 128 + E + 1) * (size_t)(2 + (H + 255) / 256) + 1) * 4;
}

FwdLayout fwd_layout(int64_t T, int64_t E, int64_t H, int64_t I, int k, int ldt, int wdt) {
  const int64_t R = T * k;
  FwdLayout l;
  Cursor c;
  c.take(kWsHeader);
  l.idx = c.take((size_t)R * 4);
  l.w = c.take((size_t)R * dtype_size(ldt));
  l.ros = c.take((size_t)R * 4);
  l.tor = c.take((size_t)R * 4);
  l.offsets = c.take((size_t)(E + 1) * 4);
  l.hist = c.take(dispatch_scratch_bytes(R, (int)E));
  l.ready = c.take(ready_bytes(R, E, H));  // per-m-tile counters of the fused short-batch path
  l.xd = c.take((size_t)R * H * dtype_size(wdt));  // x_d, later reused for y
  l.a = c.take((size_t)R * I * dtype_size(wdt));
  l.total = c.off;
  return l;
}

int check_route_shape(int64_t T, int64_t E, int top_k) {
  if (T < 0 || E < 1 || E > kMaxE || top_k < 1 || top_k > E) return MOE_ERR_SHAPE;
  if (T * top_k >= kMaxRows) return MOE_ERR_SHAPE;
  return MOE_OK;
}

// Conditions of the tensor-core path: 16-byte aligned operands and 16-byte row pitches for TMA.
int check_tc_align(int64_t H, int64_t I, const void* const* ptrs, int n) {
  if (H % 8 != 0 || I % 8 != 0) return MOE_ERR_ALIGN;
  for (int i = 0; i < n; ++i)
    if (!aligned16(ptrs[i])) return MOE_ERR_ALIGN;
  return MOE_OK;
}

int check_experts_shape(int64_t rows, int64_t E, int64_t H, int64_t I) {
  if (rows < 0 || rows >= kMaxRows || E < 1 || E > kMaxE || H < 1 || I < 1) return MOE_ERR_SHAPE;
  if (E * I >= kMaxRows || E * H >= kMaxRows) return MOE_ERR_SHAPE;
  return MOE_OK;
}

int run_experts(const void* x_d, const int32_t* offsets, int64_t rows, const void* gate,
                const void* up, const void* down, int wdt, int64_t E, int64_t H, int64_t I,
                void* y, void* a, unsigned* status, cudaStream_t s, cudaEvent_t between = nullptr) {
  if (wdt == MOE_F32)
    return cuda_status(launch_experts_simt((const float*)x_d, offsets, rows, (const float*)gate,
                                           (const float*)up, (const float*)down, (int)E, (int)H,
                                           (int)I, (float*)y, (float*)a, s, between));
  return cuda_status(launch_experts_tc(x_d, offsets, rows, gate, up, down, wdt, (int)E, (int)H,
                                       (int)I, y, a, status, s, between));
}

int check_sigmoid_args(int64_t T, int64_t E, int top_k, int G, int SG, int top_two, float scale) {
  if (T < 0 || E < 1 || E > kMaxE || G < 1 || G > 128 || E % G != 0) return MOE_ERR_SHAPE;
  if (SG < 1 || SG > G || top_k < 1 || top_k > 64) return MOE_ERR_SHAPE;
  if ((int64_t)top_k > (int64_t)SG * (E / G)) return MOE_ERR_SHAPE;
  if (top_two && E / G < 2) return MOE_ERR_SHAPE;
  if (T * top_k >= kMaxRows) return MOE_ERR_SHAPE;
  if (!(scale > 0.f) || !isfinite(scale)) return MOE_ERR_ARG;
  return MOE_OK;
}

// How a forward routes its tokens: the softmax router of §4 or the sigmoid router of §10.
struct RouteSpec {
  bool sigmoid;
  int renormalize;
  const float* bias;
  int groups, selected_groups, top_two;
  float scale;
};

// Records events[i] on s when an event array is given.
bool record(void* const* events, int i, cudaStream_t s) {
  return !events || cudaEventRecord((cudaEvent_t)events[i], s) == cudaSuccess;
}

// The fused forward: route (softmax or sigmoid), dispatch, experts, combine on one stream.
// Whether moe_forward runs the single-launch fused path (softmax routing, no stage events).
bool takes_fused(const RouteSpec& rs, int64_t T, int64_t E, int64_t H, int64_t I, int top_k,
                 int ldt, int wdt) {
  if (!valid_dtype(ldt) || !valid_dtype(wdt)) return false;
  if (E > kFusedDecodeMaxExperts || H > INT32_MAX || I > INT32_MAX) return false;
  if (!fused_decode_supported(T, (int)E, H, I, top_k, ldt, wdt)) return false;
  // 1: cooperative launch supported, 2: not (per device; relaxed atomics, host threads may race
  // on the first query and every one stores the same value)
  static std::atomic<int> coop[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  int c = coop[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    int v = 0;
    c = (cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && v) ? 1 : 2;
    coop[dev].store(c, std::memory_order_relaxed);
  }
  return c == 1;
}

int run_forward(const void* x, const void* logits, int ldt, const void* gate, const void* up,
                const void* down, int wdt, int64_t T, int64_t E, int64_t H, int64_t I, int top_k,
                const RouteSpec& rs, void* out, void* ws, size_t ws_bytes, cudaStream_t s,
                void* const* events, bool allow_fused) {
  if (!valid_dtype(ldt) || !valid_dtype(wdt)) return MOE_ERR_DTYPE;
  int st = check_experts_shape(T * top_k, E, H, I);
  if (st != MOE_OK) return st;
  if (!gate || !up || !down) return MOE_ERR_NULL;
  if (T == 0) return MOE_OK;
  if (!x || !logits || !out) return MOE_ERR_NULL;
  if (!aligned16(x) || (H * (int64_t)dtype_size(wdt)) % 16 != 0) return MOE_ERR_ALIGN;
  if (wdt != MOE_F32) {
    const void* ptrs[5] = {x, gate, up, down, out};
    st = check_tc_align(H, I, ptrs, 5);
    if (st != MOE_OK) return st;
  }
  const FwdLayout L = fwd_layout(T, E, H, I, top_k, ldt, wdt);
  if (!ws || ((uintptr_t)ws & 255u) != 0 || ws_bytes < L.total) return MOE_ERR_WORKSPACE;

  uint8_t* b = (uint8_t*)ws;
  unsigned* status = (unsigned*)ws;
  uint32_t* idx = (uint32_t*)(b + L.idx);
  void* w = b + L.w;
  uint32_t* ros = (uint32_t*)(b + L.ros);
  uint32_t* tor = (uint32_t*)(b + L.tor);
  int32_t* offsets = (int32_t*)(b + L.offsets);
  int32_t* hist = (int32_t*)(b + L.hist);
  void* xd = b + L.xd;
  void* a = b + L.a;
  const int64_t R = T * top_k;

  if (allow_fused && !events && aligned16(logits) &&
      takes_fused(rs, T, E, H, I, top_k, ldt, wdt)) {
    // status word at byte 0 and grid-barrier counter at byte 64 of the header zeroed here; the
    // tile counter (byte 128) and the per-m-tile counters are zeroed by the kernel
    if (cudaMemsetAsync(ws, 0, 128, s) != cudaSuccess) return MOE_ERR_CUDA;
    FusedDecodeArgs f{};
    f.logits = logits;
    f.x = x;
    f.gate = gate;
    f.up = up;
    f.down = down;
    f.T = T;
    f.E = (int)E;
    f.H = (int)H;
    f.I = (int)I;
    f.k = top_k;
    f.renorm = rs.renormalize != 0;
    f.sigmoid = rs.sigmoid ? 1 : 0;
    f.bias = rs.bias;
    f.G = rs.groups;
    f.SG = rs.selected_groups;
    f.top_two = rs.top_two != 0;
    f.scale = rs.scale;
    f.idx = idx;
    f.w = w;
    f.row_of_slot = ros;
    f.offsets = offsets;
    f.x_d = xd;
    f.a = a;
    f.out = out;
    f.status = status;
    f.grid_count = (unsigned*)(b + 64);
    f.tile_count = (unsigned*)(b + 128);
    f.mtile_ready = (unsigned*)(b + L.ready);
    const cudaError_t ferr = launch_decode_fused(f, ldt, wdt, s);
    if (ferr != cudaErrorCooperativeLaunchTooLarge) return cuda_status(ferr);
    // not all CTAs could be resident (the GPU is shared): the staged launches below instead
    (void)cudaGetLastError();
  }
  if (cudaMemsetAsync(status, 0, sizeof(unsigned), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (!record(events, 0, s)) return MOE_ERR_CUDA;
  cudaError_t err =
      rs.sigmoid
          ? launch_route_sigmoid(logits, ldt, rs.bias, T, (int)E, top_k, rs.groups,
                                 rs.selected_groups, rs.top_two != 0, rs.renormalize != 0,
                                 rs.scale, idx, w, s)
          : launch_route(logits, ldt, T, (int)E, top_k, rs.renormalize != 0, idx, w, s);
  if (err != cudaSuccess || !record(events, 1, s)) return MOE_ERR_CUDA;
  err = launch_dispatch(x, wdt, T, H, idx, (int)E, top_k, xd, offsets, tor, ros, hist, status, s);
  if (err != cudaSuccess || !record(events, 2, s)) return MOE_ERR_CUDA;
  st = run_experts(xd, offsets, R, gate, up, down, wdt, E, H, I, /*y=*/xd, a, status, s,
                   events ? (cudaEvent_t)events[3] : nullptr);
  if (st != MOE_OK || !record(events, 4, s)) return st != MOE_OK ? st : MOE_ERR_CUDA;
  err = launch_combine(xd, wdt, ros, w, ldt, T, H, top_k, out, s);
  if (err != cudaSuccess || !record(events, 5, s)) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return 1; }

const char* moe_status_string(int st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_SHAPE: return "sizes out of range or inconsistent";
    case MOE_ERR_DTYPE: return "dtype not allowed for this argument";
    case MOE_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "a device pipeline wait timed out";
    case MOE_ERR_INDEX: return "an expert index >= E reached dispatch";
    case MOE_ERR_ARG: return "a scalar argument is out of range";
  }
  return "unknown status";
}

int moe_route(const void* logits, int ldt, int64_t T, int64_t E, int top_k, int renormalize,
              uint32_t* idx, void* w, moe_stream_t stream) {
  if (!valid_dtype(ldt)) return MOE_ERR_DTYPE;
  int st = check_route_shape(T, E, top_k);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !w) return MOE_ERR_NULL;
  return cuda_status(launch_route(logits, ldt, T, (int)E, top_k, renormalize != 0, idx, w,
                                  (cudaStream_t)stream));
}

int moe_route_sigmoid_grouped(const void* logits, int ldt, const float* bias, int64_t T,
                              int64_t E, int top_k, int groups, int selected_groups,
                              int group_top_two, int renormalize, float scale, uint32_t* idx,
                              void* w, moe_stream_t stream) {
  if (!valid_dtype(ldt)) return MOE_ERR_DTYPE;
  const int st = check_sigmoid_args(T, E, top_k, groups, selected_groups, group_top_two, scale);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !w) return MOE_ERR_NULL;
  return cuda_status(launch_route_sigmoid(logits, ldt, bias, T, (int)E, top_k, groups,
                                          selected_groups, group_top_two != 0, renormalize != 0,
                                          scale, idx, w, (cudaStream_t)stream));
}

static int check_router_train(int ldt, int idt, int64_t T, int64_t E, int top_k, int scoring,
                              float scale) {
  if (!valid_dtype(ldt)) return MOE_ERR_DTYPE;
  if (idt != MOE_IDX_U32 && idt != MOE_IDX_I32 && idt != MOE_IDX_I64) return MOE_ERR_DTYPE;
  if (scoring != MOE_SCORE_SOFTMAX && scoring != MOE_SCORE_SIGMOID) return MOE_ERR_ARG;
  if (T < 0 || E < 1 || E > kMaxE || top_k < 1 || top_k > 64 || top_k > E) return MOE_ERR_SHAPE;
  if (T * top_k >= kMaxRows || T * E >= ((int64_t)1 << 40)) return MOE_ERR_SHAPE;
  if (!(scale > 0.f) || !isfinite(scale)) return MOE_ERR_ARG;
  return MOE_OK;
}

int moe_selected_router_weights(const void* logits, int ldt, const void* idx, int idt, int64_t T,
                                int64_t E, int top_k, int scoring, int renormalize, float scale,
                                float* w, moe_stream_t stream) {
  const int st = check_router_train(ldt, idt, T, E, top_k, scoring, scale);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !w) return MOE_ERR_NULL;
  return cuda_status(launch_router_train(logits, ldt, idx, idt, nullptr, T, (int)E, top_k,
                                         scoring, renormalize != 0, scale, w, nullptr,
                                         (cudaStream_t)stream));
}

int moe_selected_router_backward(const void* logits, int ldt, const void* idx, int idt,
                                 const float* grad_w, int64_t T, int64_t E, int top_k, int scoring,
                                 int renormalize, float scale, void* grad_logits,
                                 moe_stream_t stream) {
  const int st = check_router_train(ldt, idt, T, E, top_k, scoring, scale);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !grad_w || !grad_logits) return MOE_ERR_NULL;
  return cuda_status(launch_router_train(logits, ldt, idx, idt, grad_w, T, (int)E, top_k, scoring,
                                         renormalize != 0, scale, nullptr, grad_logits,
                                         (cudaStream_t)stream));
}

size_t moe_dispatch_workspace_bytes(int64_t T, int64_t E, int top_k) {
  if (check_route_shape(T, E, top_k) != MOE_OK) return 0;
  return align_up(kWsHeader, 256) + dispatch_scratch_bytes(T * top_k, (int)E);
}

int moe_dispatch(const void* x, int xdt, int64_t T, int64_t H, const uint32_t* idx, int64_t E,
                 int top_k, void* x_d, int32_t* offsets, uint32_t* token_of_row,
                 uint32_t* row_of_slot, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!valid_dtype(xdt)) return MOE_ERR_DTYPE;
  int st = check_route_shape(T, E, top_k);
  if (st != MOE_OK) return st;
  if (H < 1) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!x || !idx || !x_d || !offsets || !token_of_row || !row_of_slot) return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(x_d) || (H * (int64_t)dtype_size(xdt)) % 16 != 0)
    return MOE_ERR_ALIGN;
  if (!ws || !aligned16(ws) || ws_bytes < moe_dispatch_workspace_bytes(T, E, top_k))
    return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned* status = (unsigned*)ws;
  cudaError_t err = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* hist = (int32_t*)((uint8_t*)ws + align_up(kWsHeader, 256));
  return cuda_status(launch_dispatch(x, xdt, T, H, idx, (int)E, top_k, x_d, offsets,
                                     token_of_row, row_of_slot, hist, status, s));
}

int moe_dispatch_static(const void* x, int xdt, int64_t T, int64_t H, const uint32_t* idx,
                        int64_t E, int top_k, void* x_d, int32_t* offsets, uint32_t* token_of_row,
                        uint32_t* row_of_slot, moe_stream_t stream) {
  if (!valid_dtype(xdt)) return MOE_ERR_DTYPE;
  int st = check_route_shape(T, E, top_k);
  if (st != MOE_OK) return st;
  if (H < 1) return MOE_ERR_SHAPE;
  if (moe_dispatch_workspace_bytes(T, E, top_k) > kStaticDispatchScratchBytes) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!x || !idx || !x_d || !offsets || !token_of_row || !row_of_slot) return MOE_ERR_NULL;
  if (!aligned16(x) || !aligned16(x_d) || (H * (int64_t)dtype_size(xdt)) % 16 != 0)
    return MOE_ERR_ALIGN;
  void* scratch = nullptr;
  if (static_dispatch_scratch(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned* status = (unsigned*)scratch;  // the count kernel ORs into it: clear it first
  if (cudaMemsetAsync(status, 0, sizeof(unsigned), s) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* hist = (int32_t*)((uint8_t*)scratch + align_up(kWsHeader, 256));
  return cuda_status(launch_dispatch(x, xdt, T, H, idx, (int)E, top_k, x_d, offsets,
                                     token_of_row, row_of_slot, hist, status, s));
}

size_t moe_experts_workspace_bytes(int64_t rows, int64_t E, int64_t H, int64_t I, int wdt) {
  if (!valid_dtype(wdt) || check_experts_shape(rows, E, H, I) != MOE_OK) return 0;
  return align_up(kWsHeader, 256) + align_up((size_t)rows * I * dtype_size(wdt), 256);
}

int moe_experts_forward_dispatched(const void* x_d, const int32_t* offsets, int64_t rows,
                                   const void* gate, const void* up, const void* down, int wdt,
                                   int64_t E, int64_t H, int64_t I, void* y, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  if (!valid_dtype(wdt)) return MOE_ERR_DTYPE;
  int st = check_experts_shape(rows, E, H, I);
  if (st != MOE_OK) return st;
  if (!gate || !up || !down) return MOE_ERR_NULL;
  if (rows == 0) return MOE_OK;
  if (!x_d || !offsets || !y) return MOE_ERR_NULL;
  if (!ws || ((uintptr_t)ws & 255u) != 0 ||
      ws_bytes < moe_experts_workspace_bytes(rows, E, H, I, wdt))
    return MOE_ERR_WORKSPACE;
  void* a = (uint8_t*)ws + align_up(kWsHeader, 256);
  if (wdt != MOE_F32) {
    const void* ptrs[5] = {x_d, gate, up, down, y};
    st = check_tc_align(H, I, ptrs, 5);
    if (st != MOE_OK) return st;
  }
  cudaStream_t s = (cudaStream_t)stream;
  unsigned* status = (unsigned*)ws;
  if (cudaMemsetAsync(status, 0, sizeof(unsigned), s) != cudaSuccess) return MOE_ERR_CUDA;
  return run_experts(x_d, offsets, rows, gate, up, down, wdt, E, H, I, y, a, status, s);
}

int moe_combine(const void* y, int ydt, const uint32_t* row_of_slot, const void* w, int wdt,
                int64_t T, int64_t H, int top_k, void* out, moe_stream_t stream) {
  if (!valid_dtype(ydt) || !valid_dtype(wdt)) return MOE_ERR_DTYPE;
  if (T < 0 || H < 1 || top_k < 1 || top_k > kMaxE || T * top_k >= kMaxRows) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!y || !row_of_slot || !w || !out) return MOE_ERR_NULL;
  return cuda_status(launch_combine(y, ydt, row_of_slot, w, wdt, T, H, top_k, out,
                                    (cudaStream_t)stream));
}

size_t moe_forward_workspace_bytes(int64_t T, int64_t E, int64_t H, int64_t I, int top_k,
                                   int ldt, int wdt) {
  if (!valid_dtype(ldt) || !valid_dtype(wdt)) return 0;
  if (check_route_shape(T, E, top_k) != MOE_OK || check_experts_shape(T * top_k, E, H, I) != MOE_OK)
    return 0;
  return fwd_layout(T, E, H, I, top_k, ldt, wdt).total;
}

int moe_forward(const void* x, const void* logits, int ldt, const void* gate, const void* up,
                const void* down, int wdt, int64_t T, int64_t E, int64_t H, int64_t I, int top_k,
                int renormalize, void* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  const int st = check_route_shape(T, E, top_k);
  if (st != MOE_OK) return st;
  const RouteSpec r{false, renormalize, nullptr, 1, 1, 0, 1.f};
  return run_forward(x, logits, ldt, gate, up, down, wdt, T, E, H, I, top_k, r, out, ws, ws_bytes,
                     (cudaStream_t)stream, nullptr, /*allow_fused=*/true);
}

int moe_wait_selftest(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws) return MOE_ERR_NULL;
  if (((uintptr_t)ws & 255u) != 0 || ws_bytes < kWsHeader) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_wait_selftest((unsigned*)ws, (cudaStream_t)stream));
}

int moe_forward_fused(int64_t T, int64_t E, int64_t H, int64_t I, int top_k, int ldt, int wdt) {
  if (check_route_shape(T, E, top_k) != MOE_OK || check_experts_shape(T * top_k, E, H, I) != MOE_OK)
    return 0;
  const RouteSpec r{false, 1, nullptr, 1, 1, 0, 1.f};
  return takes_fused(r, T, E, H, I, top_k, ldt, wdt) ? 1 : 0;
}

int moe_forward_with_events(const void* x, const void* logits, int ldt, const void* gate,
                            const void* up, const void* down, int wdt, int64_t T, int64_t E,
                            int64_t H, int64_t I, int top_k, int renormalize, void* out, void* ws,
                            size_t ws_bytes, moe_stream_t stream, void* const* events) {
  const int st = check_route_shape(T, E, top_k);
  if (st != MOE_OK) return st;
  const RouteSpec r{false, renormalize, nullptr, 1, 1, 0, 1.f};
  return run_forward(x, logits, ldt, gate, up, down, wdt, T, E, H, I, top_k, r, out, ws, ws_bytes,
                     (cudaStream_t)stream, events, /*allow_fused=*/false);
}

int moe_forward_sigmoid_grouped(const void* x, const void* logits, int ldt, const float* bias,
                                const void* gate, const void* up, const void* down, int wdt,
                                int64_t T, int64_t E, int64_t H, int64_t I, int top_k, int groups,
                                int selected_groups, int group_top_two, int renormalize,
                                float scale, void* out, void* ws, size_t ws_bytes,
                                moe_stream_t stream) {
  if (!valid_dtype(ldt)) return MOE_ERR_DTYPE;
  const int st = check_sigmoid_args(T, E, top_k, groups, selected_groups, group_top_two, scale);
  if (st != MOE_OK) return st;
  const RouteSpec r{true, renormalize, bias, groups, selected_groups, group_top_two, scale};
  return run_forward(x, logits, ldt, gate, up, down, wdt, T, E, H, I, top_k, r, out, ws, ws_bytes,
                     (cudaStream_t)stream, nullptr, /*allow_fused=*/true);
}

int moe_combine_backward(const void* y, int ydt, const uint32_t* row_of_slot, const void* w,
                         int wdt, const void* dout, int64_t T, int64_t H, int top_k,
                         void* dexpert, float* dweights, moe_stream_t stream) {
  if (!valid_dtype(ydt) || !valid_dtype(wdt)) return MOE_ERR_DTYPE;
  if (T < 0 || H < 1 || top_k < 1 || top_k > kMaxE || T * top_k >= kMaxRows) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!y || !row_of_slot || !w || !dout || !dexpert || !dweights) return MOE_ERR_NULL;
  return cuda_status(launch_combine_backward(y, ydt, row_of_slot, w, wdt, dout, T, H, top_k,
                                             dexpert, dweights, (cudaStream_t)stream));
}

size_t moe_experts_backward_workspace_bytes(int64_t rows, int64_t I) {
  if (rows < 0 || rows >= kMaxRows || I < 1) return 0;
  const size_t simt = experts_backward_scratch_bytes(rows, I);
  const size_t tc = experts_backward_tc_scratch_bytes(rows, I);
  return align_up(kWsHeader, 256) + align_up(simt > tc ? simt : tc, 256);
}

int moe_experts_backward(const void* x_d, const int32_t* offsets, int64_t rows, const void* gate,
                         const void* up, const void* down, int wdt, int64_t E, int64_t H,
                         int64_t I, const void* dy, void* dinput, float* dgate, float* dup,
                         float* ddown, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!valid_dtype(wdt)) return MOE_ERR_DTYPE;
  const int st = check_experts_shape(rows, E, H, I);
  if (st != MOE_OK) return st;
  if (!gate || !up || !down || !dgate || !dup || !ddown) return MOE_ERR_NULL;
  if (rows > 0 && (!x_d || !offsets || !dy || !dinput)) return MOE_ERR_NULL;
  if (!ws || ((uintptr_t)ws & 255u) != 0 || ws_bytes < moe_experts_backward_workspace_bytes(rows, I))
    return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  if (rows == 0) {  // no rows: every weight gradient is zero
    const size_t n = (size_t)E * H * I * sizeof(float);
    if (cudaMemsetAsync(dgate, 0, n, s) != cudaSuccess || cudaMemsetAsync(dup, 0, n, s) != cudaSuccess ||
        cudaMemsetAsync(ddown, 0, n, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  float* scratch = (float*)((uint8_t*)ws + align_up(kWsHeader, 256));
  unsigned* status = (unsigned*)ws;
  if (cudaMemsetAsync(status, 0, sizeof(unsigned), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (wdt != MOE_F32 && I % 64 == 0) {
    const void* ptrs[8] = {x_d, gate, up, down, dy, dinput, dgate, ddown};
    if (check_tc_align(H, I, ptrs, 8) == MOE_OK && aligned16(dup))
      return cuda_status(launch_experts_backward_tc(x_d, offsets, rows, gate, up, down, wdt,
                                                    (int)E, (int)H, (int)I, dy, dinput, dgate,
                                                    dup, ddown, scratch, status, s));
  }
  return cuda_status(launch_experts_backward(x_d, offsets, rows, gate, up, down, wdt, (int)E,
                                             (int)H, (int)I, dy, dinput, dgate, dup, ddown,
                                             scratch, s));
}

int moe_dispatch_backward(const void* dinput, int dt, const uint32_t* row_of_slot, int64_t T,
                          int64_t H, int top_k, void* dx, moe_stream_t stream) {
  if (!valid_dtype(dt)) return MOE_ERR_DTYPE;
  if (T < 0 || H < 1 || top_k < 1 || top_k > kMaxE || T * top_k >= kMaxRows) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!dinput || !row_of_slot || !dx) return MOE_ERR_NULL;
  return cuda_status(launch_dispatch_backward(dinput, dt, row_of_slot, T, H, top_k, dx,
                                              (cudaStream_t)stream));
}

int moe_device_status(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || ws_bytes < sizeof(unsigned)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(ws, 0, sizeof(unsigned)) != cudaSuccess) return MOE_ERR_CUDA;
  if (v & kStatusTimeout) return MOE_ERR_TIMEOUT;
  if (v & kStatusIndex) return MOE_ERR_INDEX;
  return MOE_OK;
}

}  // extern "C"
