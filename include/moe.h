/*
 * moe.h — C ABI of libmoe: the local Mixture-of-Experts forward on one GB300 (sm_103a).
 *
 * The operation is the MoE sequence of the ruDNN user guide (docs.rs, ruDNN 0.1.72,
 * docs/de/README.md), §3 "MoE-Workflow": router logits -> softmax / top-k -> compact dispatch ->
 * bias-free SwiGLU experts -> weighted combine that restores token order.  Each entry point below
 * is one stage of §6 "MoE aufrufen" (route, RoutingPlan::dispatch, forward_dispatched, combine)
 * or the whole forward.
 *
 * Conventions shared by every entry point
 *  - Buffers are DEVICE pointers owned by the caller, contiguous and row-major.  The library never
 *    allocates device memory, frees or synchronises on these paths; scratch memory comes from the
 *    caller through (ws, ws_bytes), sized by the matching *_workspace_bytes() query.  (The one
 *    other resource: moe_experts_backward keeps a second stream per device and creates two
 *    events per call, see there.)
 *  - Work is enqueued on the caller's stream `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  Every call returns as soon as the work is enqueued.
 *  - Every argument is checked on the host before anything is enqueued; a rejected call enqueues
 *    nothing and returns the status below.  T = 0 is valid and enqueues nothing.
 *  - MOE_ERR_CUDA means a CUDA launch or query failed (including "no device").
 *  - Kernels never trap.  Conditions only the device can see (an expert index >= E handed to
 *    moe_dispatch; a pipeline wait in the tensor-core kernels that exceeded its time limit) are
 *    recorded in a status word at the start of the workspace; moe_device_status() reads it.
 *    The workspace's first 256 bytes are the library's own (the status word and counters the
 *    kernels of one call use, e.g. the tile-claim counter of the tensor-core grouped GEMMs); one
 *    workspace therefore serves one call in flight at a time.
 *  - dtype codes: MOE_F32, MOE_F16, MOE_BF16 (unquantised, as §4 "Routing-Vertrag" requires).
 *  - Limits: 1 <= top_k <= E <= 1024; T * top_k < 2^31; H, I >= 1.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL = 1,      /* a required pointer is NULL                                  */
  MOE_ERR_SHAPE = 2,     /* sizes out of range or inconsistent (incl. top_k > E)        */
  MOE_ERR_DTYPE = 3,     /* dtype code unknown or not allowed for this argument          */
  MOE_ERR_ALIGN = 4,     /* pointer or row pitch breaks the 16-byte rule of the kernels   */
  MOE_ERR_WORKSPACE = 5, /* ws is NULL, misaligned or smaller than the query result       */
  MOE_ERR_CUDA = 6,      /* CUDA runtime / launch error                                   */
  MOE_ERR_TIMEOUT = 7,   /* (device status only) a pipeline wait exceeded its time limit  */
  MOE_ERR_INDEX = 8,     /* (device status only) an expert index >= E reached dispatch    */
  MOE_ERR_ARG = 9        /* a scalar argument is out of range (e.g. scale not finite > 0)  */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_F16 = 1, MOE_BF16 = 2 } moe_dtype;
typedef enum { MOE_IDX_U32 = 0, MOE_IDX_I32 = 1, MOE_IDX_I64 = 2 } moe_index_dtype;
typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_scoring;

/* Static text for a status code (never NULL). */
const char* moe_status_string(int status);

/* ABI version of this header (bumped on any signature change). */
int moe_abi_version(void);

/*
 * moe_route — route(logits, RoutingOptions{top_k, renormalize}) of §3/§4 "Routing-Vertrag".
 *
 * logits  [T, E] in dtype `ldt` (f32 / f16 / bf16).
 * idx     [T, top_k] uint32 out: selected experts, ordered by descending weight; equal logits
 *         give the lower expert id first.  Selection ranks experts by their logit (the ranking
 *         of the exact softmax).
 * w       [T, top_k] out, dtype `ldt`: p_e = exp(l_e - max) / sum_all exp(l - max) computed in
 *         FP32 over all E experts; with renormalize != 0 the selected p are divided by their sum;
 *         then cast (round-to-nearest-even) to `ldt`.
 * Rows holding a NaN, a +inf, or only -inf get NaN weights and indices 0..top_k-1 (they are
 * still dispatched; nothing is dropped).
 * Alignment: none required (16-byte aligned rows take a vectorised path).
 */
int moe_route(const void* logits, int ldt, int64_t T, int64_t E, int top_k, int renormalize,
              uint32_t* idx, void* w, moe_stream_t stream);

/*
 * moe_route_sigmoid_grouped — route_sigmoid_grouped(logits, bias, GroupRoutingOptions) of §10
 * "Gruppenbeschränktes Sigmoid-MoE-Routing".
 *
 * s = sigmoid(logit); c = s + bias[e] (bias: FP32 [E] device pointer, or NULL for none; it changes
 * the selection only).  The E experts form `groups` contiguous groups of E / groups; a group's
 * score is its largest c, or with group_top_two != 0 the sum of its two largest c.  The
 * `selected_groups` best groups are kept (ties: lower group id), then the top_k experts inside
 * them by c (ties: lower id); idx lists them in that order.  w = s of the chosen experts,
 * divided by their sum if renormalize != 0, times `scale`, rounded to `ldt`.  The selection is
 * decided in float64.  Rows whose corrected scores hold a NaN get NaN weights and ids 0..k-1.
 * Limits (as §10 states): 1 <= E <= 1024, 1 <= groups <= 128, E % groups == 0,
 * 1 <= selected_groups <= groups, 1 <= top_k <= 64, top_k <= selected_groups * E / groups,
 * E / groups >= 2 with group_top_two (else MOE_ERR_SHAPE); scale finite and > 0 (else MOE_ERR_ARG).
 * logits [T, E] dtype ldt; idx [T, top_k] uint32; w [T, top_k] dtype ldt.
 */
int moe_route_sigmoid_grouped(const void* logits, int ldt, const float* bias, int64_t T,
                              int64_t E, int top_k, int groups, int selected_groups,
                              int group_top_two, int renormalize, float scale, uint32_t* idx,
                              void* w, moe_stream_t stream);

/*
 * moe_selected_router_weights — selected_router_weights(logits, indices, RouterWeightOptions) of
 * §12 "MoE-Training erster Ordnung": the continuous weights of a FIXED selection.
 *
 * For slot j of row t with expert i = idx[t, j]: q = p[t, i], p the softmax over all E experts
 * (scoring = MOE_SCORE_SOFTMAX, FP32) or sigmoid(logit) (MOE_SCORE_SIGMOID).
 * w[t, j] = scale * q, or scale * q / sum_j q with renormalize != 0.  Repeated indices gather the
 * same q.  A row holding an index outside [0, E) (or, with softmax, a NaN / +inf / only -inf
 * logit) is all NaN; out-of-range indices are never dereferenced and nothing is synchronised.
 * logits [T, E] dtype ldt; idx [T, top_k] of index dtype idt; w [T, top_k] FP32.
 * Limits: 1 <= top_k <= min(E, 64), E <= 1024; scale finite and > 0 (else MOE_ERR_ARG).
 */
int moe_selected_router_weights(const void* logits, int ldt, const void* idx, int idt, int64_t T,
                                int64_t E, int top_k, int scoring, int renormalize, float scale,
                                float* w, moe_stream_t stream);

/*
 * moe_selected_router_backward — selected_router_backward(logits, indices, grad_weights, options)
 * of §12: dL/dlogits [T, E] (dtype ldt) of the weights above for dL/dw = grad_w [T, top_k] (FP32).
 * Only the continuous weights are differentiated, not the top-k / group decisions or a bias.
 * Rows that are NaN in the forward are NaN here.  Per-expert sums over repeated indices are
 * accumulated in slot order (run-to-run identical).  Same limits as the forward.
 */
int moe_selected_router_backward(const void* logits, int ldt, const void* idx, int idt,
                                 const float* grad_w, int64_t T, int64_t E, int top_k, int scoring,
                                 int renormalize, float scale, void* grad_logits,
                                 moe_stream_t stream);

/*
 * moe_dispatch — RoutingPlan::dispatch(input) of §3/§5 "Expertengewichte und Verteilung".
 *
 * Capacity-free: every one of the R = T*top_k routed slots (slot s = t*top_k + j) becomes one
 * dispatched row.  Rows are grouped by expert; inside an expert they keep ascending slot order,
 * so the result does not depend on thread timing.
 *
 * x            [T, H] tokens, dtype `xdt`.
 * idx          [T, top_k] uint32 expert ids (from moe_route or the caller; ids >= E are not
 *              dispatched, their row_of_slot entry is 0xFFFFFFFF and the device status records
 *              MOE_ERR_INDEX).
 * x_d          [R, H] out, dtype `xdt`: x_d[r] = x[token_of_row[r]].
 * offsets      [E + 1] int32 out: rows of expert e are offsets[e] .. offsets[e+1]-1.
 * token_of_row [R] uint32 out: token feeding row r.
 * row_of_slot  [R] uint32 out: row holding slot s (the saved map that restores token order).
 * ws           workspace of at least moe_dispatch_workspace_bytes(T, E, top_k) bytes,
 *              16-byte aligned; contents on entry are ignored.
 * Alignment: x and x_d 16-byte aligned with H * sizeof(xdt) a multiple of 16, else MOE_ERR_ALIGN.
 */
size_t moe_dispatch_workspace_bytes(int64_t T, int64_t E, int top_k);
int moe_dispatch(const void* x, int xdt, int64_t T, int64_t H, const uint32_t* idx, int64_t E,
                 int top_k, void* x_d, int32_t* offsets, uint32_t* token_of_row,
                 uint32_t* row_of_slot, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_dispatch_static — moe_dispatch without a workspace argument.  The ruDNN pages have no
 * counterpart: this entry point exists for callers that cannot provide device scratch memory,
 * such as a plugin whose interface hands over only inputs and outputs, or a runtime whose memory
 * plan fixes every device allocation at start-up and offers none per call.
 *
 * Same arguments, results and alignment rules as moe_dispatch, minus (ws, ws_bytes).  Its scratch
 * (a status word and the per-chunk histograms) lives in a file-scope device array of
 * MOE_STATIC_DISPATCH_SCRATCH_BYTES = 256 + 1 MiB that every GPU loading the library holds until
 * the process exits; it allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 * Sizes needing more than that (moe_dispatch_workspace_bytes(T, E, top_k) > the capacity, e.g.
 * T * top_k = 131072 with E = 1024) are rejected with MOE_ERR_SHAPE before anything is enqueued.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current); make that first call before any stream capture.  The address is kept
 * per device and looked up again only when the device's context has changed (after a
 * cudaDeviceReset, for example); make the first call after such a change before any capture too.
 * All calls share the one array: calls whose work overlaps on the GPU (different streams, or
 * several host threads) race on it and must be serialised by the caller.  Ids >= E are handled
 * as in moe_dispatch (row_of_slot 0xFFFFFFFF); the device status word is not exposed.
 */
#define MOE_STATIC_DISPATCH_SCRATCH_BYTES (256u + (1u << 20))
int moe_dispatch_static(const void* x, int xdt, int64_t T, int64_t H, const uint32_t* idx,
                        int64_t E, int top_k, void* x_d, int32_t* offsets, uint32_t* token_of_row,
                        uint32_t* row_of_slot, moe_stream_t stream);

/*
 * moe_experts_forward_dispatched — SwiGluExperts::forward_dispatched of §3/§5/§6.
 *
 * For every expert e and every row r in offsets[e] .. offsets[e+1]-1:
 *   g = x_d[r] gate[e]^T,  u = x_d[r] up[e]^T          (both [I])
 *   a = silu(g) * u,       silu(z) = z / (1 + exp(-z))
 *   y[r] = a down[e]^T                                  ([H]); no bias.
 * x_d [rows, H], gate/up [E, I, H], down [E, H, I], y [rows, H]; all in dtype `wdt`.
 * offsets [E + 1] int32 on the device (non-decreasing, offsets[0] = 0, offsets[E] <= rows).
 * bf16 / f16: 5th-generation tensor cores, FP32 accumulation, `a` rounded to `wdt` between the
 *   two projections, y rounded once.  Requires H % 8 == 0, I % 8 == 0 and 16-byte aligned
 *   pointers (TMA), else MOE_ERR_ALIGN.
 * f32: FP32 CUDA-core GEMMs, `a` kept in FP32.
 * ws: at least moe_experts_workspace_bytes(rows, E, H, I, wdt) bytes, 256-byte aligned.
 */
size_t moe_experts_workspace_bytes(int64_t rows, int64_t E, int64_t H, int64_t I, int wdt);
int moe_experts_forward_dispatched(const void* x_d, const int32_t* offsets, int64_t rows,
                                   const void* gate, const void* up, const void* down, int wdt,
                                   int64_t E, int64_t H, int64_t I, void* y, void* ws,
                                   size_t ws_bytes, moe_stream_t stream);

/*
 * moe_combine — DispatchedTokens::combine(expert_output) of §3/§6.
 *
 * out[t] = sum_{j = 0..top_k-1} w[t, j] * y[row_of_slot[t*top_k + j]], accumulated in FP32 in
 * that fixed slot order (run-to-run deterministic), rounded once to `ydt`.  A slot whose
 * row_of_slot is 0xFFFFFFFF (an undispatched invalid index) makes the token's row NaN.
 * y [R, H] dtype `ydt`; w [T, top_k] dtype `wdt` (the logits dtype); out [T, H] dtype `ydt`.
 * Alignment: none required (16-byte aligned rows take a vectorised path).
 */
int moe_combine(const void* y, int ydt, const uint32_t* row_of_slot, const void* w, int wdt,
                int64_t T, int64_t H, int top_k, void* out, moe_stream_t stream);

/*
 * moe_forward — SwiGluExperts::forward(input, logits, options) of §6: route, dispatch, experts
 * and combine on one stream with no host synchronisation.
 * x [T, H] and the expert weights share dtype `wdt`; logits [T, E] have dtype `ldt`;
 * out [T, H] has dtype `wdt`.  Same alignment rules as the stages.
 * ws: at least moe_forward_workspace_bytes(T, E, H, I, top_k, ldt, wdt) bytes, 256-byte aligned.
 * Short batches (see moe_forward_fused) run as ONE cooperative launch that performs the same
 * steps between grid barriers; longer ones as the staged launches.  Both give the same routing,
 * dispatch order and combine order.  If the cooperative launch cannot have all its blocks
 * resident (another context holds SMs), the staged launches run instead.
 */
size_t moe_forward_workspace_bytes(int64_t T, int64_t E, int64_t H, int64_t I, int top_k,
                                   int ldt, int wdt);
int moe_forward(const void* x, const void* logits, int ldt, const void* gate, const void* up,
                const void* down, int wdt, int64_t T, int64_t E, int64_t H, int64_t I, int top_k,
                int renormalize, void* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_forward_fused — 1 when moe_forward runs these sizes as the single fused launch, else 0
 * (given 16-byte aligned logits, x, weights and out).  That is: bf16/f16 experts, T*top_k <= 4096
 * and fewer than 128 rows per expert on average (T*top_k < 128 E), E <= 256 with E * sizeof(ldt)
 * a multiple of 16, H and I multiples of 64, and a device with cooperative launch.  Otherwise 0.
 * The fused route reads each row of logits with one full warp; for 64 < E <= 256 and 16-bit
 * logits that is the staged route's arithmetic exactly, elsewhere the softmax denominator of a
 * non-renormalised route may be summed in another order (last-ulp differences in w).
 */
int moe_forward_fused(int64_t T, int64_t E, int64_t H, int64_t I, int top_k, int ldt, int wdt);

/*
 * moe_forward_sigmoid_grouped — SwiGluExperts::forward_sigmoid_grouped of §10: group-limited
 * sigmoid routing (as moe_route_sigmoid_grouped), then dispatch, experts and combine exactly as
 * moe_forward, including the single fused launch for the sizes moe_forward_fused reports.
 * Workspace: moe_forward_workspace_bytes(T, E, H, I, top_k, ldt, wdt).
 */
int moe_forward_sigmoid_grouped(const void* x, const void* logits, int ldt, const float* bias,
                                const void* gate, const void* up, const void* down, int wdt,
                                int64_t T, int64_t E, int64_t H, int64_t I, int top_k, int groups,
                                int selected_groups, int group_top_two, int renormalize,
                                float scale, void* out, void* ws, size_t ws_bytes,
                                moe_stream_t stream);

/*
 * Backward chain of §12 "MoE-Training erster Ordnung" (first order).  The forward saves nothing
 * beyond its inputs: the expert backward recomputes g = x_d gate^T and u = x_d up^T from x_d, so
 * the "cache" of forward_dispatched_training is (x_d, offsets) as returned by moe_dispatch.
 *
 * moe_combine_backward — DispatchedTokens::combine_backward(expert_output, grad_output):
 *   dexpert[row_of_slot[t*k+j]] = w[t, j] * dout[t]   ([T*k, H], dtype ydt; slots whose
 *                                                       row_of_slot is 0xFFFFFFFF are skipped)
 *   Every row of dexpert is written: row_of_slot as moe_dispatch returns it maps the n valid
 *   slots onto rows 0 .. n-1, and the T*k - n rows after them (present only when some expert ids
 *   were invalid) are set to zero, so dexpert needs no initialisation by the caller.
 *   dweights[t, j] = sum_h dout[t, h] * y[row_of_slot[t*k+j], h]   ([T, k] FP32, NaN for such slots)
 *   y [T*k, H] the expert output, w [T, k] the routing weights (dtype wdt), dout [T, H] dtype ydt.
 */
int moe_combine_backward(const void* y, int ydt, const uint32_t* row_of_slot, const void* w,
                         int wdt, const void* dout, int64_t T, int64_t H, int top_k,
                         void* dexpert, float* dweights, moe_stream_t stream);

/*
 * moe_experts_backward — cache.backward(dexpert): for every expert e and its rows,
 *   da = dy down_e;  s = sigmoid(g);  du = da * g s;  dg = da * u * s (1 + g (1 - s))
 *   dinput = dg gate_e + du up_e                 ([rows, H], dtype wdt)
 *   ddown[e] = dy^T (g s u); dgate[e] = dg^T x_d; dup[e] = du^T x_d   (FP32, [E,H,I], [E,I,H] x2)
 * with FP32 accumulation: on tensor cores (tcgen05) for bf16/f16 with I % 64 == 0 and 16-byte
 * aligned operands, whose GEMM operands dy, dg, du and g s u are then rounded to `wdt` as the
 * forward rounds a; on CUDA cores with FP32 operands otherwise.  Experts without rows get zero
 * gradients.  On the tensor-core path those zeros are written beside the GEMMs on a second stream
 * that the library keeps per device and context (created on the first call), forked from
 * `stream` and joined back into it with two events created and released within the call, so
 * every write is ordered before work enqueued on `stream` after the call.  While `stream` is
 * being captured into a CUDA graph they are written on `stream` itself.
 * dy [rows, H] dtype wdt.  ws: moe_experts_backward_workspace_bytes(rows, I), 256-byte aligned.
 */
size_t moe_experts_backward_workspace_bytes(int64_t rows, int64_t I);
int moe_experts_backward(const void* x_d, const int32_t* offsets, int64_t rows, const void* gate,
                         const void* up, const void* down, int wdt, int64_t E, int64_t H,
                         int64_t I, const void* dy, void* dinput, float* dgate, float* dup,
                         float* ddown, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_dispatch_backward — DispatchedTokens::dispatch_backward(dinput): dx[t] = sum over the slots
 * j of token t of dinput[row_of_slot[t*k+j]], FP32 in slot order, rounded to `dt`; the routing
 * weights are not applied again.  dinput [T*k, H], dx [T, H], both dtype dt.
 */
int moe_dispatch_backward(const void* dinput, int dt, const uint32_t* row_of_slot, int64_t T,
                          int64_t H, int top_k, void* dx, moe_stream_t stream);

/*
 * moe_forward_with_events — the staged path of moe_forward (route, dispatch, gate/up GEMM, down
 * GEMM and combine as separate launches, whatever the sizes) that also records caller-created
 * CUDA events (cudaEvent_t, passed as void*) on `stream` at the stage boundaries, for timing:
 *   events[0] before the route      events[1] after the route     events[2] after dispatch
 *   events[3] after the gate/up GEMM events[4] after the down GEMM events[5] after the combine
 * `events` may be NULL (then this runs the staged path untimed).
 */
int moe_forward_with_events(const void* x, const void* logits, int ldt, const void* gate,
                            const void* up, const void* down, int wdt, int64_t T, int64_t E,
                            int64_t H, int64_t I, int top_k, int renormalize, void* out, void* ws,
                            size_t ws_bytes, moe_stream_t stream, void* const* events);

/*
 * moe_wait_selftest — exercises the failure path of the tensor-core kernels without a fault: one
 * bounded mbarrier wait (the same routine those kernels use) on a barrier that nothing completes.
 * It gives up after about a second, sets the timeout bit in the status word at the start of `ws`
 * (>= 256 bytes, 256-byte aligned) and returns; moe_device_status then reports MOE_ERR_TIMEOUT and
 * the context stays usable.  For tests and diagnostics; it touches nothing else.
 */
int moe_wait_selftest(void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_device_status — synchronises `stream`, then reads and clears the status word at the start
 * of a workspace used by moe_dispatch, moe_experts_forward_dispatched or moe_forward.
 * Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_INDEX, or MOE_ERR_CUDA if the read itself failed.
 */
int moe_device_status(void* ws, size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
