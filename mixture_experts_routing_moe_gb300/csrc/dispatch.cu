// Dispatch: RoutingPlan::dispatch of the ruDNN user guide, §5 "Expertengewichte und Verteilung".
//
// Capacity-free and deterministic.  The page leaves the order inside an expert open (it comes
// from atomics there); here rows keep ascending slot order s = t*k + j, built as a stable
// counting sort without atomics on global memory:
//   1. count   — warp w owns slots [w*CH, w*CH + CH); it histograms its chunk in a warp-private
//                shared-memory array (lanes with the same expert are merged with match.any) and
//                writes hist[w][e].
//   2. scan    — one block per expert: hist[w][e] becomes the exclusive prefix over w, and
//                totals[e] the expert's row count.
//   3. scatter — every warp derives offsets = exclusive prefix over e of totals (warp 0 also
//                writes them out), then walks its chunk again in slot order; a slot's row is
//                offsets[e] + hist[w][e] + (earlier slots of the chunk with the same expert), the
//                last term from match.any ranks.  Writes row_of_slot and token_of_row.
//   4. rows    — one block per token reads x[t] once (16-byte loads) and writes it to the k rows
//                row_of_slot[t*k + 0..k-1] of x_d.
// Batches of at most 4096 slots run steps 1-3 in one block with the histograms in shared memory.
// Expert ids >= E are not dispatched: their row_of_slot is 0xFFFFFFFF and the status word gets
// the index bit.  No access goes out of bounds for any id value.
#include <cuda.h>

#include <mutex>
#include <utility>

#include "common.cuh"
#include "dispatch_core.cuh"
#include "launch.h"

// Scratch of moe_dispatch_static(): a status word (in the first 256 bytes) followed by the
// per-chunk histograms, in a file-scope device array instead of caller-provided memory.  Every
// GPU that loads this library holds it until the process exits.
static __device__ __align__(256) unsigned char g_static_dispatch_scratch[kStaticDispatchScratchBytes];

namespace moe {
namespace {

constexpr int kDispWarps = 4;  // warps per block in count / scatter
constexpr int kMaxE = 1024;

__global__ void __launch_bounds__(kDispWarps * 32)
    moe_dispatch_count(const uint32_t* __restrict__ idx, int64_t R, int E, int W, int CH,
                       int32_t* __restrict__ hist, unsigned* status) {
  extern __shared__ int32_t disp_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wg = blockIdx.x * kDispWarps + warp;
  if (wg >= W) return;
  int32_t* h = disp_smem + warp * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  const int64_t s0 = (int64_t)wg * CH, s1 = (R < s0 + CH) ? R : s0 + CH;
  bool bad = false;
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t s = base + lane;
    const bool act = s < s1;
    const uint32_t e = act ? idx[s] : 0xFFFFFFFFu;
    const bool valid = act && e < (uint32_t)E;
    bad |= act && !valid;
    const uint32_t key = valid ? e : 0xFFFFFFFFu;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, key);
    if (valid && lane == __ffs(peers) - 1) h[e] += __popc(peers);
    __syncwarp();
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(status, kStatusIndex);
  for (int e = lane; e < E; e += 32) hist[(int64_t)wg * E + e] = h[e];
}

// One block per expert e: the column hist[0..W-1][e] becomes its exclusive prefix over the
// chunks (a block-wide scan), and totals[e] receives the column sum.
constexpr int kScanThreads = 256;
__global__ void __launch_bounds__(kScanThreads)
    moe_dispatch_scan(int32_t* __restrict__ hist, int W, int E, int32_t* __restrict__ totals) {
  __shared__ int32_t warp_tot[kScanThreads / 32];
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int PER = kMaxE / kScanThreads;  // W <= 1024 chunks: up to 4 per thread
  int32_t v[PER];
  int32_t local = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int w = tid * PER + i;
    v[i] = w < W ? hist[(int64_t)w * E + e] : 0;
    local += v[i];
  }
  int32_t x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t t = lane < kScanThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kScanThreads / 32) warp_tot[lane] = t;
  }
  __syncthreads();
  int32_t run = (warp > 0 ? warp_tot[warp - 1] : 0) + x - local;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int w = tid * PER + i;
    if (w < W) hist[(int64_t)w * E + e] = run;
    run += v[i];
  }
  if (tid == kScanThreads - 1) totals[e] = run;
}

__global__ void __launch_bounds__(kDispWarps * 32)
    moe_dispatch_scatter(const uint32_t* __restrict__ idx, int64_t R, int E, int k, int W, int CH,
                         const int32_t* __restrict__ hist, const int32_t* __restrict__ totals,
                         int32_t* __restrict__ offsets, uint32_t* __restrict__ token_of_row,
                         uint32_t* __restrict__ row_of_slot) {
  extern __shared__ int32_t disp_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wg = blockIdx.x * kDispWarps + warp;
  if (wg >= W) return;
  int32_t* run = disp_smem + warp * E;
  // offsets = exclusive prefix of the per-expert totals, recomputed by every warp (E <= 1024)
  int32_t carry = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    const int32_t c = e < E ? totals[e] : 0;
    int32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (e < E) {
      const int32_t off = carry + x - c;
      run[e] = off + hist[(int64_t)wg * E + e];
      if (wg == 0) offsets[e] = off;
    }
    carry += __shfl_sync(0xFFFFFFFFu, x, 31);
  }
  if (wg == 0 && lane == 0) offsets[E] = carry;
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  const int64_t s0 = (int64_t)wg * CH, s1 = (R < s0 + CH) ? R : s0 + CH;
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t s = base + lane;
    const bool act = s < s1;
    const uint32_t e = act ? idx[s] : 0xFFFFFFFFu;
    const bool valid = act && e < (uint32_t)E;
    const uint32_t key = valid ? e : 0xFFFFFFFFu;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, key);
    if (valid) {
      const uint32_t row = (uint32_t)(run[e] + __popc(peers & lt));
      row_of_slot[s] = row;
      token_of_row[row] = (uint32_t)(s / k);
    } else if (act) {
      row_of_slot[s] = kInvalidRow;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) run[e] += __popc(peers);
    __syncwarp();
  }
}

// Short batches (R <= kSmallR slots): count, scan and scatter in one block of kSmallWarps warps,
// histograms in shared memory; the same stable order as the three-kernel path (warp w owns the
// contiguous chunk [w*CH, w*CH + CH) and ranks inside a chunk come from match.any).
constexpr int kSmallWarps = 8;
constexpr int64_t kSmallR = 4096;
__global__ void __launch_bounds__(kSmallWarps * 32)
    moe_dispatch_small(const uint32_t* __restrict__ idx, int64_t R, int E, int k, int CH,
                       int32_t* __restrict__ offsets, uint32_t* __restrict__ token_of_row,
                       uint32_t* __restrict__ row_of_slot, unsigned* status) {
  extern __shared__ int32_t small_smem[];
  dispatch_block<false>(idx, R, E, k, kSmallWarps, CH, small_smem, small_smem + kSmallWarps * E,
                        offsets, token_of_row, row_of_slot, status);
}

// One block per token (grid-stride): x[t] is read once and written to its k dispatched rows.
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
    moe_dispatch_rows(const uint4* __restrict__ x, int64_t T, int64_t vecs_per_row, int k,
                      const uint32_t* __restrict__ row_of_slot, uint4* __restrict__ x_d) {
  extern __shared__ uint32_t rows_smem[];
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    for (int j = threadIdx.x; j < k; j += THREADS) rows_smem[j] = row_of_slot[t * k + j];
    __syncthreads();
    const uint4* src = x + t * vecs_per_row;
    for (int64_t c = threadIdx.x; c < vecs_per_row; c += THREADS) {
      const uint4 v = ld_nc_v4(src + c);
      for (int j = 0; j < k; ++j) {
        const uint32_t r = rows_smem[j];
        if (r != kInvalidRow) st_v4(x_d + (int64_t)r * vecs_per_row + c, v);
      }
    }
    __syncthreads();
  }
}

}  // namespace

DispatchPlan dispatch_plan(int64_t R) {
  DispatchPlan p;
  int64_t W = (R + 255) / 256;
  if (W > 1024) W = 1024;
  if (W < 1) W = 1;
  int64_t CH = (R + W - 1) / W;
  CH = (CH + 31) / 32 * 32;
  if (CH < 32) CH = 32;
  p.CH = (int)CH;
  p.W = (int)((R + CH - 1) / CH);
  if (p.W < 1) p.W = 1;
  return p;
}

// The id of the calling thread's current CUDA context (0 when none is current or the driver
// entry points are unavailable).  Context ids are unique for the life of the process, so a
// context that replaces a destroyed one (after cudaDeviceReset) never matches a cached id.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static const std::pair<GetCurrentFn, GetIdFn> fns = []() {
    void* cur = nullptr;
    void* id = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &cur, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess || q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &id, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess || q2 != cudaDriverEntryPointSuccess)
      return std::pair<GetCurrentFn, GetIdFn>(nullptr, nullptr);
    return std::pair<GetCurrentFn, GetIdFn>(reinterpret_cast<GetCurrentFn>(cur),
                                            reinterpret_cast<GetIdFn>(id));
  }();
  if (!fns.first || !fns.second) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (fns.first(&ctx) != CUDA_SUCCESS || !ctx || fns.second(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

cudaError_t static_dispatch_scratch(void** ptr) {
  // Host code must not use g_static_dispatch_scratch as an address: that name is a host-side
  // stand-in.  The device address is looked up with the device current, on the first call on
  // that device, and again whenever the device's context has changed since (a cudaDeviceReset
  // destroys the context, and the array gets a new address in the next one).
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_static_dispatch_scratch);  // binds the context if needed
    if (err != cudaSuccess) return err;
    addr[dev] = p;
    ctx_of[dev] = current_context_id();
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

size_t dispatch_scratch_bytes(int64_t R, int E) {  // per-chunk histograms + per-expert totals
  return ((size_t)dispatch_plan(R).W + 1) * (size_t)E * sizeof(int32_t);
}

cudaError_t launch_dispatch(const void* x, int xdt, int64_t T, int64_t H, const uint32_t* idx,
                            int E, int k, void* x_d, int32_t* offsets, uint32_t* token_of_row,
                            uint32_t* row_of_slot, int32_t* hist, unsigned* status,
                            cudaStream_t s) {
  const int64_t R = T * k;
  if (R <= kSmallR) {
    const int CH = (int)(((R + kSmallWarps - 1) / kSmallWarps + 31) / 32 * 32);
    const size_t smem = ((size_t)kSmallWarps * E + E + 1) * sizeof(int32_t);
    moe_dispatch_small<<<1, kSmallWarps * 32, smem, s>>>(idx, R, E, k, CH, offsets, token_of_row,
                                                         row_of_slot, status);
  } else {
    const DispatchPlan p = dispatch_plan(R);
    const size_t smem = (size_t)kDispWarps * E * sizeof(int32_t);
    const unsigned blocks = (unsigned)((p.W + kDispWarps - 1) / kDispWarps);
    moe_dispatch_count<<<blocks, kDispWarps * 32, smem, s>>>(idx, R, E, p.W, p.CH, hist, status);
    int32_t* totals = hist + (size_t)p.W * E;
    moe_dispatch_scan<<<E, kScanThreads, 0, s>>>(hist, p.W, E, totals);
    moe_dispatch_scatter<<<blocks, kDispWarps * 32, smem, s>>>(
        idx, R, E, k, p.W, p.CH, hist, totals, offsets, token_of_row, row_of_slot);
  }
  const size_t esz = xdt == MOE_F32 ? 4 : 2;
  const int64_t vecs = H * (int64_t)esz / 16;
  int64_t grid = T < 65536 ? T : 65536;
  moe_dispatch_rows<128><<<(unsigned)grid, 128, (size_t)k * 4, s>>>(
      (const uint4*)x, T, vecs, k, row_of_slot, (uint4*)x_d);
  return cudaGetLastError();
}

}  // namespace moe
