// Fused forward for short batches (decode): route -> dispatch -> gate/up -> down -> combine of the
// ruDNN user guide (§3 "MoE-Workflow", §4 "Routing-Vertrag", §5 "Expertengewichte und
// Verteilung", §6 "MoE aufrufen") in ONE persistent launch, instead of the six launches of the
// staged path.  With T * top_k <= 4096 rows the staged path spends about as long on launch gaps,
// the route and the dispatch as on streaming the expert weights; here those steps take a few
// microseconds between grid barriers.
//
// One CTA per SM (cooperative launch, so all CTAs are resident and may wait on each other), the
// warp roles of the single-CTA expert GEMM (gemm_cta.cuh), phases separated by grid barriers:
//   1. route     token rows strided over all warps of the grid; one warp per row, the same
//                arithmetic as the route kernel (route_core.cuh) -> idx, w in the workspace.
//   2. dispatch  every CTA sorts all T * k slots in shared memory (dispatch_core.cuh; the same
//                stable order as the dispatch kernels); CTA 0 publishes offsets and row_of_slot;
//                each CTA gathers its contiguous share of the rows of x_d.
//   3. gate/up   the single-CTA tcgen05 GEMM over the tile list of the offsets -> a.
//   4. down      the same GEMM on a -> y (y reuses the x_d buffer).
//   5. combine   (token, 256-column chunk) items strided over all warps (combine_core.cuh).
// Data written in one phase and read in a later one goes through L2 only: generic loads use
// ld.global.cg, and x_d / a, which the next phase reads with TMA, are ordered for the async proxy
// by fence.proxy.async on both sides of the barrier.  Every wait (mbarriers and the grid barrier)
// is bounded; on expiry the status word gets the timeout bit, later phases are skipped and the
// kernel still releases TMEM and exits.
#include <cuda.h>

#include <type_traits>

#include "combine_core.cuh"
#include "common.cuh"
#include "dispatch_core.cuh"
#include "gemm_cta.cuh"
#include "launch.h"
#include "route_core.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {
using namespace tc;
using namespace cta_gemm;

constexpr int kWarps = kThreads / 32;
constexpr int kOffInts = kFusedDecodeMaxExperts + 8;  // persistent copy of the offsets
constexpr size_t kFusedSmemBytes = kSmemBytes + kOffInts * sizeof(int);

struct DecodeParams {
  const void* logits;
  const void* x;
  int T, E, H, I, k, renorm;
  uint32_t* idx;          // [T k]
  void* w;                // [T k] in the logits dtype
  uint32_t* row_of_slot;  // [T k]
  int32_t* offsets;       // [E + 1]
  void* x_d;              // [T k, H]; y afterwards
  void* a;                // [T k, I]
  void* out;              // [T, H]
  unsigned* status;
  unsigned* grid_count;   // zero at launch
  TcParams gu, dn;        // offsets filled in by the kernel (shared memory)
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Generic-proxy writes of this thread (global and shared) before later async-proxy accesses.
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

// Grid barrier number `n` (1, 2, ...): every CTA arrives once; returns when all gridDim.x have.
// Bounded: after kWaitLimit cycles the status word gets the timeout bit and the abort flag is set.
__device__ __forceinline__ void grid_barrier(unsigned* count, unsigned n, volatile int* abort_f,
                                             unsigned* status) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(count, 1u);
    const unsigned target = n * gridDim.x;
    const long long t0 = clock64();
    while (ld_acquire_gpu(count) < target) {
      if (clock64() - t0 > kWaitLimit) {
        *abort_f = 1;
        atomicOr(status, kStatusTimeout);
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
  }
  __syncthreads();
}

template <typename TL, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    moe_decode_fused(const __grid_constant__ CUtensorMap map_xd,
                     const __grid_constant__ CUtensorMap map_gate,
                     const __grid_constant__ CUtensorMap map_up,
                     const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_down, const DecodeParams p) {
  using TX = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t fd_smem_raw[];
  uint32_t* tmem_slot;
  int* pref;
  Ring ring = carve_ring(fd_smem_raw, &tmem_slot, &pref);
  int32_t* offs = reinterpret_cast<int32_t*>(pref + kMaxExperts + 4);
  // the stage ring doubles as scratch for the phases that run before and after the GEMMs
  uint8_t* scratch = fd_smem_raw + (ring.base - smem_u32(fd_smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t R = (int64_t)p.T * p.k;

  if (threadIdx.x == 0) init_ring(ring);
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (warp == 0 && lane == 0) {
    tma_prefetch(&map_xd);
    tma_prefetch(&map_gate);
    tma_prefetch(&map_up);
    tma_prefetch(&map_a);
    tma_prefetch(&map_down);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  ring.tmem_base = *tmem_slot;
  ProducerState pst;
  MmaState mst;
  EpilogueState est;

  // ---------------------------------------------------------------- 1. route
  {
    uint32_t* s_id = reinterpret_cast<uint32_t*>(scratch) + warp * p.k;
    float* s_e = reinterpret_cast<float*>(scratch + (size_t)kWarps * p.k * 4) + warp * p.k;
    for (int64_t row = (int64_t)blockIdx.x * kWarps + warp; row < p.T;
         row += (int64_t)gridDim.x * kWarps) {
      route_row<TL, 32, 8, true>(reinterpret_cast<const TL*>(p.logits), row, true, p.E, p.k,
                                 p.renorm, lane, s_id, s_e, p.idx, reinterpret_cast<TL*>(p.w));
      __syncwarp();
    }
  }
  grid_barrier(p.grid_count, 1, ring.abort_f, p.status);

  // ---------------------------------------------------------------- 2. dispatch + gather
  if (!*ring.abort_f) {
    int32_t* hist = reinterpret_cast<int32_t*>(scratch);  // [kWarps][E]
    int32_t* off_s = hist + kWarps * p.E;                  // [E + 1]
    uint32_t* tor = reinterpret_cast<uint32_t*>(off_s + p.E + 8);
    const int CH = (int)(((R + kWarps - 1) / kWarps + 31) / 32 * 32);
    const bool lead = blockIdx.x == 0;
    dispatch_block<true>(p.idx, R, p.E, p.k, kWarps, CH, hist, off_s, lead ? p.offsets : nullptr,
                         tor, lead ? p.row_of_slot : nullptr, lead ? p.status : nullptr);
    __syncthreads();
    for (int e = threadIdx.x; e <= p.E; e += blockDim.x) offs[e] = off_s[e];
    // rows [r0, r1) of x_d: x_d[r] = x[token_of_row[r]], 16-byte vectors
    const int64_t per = (R + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = min(R, (int64_t)blockIdx.x * per), r1 = min(R, r0 + per);
    const int64_t vec_per_row = (int64_t)p.H * 2 / 16;
    const uint4* xs = reinterpret_cast<const uint4*>(p.x);
    uint4* xd = reinterpret_cast<uint4*>(p.x_d);
    for (int64_t i = threadIdx.x; i < (r1 - r0) * vec_per_row; i += blockDim.x) {
      const int64_t r = r0 + i / vec_per_row, c = i % vec_per_row;
      st_v4(xd + r * vec_per_row + c, ld_nc_v4(xs + (int64_t)tor[r] * vec_per_row + c));
    }
    // x_d is read by TMA after the barrier, and TMA refills this scratch shared memory
    fence_proxy_async_all();
    __syncthreads();
    if (warp == 2) build_mtile_prefix(offs, p.E, BM, pref, lane);
  }
  grid_barrier(p.grid_count, 2, ring.abort_f, p.status);

  // ---------------------------------------------------------------- 3. gate/up, 4. down
  TcParams gu = p.gu, dn = p.dn;
  gu.offsets = offs;
  dn.offsets = offs;
  for (int g = 0; g < 2 && !*ring.abort_f; ++g) {
    const TcParams& tp = g == 0 ? gu : dn;
    if (warp == 0) {
      if (lane == 0) {
        fence_proxy_async_global();
        if (g == 0)
          producer<true, true>(&map_xd, &map_gate, &map_up, tp, pref, ring, pst);
        else
          producer<false, true>(&map_a, &map_down, &map_down, tp, pref, ring, pst);
      }
    } else if (warp == 1) {
      if (lane == 0) mma<BF16>(tp, pref, ring, mst);
    } else {
      if (g == 0)
        epilogue<true, BF16, true>(tp, pref, ring, est, warp, lane);
      else
        epilogue<false, BF16, true>(tp, pref, ring, est, warp, lane);
      fence_proxy_async_global();  // a is read by TMA after the barrier
    }
    grid_barrier(p.grid_count, 3 + g, ring.abort_f, p.status);
  }

  // ---------------------------------------------------------------- 5. combine
  if (!*ring.abort_f) {
    const int64_t chunks = (int64_t)p.H * 2 / 16;
    const int64_t wpt = (chunks + 31) / 32;
    for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < (int64_t)p.T * wpt;
         it += (int64_t)gridDim.x * kWarps) {
      const int64_t t = it / wpt;
      combine_warp<TX, TL, true, true>(reinterpret_cast<const TX*>(p.x_d), p.row_of_slot,
                                       reinterpret_cast<const TL*>(p.w), t, p.H, p.k,
                                       it - t * wpt, reinterpret_cast<TX*>(p.out), lane);
    }
  }

  // ---------------------------------------------------------------- teardown
  if (warp == 0 && lane == 0 && *ring.abort_f) producer_drain(ring, pst);
  if (warp == 1 && lane == 0) mma_drain(ring);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(ring.tmem_base, kTmemCols);
  }
}

template <typename TL, bool BF16>
cudaError_t launch_t(const FusedDecodeArgs& f, cudaStream_t s) {
  auto kern = moe_decode_fused<TL, BF16>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kFusedSmemBytes);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0, per_sm = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads,
                                                           kFusedSmemBytes)) != cudaSuccess)
    return err;
  if (per_sm < 1) return cudaErrorLaunchOutOfResources;
  const int grid = sms;  // one CTA per SM, all resident (cooperative launch)

  const int64_t R = (int64_t)f.T * f.k;
  CUtensorMap m_xd, m_gate, m_up, m_a, m_down;
  if (!make_map_2d(&m_xd, f.x_d, BF16, f.H, R, BK, BM) ||
      !make_map_2d(&m_gate, f.gate, BF16, f.H, (int64_t)f.E * f.I, BK, BN / 2) ||
      !make_map_2d(&m_up, f.up, BF16, f.H, (int64_t)f.E * f.I, BK, BN / 2) ||
      !make_map_2d(&m_a, f.a, BF16, f.I, R, BK, BM) ||
      !make_map_2d(&m_down, f.down, BF16, f.I, (int64_t)f.E * f.H, BK, BN))
    return cudaErrorInvalidValue;

  DecodeParams p{};
  p.logits = f.logits;
  p.x = f.x;
  p.T = (int)f.T;
  p.E = f.E;
  p.H = f.H;
  p.I = f.I;
  p.k = f.k;
  p.renorm = f.renorm;
  p.idx = f.idx;
  p.w = f.w;
  p.row_of_slot = f.row_of_slot;
  p.offsets = f.offsets;
  p.x_d = f.x_d;
  p.a = f.a;
  p.out = f.out;
  p.status = f.status;
  p.grid_count = f.grid_count;
  p.gu.out = (uint8_t*)f.a;
  p.gu.status = f.status;
  p.gu.E = f.E;
  p.gu.N = f.I;
  p.gu.KB = (f.H + BK - 1) / BK;
  p.gu.NT = (f.I + BN / 2 - 1) / (BN / 2);
  p.gu.b_rows = f.I;
  p.dn.out = (uint8_t*)f.x_d;
  p.dn.status = f.status;
  p.dn.E = f.E;
  p.dn.N = f.H;
  p.dn.KB = (f.I + BK - 1) / BK;
  p.dn.NT = (f.H + BN - 1) / BN;
  p.dn.b_rows = f.H;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kFusedSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, m_xd, m_gate, m_up, m_a, m_down, p);
}

}  // namespace

bool fused_decode_supported(int64_t T, int E, int64_t H, int64_t I, int k, int ldt, int wdt) {
  if (wdt != MOE_BF16 && wdt != MOE_F16) return false;
  const int64_t R = T * k;
  if (R < 1 || R > kFusedDecodeMaxRows) return false;
  if (E < 1 || E > kFusedDecodeMaxExperts || k < 1 || k > E) return false;
  const int lsize = ldt == MOE_F32 ? 4 : 2;
  if ((E * lsize) % 16 != 0) return false;     // 16-byte route loads
  if (H % 64 != 0 || I % 64 != 0) return false;  // whole 16-byte vectors and TMA boxes
  if (R >= (int64_t)128 * E) return false;     // experts average < 128 rows: the CTA GEMM's regime
  return true;
}

cudaError_t launch_decode_fused(const FusedDecodeArgs& f, int ldt, int wdt, cudaStream_t s) {
  const bool bf = wdt == MOE_BF16;
  switch (ldt) {
    case MOE_F32: return bf ? launch_t<float, true>(f, s) : launch_t<float, false>(f, s);
    case MOE_F16: return bf ? launch_t<__half, true>(f, s) : launch_t<__half, false>(f, s);
    case MOE_BF16:
      return bf ? launch_t<__nv_bfloat16, true>(f, s) : launch_t<__nv_bfloat16, false>(f, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
