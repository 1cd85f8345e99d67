// Fused forward for short batches (decode): route -> dispatch -> gate/up -> down -> combine of the
// ruDNN user guide (§3 "MoE-Workflow", §4 "Routing-Vertrag", §5 "Expertengewichte und
// Verteilung", §6 "MoE aufrufen") in ONE persistent launch, instead of the six launches of the
// staged path.  With T * top_k <= 4096 rows the staged path spends about as long on launch gaps,
// the route and the dispatch as on streaming the expert weights; here those steps take a few
// microseconds between grid barriers.
//
// One CTA per SM (cooperative launch, so all CTAs are resident and may wait on each other), the
// warp roles of the single-CTA expert GEMM (gemm_cta.cuh); one grid barrier, after the route,
// and counters in global memory for every later hand-over between CTAs:
//   1. route     token rows strided over all warps of the grid; one warp per row, the same
//                arithmetic as the route kernel (route_core.cuh) -> idx, w in the workspace.
//   2. dispatch  every CTA counts all T * k slots in shared memory (dispatch_core.cuh: the
//                offsets and, per warp chunk, each expert's first row; CTA 0 publishes the
//                offsets); each CTA takes a contiguous share of the rows of x_d, finds each row's
//                slot in the stable order (ascending slot order inside an expert, as in the
//                dispatch kernels), writes its row_of_slot entry, gathers the row, and adds the
//                rows it copied to a per-m-tile count and to a row_of_slot count the combine
//                waits for.
//   3. gate/up   the single-CTA tcgen05 GEMM over the tile list of the offsets -> a; a tile's
//                producer loads B at once and A once the m-tile's gathered count equals its
//                rows.  Every CTA finishes its gather before its first tile, so every wait ends.
//   4. down      the same GEMM on a -> y (y reuses the x_d buffer).  No barrier before it: a
//                per-m-tile count of stored gate/up warps gates the A loads of each down tile,
//                so the down GEMM starts while the last gate/up tiles are still running.
//   5. combine   (token, 256-column chunk) items strided over all warps (combine_core.cuh), each
//                waiting only for the down tiles it reads (no grid barrier before it).
// Data written in one phase and read in a later one goes through L2 only: generic loads use
// ld.global.cg, and x_d / a, which the next phase reads with TMA, are ordered for the async proxy
// by fence.proxy.async on both sides of the count that hands them over.  Every wait (mbarriers,
// the grid barrier and the counts) is bounded; on expiry the status word gets the timeout bit,
// later phases are skipped and the kernel still releases TMEM and exits.
#include <cuda.h>

#include <type_traits>

#include "combine_core.cuh"
#include "common.cuh"
#include "dispatch_core.cuh"
#include "gemm_cta.cuh"
#include "launch.h"
#include "route_core.cuh"
#include "route_sigmoid_core.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {
using namespace tc;
using namespace cta_gemm;

constexpr int kWarps = kThreads / 32;
constexpr int kOffInts = kFusedDecodeMaxExperts + 8;  // persistent copy of the offsets
// Tile ring of the dynamic scheduler: ids of the next tiles, claimed by the producer from a
// global counter and read in order by the MMA thread and the four epilogue warps.
constexpr int kTileSlots = 4;
constexpr int kSchedBytes = 2 * kTileSlots * 8 + kTileSlots * 4 + 16;
constexpr size_t kFusedSmemBytes = kSmemBytes + kOffInts * sizeof(int) + kSchedBytes;

struct TileRing {
  uint32_t bar0;      // full[0..3] then empty[0..3]
  volatile int* ids;  // [kTileSlots]; -1 = no more tiles
  __device__ uint32_t full(int q) const { return bar0 + 8u * q; }
  __device__ uint32_t empty(int q) const { return bar0 + 8u * (kTileSlots + q); }
};

struct DecodeParams {
  const void* logits;
  const void* x;
  const void* gate;       // [E, I, H]
  const void* up;         // [E, I, H]
  int T, E, H, I, k, renorm;
  // group-limited sigmoid routing (template SIG): bias may be null
  const float* bias;
  int G, SG, top_two;
  float scale;
  uint32_t* idx;          // [T k]
  void* w;                // [T k] in the logits dtype
  uint32_t* row_of_slot;  // [T k]
  int32_t* offsets;       // [E + 1]
  void* x_d;              // [T k, H]; y afterwards
  void* a;                // [T k, I]
  void* out;              // [T, H]
  unsigned* status;
  unsigned* grid_count;   // zero at launch
  unsigned* tile_count;   // zeroed in phase 1: GEMM tiles claimed after the static first ones
  unsigned* mtile_ready;  // [n_ready], zeroed in phase 1: stored gate/up warps per m-tile
                          // [n_mtiles], stored down warps per (m-tile, n-tile), gathered x_d
                          // rows per m-tile [n_mtiles], then the row_of_slot flag
  int n_ready, n_mtiles;
  TcParams gu, dn;        // offsets filled in by the kernel (shared memory)
};

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
    while (ld_acquire_gpu_u32(count) < target) {
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

template <typename TL, bool BF16, bool SIG>
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
  TileRing tr;
  int* first_tile;  // the first GEMM tile this CTA claimed (-1: none)
  {
    uint64_t* b = reinterpret_cast<uint64_t*>(offs + kOffInts);  // 8-byte aligned: kOffInts even
    tr.bar0 = smem_u32(b);
    tr.ids = reinterpret_cast<volatile int*>(b + 2 * kTileSlots);
    first_tile = const_cast<int*>(tr.ids + kTileSlots);
  }
  // the stage ring doubles as scratch for the phases that run before and after the GEMMs
  uint8_t* scratch = fd_smem_raw + (ring.base - smem_u32(fd_smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t R = (int64_t)p.T * p.k;
  // x_d rows gathered per m-tile, then the row_of_slot entries written (after the per-(m-tile,
  // n-tile) y counts of the down epilogue)
  unsigned* gathered = p.mtile_ready + (size_t)p.n_mtiles * (1 + p.dn.NT);
  unsigned* ros_count = gathered + p.n_mtiles;

  if (threadIdx.x == 0) {
    for (int q = 0; q < kTileSlots; ++q) {
      mbar_init(tr.full(q), 1);
      mbar_init(tr.empty(q), 1 + 4);  // the MMA thread and the four epilogue warps
    }
    init_ring(ring);  // also fences the barrier initialisation
  }
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
  if (blockIdx.x == 0) {  // counters first used after the grid barrier: zeroed here, not by the host
    if (threadIdx.x == 0) *p.tile_count = 0u;
    for (int i = threadIdx.x; i < p.n_ready; i += blockDim.x) p.mtile_ready[i] = 0u;
  }
  if constexpr (SIG) {
    double* cs = reinterpret_cast<double*>(scratch) + (size_t)warp * (p.E + 128 + 64 + 32);
    for (int64_t row = (int64_t)blockIdx.x * kWarps + warp; row < p.T;
         row += (int64_t)gridDim.x * kWarps) {
      sigmoid_route_row<TL, 8>(reinterpret_cast<const TL*>(p.logits) + row * (int64_t)p.E, p.bias,
                               row, p.E, p.k, p.G, p.SG, p.top_two, p.renorm, p.scale, cs, lane,
                               p.idx, reinterpret_cast<TL*>(p.w));
      __syncwarp();
    }
  } else {
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
    uint32_t* tor = reinterpret_cast<uint32_t*>(off_s + p.E + 8);  // [R]
    uint32_t* idx_s = reinterpret_cast<uint32_t*>(                  // [R], 16-byte aligned
        (reinterpret_cast<uintptr_t>(tor + R) + 15) & ~static_cast<uintptr_t>(15));
    // all ids into shared memory first: one round trip to L2 instead of one per 32 slots
    for (int64_t i = threadIdx.x; i < (R + 3) / 4; i += blockDim.x) {
      if (4 * i + 3 < R) {
        *reinterpret_cast<uint4*>(idx_s + 4 * i) = ld_cg_v4(p.idx + 4 * i);
      } else {
        for (int64_t j = 4 * i; j < R; ++j) idx_s[j] = ld_cg_u32(p.idx + j);
      }
    }
    __syncthreads();
    const int CH = (int)(((R + kWarps - 1) / kWarps + 31) / 32 * 32);
    const bool lead = blockIdx.x == 0;  // publishes the offsets
    dispatch_count<true>(idx_s, R, p.E, kWarps, CH, hist, off_s, lead ? p.offsets : nullptr,
                         lead ? p.status : nullptr);
    for (int e = threadIdx.x; e <= p.E; e += blockDim.x) offs[e] = off_s[e];
    __syncthreads();
    if (warp == 2) build_mtile_prefix(offs, p.E, BM, pref, lane);
    __syncthreads();
    if (threadIdx.x == 0) {
      // The tile list is known now.  This CTA's first GEMM tile is tile blockIdx.x (static, so
      // no contention on the claim counter); half of its gate and up rows (contiguous in memory)
      // go to L2 while the slots are scattered and the rows of x_d gathered.  Over the grid
      // that is at most 152 x 2 x 64 rows x H x 2 bytes: 78 MB at H = 2048, within L2.
      const int n_gu = pref[p.E] * p.gu.NT;
      const int n_dn = pref[p.E] * p.dn.NT;
      int t = (int)blockIdx.x;
      if (t >= n_gu + n_dn) t = -1;
      *first_tile = t;
      if (t >= 0 && t < n_gu) {
        int e, m, n;
        decode_tile(t, pref, p.E, p.gu.NT, p.gu.KB * BK, e, m, n);
        const int rows = min(64, p.I - n * (BN / 2));
        const size_t row0 = (size_t)e * p.I + n * (BN / 2);
        const uint32_t bytes = (uint32_t)rows * p.H * 2;
        bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(p.gate) + row0 * p.H * 2, bytes);
        bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(p.up) + row0 * p.H * 2, bytes);
      }
    }
    // Rows [r0, r1) of x_d are this CTA's.  Their slots come straight from the sorted order
    // instead of a full scatter: after dispatch_count, hist[c * E + e] is the first row of
    // expert e among the slots of chunk c, so row r of expert e is the (r - hist[c * E + e])-th
    // slot holding e in the last chunk c whose first row is <= r.  Every row is gathered by
    // exactly one CTA, which also writes its slot's row_of_slot entry.
    // 32-bit index arithmetic: R <= 4096 rows of H / 8 <= 2^16 vectors (64-bit division is slow)
    const uint32_t per = (uint32_t)((R + gridDim.x - 1) / gridDim.x);
    const uint32_t r0 = min((uint32_t)R, blockIdx.x * per), r1 = min((uint32_t)R, r0 + per);
    for (uint32_t r = r0 + warp; r < r1; r += kWarps) {
      const int e = find_expert(offs, p.E, (int)r);  // offs[e] <= r < offs[e + 1]
      int c = 0;
      for (int cc = 1; cc < kWarps; ++cc)
        if (hist[cc * p.E + e] <= (int)r) c = cc;
      int q = (int)r - hist[c * p.E + e];
      const uint32_t cend = (uint32_t)min(R, (int64_t)(c + 1) * CH);
      uint32_t slot = 0;
      for (uint32_t b = (uint32_t)(c * CH); b < cend; b += 32) {
        const uint32_t sl = b + lane;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, sl < cend && idx_s[sl] == (uint32_t)e);
        const int n = __popc(m);
        if (q < n) {  // the (q+1)-th set bit of m
          slot = b + __fns(m, 0, q + 1);
          break;
        }
        q -= n;
      }
      if (lane == 0) {
        tor[r - r0] = slot / (uint32_t)p.k;
        p.row_of_slot[slot] = r;
      }
    }
    __syncthreads();
    // rows [r0, r1) of x_d: x_d[r] = x[token_of_row[r]], 16-byte vectors
    const uint32_t vpr = (uint32_t)p.H / 8;  // 16-byte vectors per row
    const uint4* xs = reinterpret_cast<const uint4*>(p.x);
    uint4* xd = reinterpret_cast<uint4*>(p.x_d);
    const uint32_t nvec = (r1 - r0) * vpr;
    constexpr int kInFlight = 8;  // 16-byte loads issued before their stores
    for (uint32_t i0 = threadIdx.x; i0 < nvec; i0 += blockDim.x * kInFlight) {
      uint4 v[kInFlight];
      uint32_t dst[kInFlight];
#pragma unroll
      for (int b = 0; b < kInFlight; ++b) {
        const uint32_t i = i0 + b * blockDim.x;
        if (i < nvec) {
          const uint32_t rr = i / vpr, c = i - rr * vpr;
          dst[b] = (r0 + rr) * vpr + c;
          v[b] = ld_nc_v4(xs + (size_t)tor[rr] * vpr + c);
        }
      }
#pragma unroll
      for (int b = 0; b < kInFlight; ++b)
        if (i0 + b * blockDim.x < nvec) st_v4(xd + dst[b], v[b]);
    }
    // x_d is read by TMA (other CTAs' gate/up producers), and TMA refills this scratch shared
    // memory: generic writes made visible to the async proxy, then the rows are counted per
    // m-tile (a producer loads an m-tile's A rows once its count equals its rows)
    fence_proxy_async_all();
    __syncthreads();
    if (threadIdx.x == 0 && r0 < r1) {
      __threadfence();
      atomicAdd(ros_count, r1 - r0);  // row_of_slot entries written (the combine waits for R)
      for (uint32_t r = r0; r < r1;) {
        const int e = find_expert(offs, p.E, (int)r);  // offs[e] <= r < offs[e + 1]
        const int m = ((int)r - offs[e]) / BM;
        const uint32_t end = min(r1, (uint32_t)min(offs[e + 1], offs[e] + (m + 1) * BM));
        atomicAdd(gathered + pref[e] + m, end - r);
        r = end;
      }
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- 3. gate/up, 4. down
  // One tile list: the gate/up tiles, then the down tiles, claimed dynamically (a global counter)
  // so that CTAs finish together.  No grid barrier between the GEMMs: the gate/up epilogue counts
  // the stored warps of every m-tile, and the down producer loads the A rows (a) of an m-tile
  // only once all 4 NT_gu warps of it have stored.  Every gate/up tile is claimed before any down
  // tile and its CTA completes it without waiting on anything, so every wait ends.
  if (!*ring.abort_f) {
    TcParams gu = p.gu, dn = p.dn;
    gu.offsets = offs;
    dn.offsets = offs;
    gu.ready_wait = gathered;  // target 0: the rows of the m-tile
    gu.ready_target = 0u;
    gu.ready_signal = p.mtile_ready;
    dn.ready_wait = p.mtile_ready;
    dn.ready_target = 4u * (unsigned)gu.NT;
    dn.ready_signal = p.mtile_ready + p.n_mtiles;  // y: per (m-tile, n-tile), for the combine
    dn.signal_nt = dn.NT;
    const int n_gu = pref[p.E] * gu.NT, total = n_gu + pref[p.E] * dn.NT;
    int q = 0;
    uint32_t ph = 0;
    if (warp == 0) {
      if (lane == 0) {
        fence_proxy_async_global();
        bool first = true;
        while (wait_bounded(tr.empty(q), ph ^ 1u, ring.abort_f, p.status)) {
          int t = first ? *first_tile : (int)(gridDim.x + atomicAdd(p.tile_count, 1u));
          first = false;
          if (t >= total) t = -1;
          tr.ids[q] = t;
          mbar_arrive(tr.full(q));
          if (t < 0) break;
          const bool ok =
              t < n_gu
                  ? producer_tile<true, true>(&map_xd, &map_gate, &map_up, gu, pref, ring, pst, t)
                  : producer_tile<false, true>(&map_a, &map_down, &map_down, dn, pref, ring, pst,
                                               t - n_gu);
          if (!ok) break;
          if (++q == kTileSlots) {
            q = 0;
            ph ^= 1u;
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        while (wait_bounded(tr.full(q), ph, ring.abort_f, p.status)) {
          const int t = tr.ids[q];
          mbar_arrive(tr.empty(q));
          if (t < 0 || !mma_tile<BF16>(t < n_gu ? gu : dn, ring, mst)) break;
          if (++q == kTileSlots) {
            q = 0;
            ph ^= 1u;
          }
        }
      }
    } else {
      while (true) {
        const bool ok = wait_bounded(tr.full(q), ph, ring.abort_f, p.status);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
        const int t = tr.ids[q];
        __syncwarp();
        if (lane == 0) mbar_arrive(tr.empty(q));
        if (t < 0) break;
        const bool done = t < n_gu
                              ? epilogue_tile<true, BF16, true>(gu, pref, ring, est, t, warp, lane)
                              : epilogue_tile<false, BF16, true>(dn, pref, ring, est, t - n_gu,
                                                                 warp, lane);
        if (!done) break;
        if (++q == kTileSlots) {
          q = 0;
          ph ^= 1u;
        }
      }
    }
  }
  __syncthreads();  // this CTA's GEMM roles are done (no grid barrier: see the combine)

  // ---------------------------------------------------------------- 5. combine
  // Item (token t, 256-column chunk c) reads column tile c of the down GEMM for the k rows of
  // t: it waits only for those tiles' epilogue warps (a per-(m-tile, n-tile) count), so it can
  // start while other CTAs still finish their last GEMM tiles.  This CTA got here after the
  // claim counter ran out, so every tile it may wait for is held by a CTA that completes it.
  if (!*ring.abort_f) {
    const int64_t chunks = (int64_t)p.H * 2 / 16;
    const int64_t wpt = (chunks + 31) / 32;  // = the down GEMM's n-tiles (256 columns each)
    const unsigned* y_ready = p.mtile_ready + p.n_mtiles;
    int ros_ok = 1;
    if (lane == 0) ros_ok = wait_count(ros_count, (unsigned)R, ring.abort_f, p.status);
    ros_ok = __shfl_sync(0xFFFFFFFFu, ros_ok, 0);
    __syncwarp();  // orders lane 0's acquire before every lane's row_of_slot reads
    for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; ros_ok && it < (int64_t)p.T * wpt;
         it += (int64_t)gridDim.x * kWarps) {
      const int64_t t = (uint32_t)it / (uint32_t)wpt;  // 32-bit division (it < T * wpt)
      const int c = (int)(it - t * wpt);
      bool ok = true;
      for (int j = lane; j < p.k; j += 32) {
        const uint32_t r = ld_cg_u32(p.row_of_slot + t * p.k + j);
        if (r != kInvalidRow) {
          const int e = find_expert(offs, p.E, (int)r);  // offs[e] <= r < offs[e + 1]
          const int gm = pref[e] + ((int)r - offs[e]) / BM;
          ok &= wait_count(y_ready + (size_t)gm * wpt + c, 4u, ring.abort_f, p.status);
        }
      }
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      __syncwarp();  // each lane's acquire of its row's count before any lane reads the k rows
      combine_warp<TX, TL, true, true, 8>(reinterpret_cast<const TX*>(p.x_d), p.row_of_slot,
                                       reinterpret_cast<const TL*>(p.w), t, p.H, p.k, c,
                                       reinterpret_cast<TX*>(p.out), lane);
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

template <typename TL, bool BF16, bool SIG>
cudaError_t launch_t(const FusedDecodeArgs& f, cudaStream_t s) {
  auto kern = moe_decode_fused<TL, BF16, SIG>;
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
  p.gate = f.gate;
  p.up = f.up;
  p.T = (int)f.T;
  p.E = f.E;
  p.H = f.H;
  p.I = f.I;
  p.k = f.k;
  p.renorm = f.renorm;
  p.bias = f.bias;
  p.G = f.G;
  p.SG = f.SG;
  p.top_two = f.top_two;
  p.scale = f.scale;
  p.idx = f.idx;
  p.w = f.w;
  p.row_of_slot = f.row_of_slot;
  p.offsets = f.offsets;
  p.x_d = f.x_d;
  p.a = f.a;
  p.out = f.out;
  p.status = f.status;
  p.grid_count = f.grid_count;
  p.tile_count = f.tile_count;
  p.mtile_ready = f.mtile_ready;
  p.n_mtiles = (int)((R + BM - 1) / BM + f.E + 1);
  p.n_ready = p.n_mtiles * (2 + (f.H + BN - 1) / BN) + 1;
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

template <bool SIG>
cudaError_t launch_r(const FusedDecodeArgs& f, int ldt, int wdt, cudaStream_t s) {
  const bool bf = wdt == MOE_BF16;
  switch (ldt) {
    case MOE_F32: return bf ? launch_t<float, true, SIG>(f, s) : launch_t<float, false, SIG>(f, s);
    case MOE_F16: return bf ? launch_t<__half, true, SIG>(f, s) : launch_t<__half, false, SIG>(f, s);
    case MOE_BF16:
      return bf ? launch_t<__nv_bfloat16, true, SIG>(f, s)
                : launch_t<__nv_bfloat16, false, SIG>(f, s);
  }
  return cudaErrorInvalidValue;
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
  return f.sigmoid ? launch_r<true>(f, ldt, wdt, s) : launch_r<false>(f, ldt, wdt, s);
}

}  // namespace moe
