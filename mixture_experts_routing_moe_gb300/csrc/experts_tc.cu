// bf16 / f16 SwiGLU experts on 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
// SwiGluExperts::forward_dispatched of the ruDNN user guide, §5 "Expertengewichte und Verteilung":
//   kernel gate/up:  a[r, i] = silu(x_d[r] . gate[e, i]) * (x_d[r] . up[e, i])   (a stored in wdt)
//   kernel down:     y[r, h] = a[r] . down[e, h]                                   (y stored in wdt)
// over the ragged row groups offsets[e] .. offsets[e+1]-1 of the dispatched rows.
//
// Two variants share the structure below: a CTA kernel (one 128 x 256 tile per CTA, its warp
// roles in gemm_cta.cuh) and a CTA-pair kernel (one 256 x 256 tile per cluster of two CTAs,
// cta_group::2, see further down); the launcher takes the pair when experts average at least 128
// rows.
// Both kernels are persistent (one CTA per SM) with three warp roles:
//   warp 0     TMA producer: per 64-deep K slice loads a 128-row A tile (x_d or a) and a
//              256-row B tile into a 4-stage shared-memory ring (128-byte swizzle).  For
//              gate/up the B tile is 128 rows of gate followed by the same 128 rows of up, so
//              one N = 256 MMA yields both projections of 128 intermediate columns.
//   warp 1     MMA issuer (one thread): tcgen05.mma kind::f16, M = 128, N = 256, K = 16, FP32
//              accumulators in TMEM, double-buffered (2 x 256 of the 512 columns) so the epilogue
//              of one tile overlaps the MMAs of the next.  tcgen05.commit frees ring slots.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (each warp reads its 32-lane quarter =
//              32 tile rows), silu(g) * u (gate/up) or plain cast (down), 16-byte stores, masked
//              to the expert's rows and to the valid columns.
// Tiles are (expert, m-tile, n-tile); the list is derived on the device from the offsets.  Within
// an expert the smaller operand (the expert's rows of x_d / a, or its weights) stays resident in
// L2 (evict_last) while the larger one streams through it (evict_normal).
// Every wait on an mbarrier is bounded (about a second); on expiry the CTA records the timeout in
// the status word, stops issuing, lets in-flight copies and MMAs land, frees TMEM and exits.
#include <atomic>
#include <cuda.h>

#include "common.cuh"
#include "gemm_cta.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tiles.cuh"

namespace moe {
namespace {
using namespace tc;
using namespace cta_gemm;

template <bool GATEUP, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    moe_experts_tc(const __grid_constant__ CUtensorMap mapA,
                   const __grid_constant__ CUtensorMap mapB0,
                   const __grid_constant__ CUtensorMap mapB1, const TcParams p) {
  extern __shared__ uint8_t tc_smem_raw[];
  uint32_t* tmem_slot;
  int* pref;
  Ring ring = carve_ring(tc_smem_raw, &tmem_slot, &pref);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) init_ring(ring);
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (warp == 2) build_mtile_prefix(p.offsets, p.E, BM, pref, lane);
  if (warp == 0 && lane == 0) {
    tma_prefetch(&mapA);
    tma_prefetch(&mapB0);
    if (GATEUP) tma_prefetch(&mapB1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  ring.tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      ProducerState st;
      producer<GATEUP, false>(&mapA, &mapB0, &mapB1, p, pref, ring, st);
      if (*ring.abort_f) producer_drain(ring, st);  // any role gave up: let copies land
    }
  } else if (warp == 1) {
    if (lane == 0) {
      MmaState st;
      mma<BF16>(p, pref, ring, st);
      mma_drain(ring);
    }
  } else {
    EpilogueState st;
    epilogue<GATEUP, BF16, false>(p, pref, ring, st, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(ring.tmem_base, kTmemCols);
  }
}

// ================================================================ CTA-pair kernels
// A cluster of two CTAs on neighbouring SMs computes one 256 x 256 tile with cta_group::2 MMAs:
// CTA r loads rows [128 r, 128 r + 128) of the tile's A rows and the r-th 128-row half of its B
// rows.  For gate/up the B halves interleave the two projections: CTA r holds gate rows and up
// rows [64 r, 64 r + 64) of the 128 intermediate columns, so accumulator columns 0-63 / 64-127
// are gate / up of one 64-column group and 128-191 / 192-255 gate / up of the other.  For down
// the halves are the two halves of the 256 output columns.  One thread of CTA 0 issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16); the MMA reads both CTAs' shared memory
// at the same offsets and leaves each CTA's 128 accumulator rows in that CTA's TMEM.
// An expert's last tile with at most 128 rows runs as M = 128 (64 rows per CTA): each CTA's TMEM
// lanes 0-63 then hold its 64 rows for N columns 0-127 and lanes 64-127 the same rows for N
// columns 128-255, in TMEM columns 0-127 (layout measured on GB300).  This keeps the padding of
// ragged experts at 128-row granularity; such a tile's CTAs load 64 A rows each (a 64-row map).  With half of B per CTA a stage is 32 KB, so six stages fit, and each CTA pulls a
// third fewer bytes per FLOP through L2 than a single-CTA 128 x 256 tile.
// GEMMs with long tiles (at least 64 K blocks) claim them dynamically: a pair's first tile is tile
// `pair`; CTA 0's producer claims each later one from a global counter, one tile ahead, and writes
// its id into an 8-slot ring in both CTAs (full / empty mbarriers; the id reaches CTA 1 by a
// cluster store ordered by a release arrive), and every role of both CTAs reads the ids in order,
// so pairs that finish early take the last tiles instead of a static share.  Short tiles keep the
// static order pair, pair + P, ... (their boundaries would pay the hand-off more often).  Each role walks its (increasing) tiles with a TileCursor over a shared-memory
// copy of the offsets, so the MMA issuer's step from one tile to the next holds no global load,
// binary search or 64-bit division while the tensor pipe drains.
// Synchronisation: both CTAs' TMA loads signal CTA 0's full barrier (CTA 0 arms it for both);
// CTA 0's MMA commits are multicast to the empty / tmem-full barriers of both CTAs; all eight
// epilogue warps arrive on CTA 0's tmem-empty barrier.  Waits are bounded as in the CTA kernel.
constexpr int BM2 = 256, STAGES2 = 6;
constexpr int A2_BYTES = 128 * BK * 2;  // 16 KB
constexpr int B2_BYTES = 128 * BK * 2;  // 16 KB: half of the 256-row B tile
constexpr int STAGE2_BYTES = A2_BYTES + B2_BYTES;
// down epilogue: one 32-row x 64-column bf16 staging buffer (4 KB) per epilogue warp
constexpr int kStage2Out = 32 * 128;
constexpr int kBar2Bytes = 512;  // mbarriers, TMEM slot, abort flag, tile-id ring
constexpr size_t kSmem2Bytes = 1024 + (size_t)STAGES2 * STAGE2_BYTES + kBar2Bytes +
                               2 * (kMaxExperts + 4) * sizeof(int) + 4 * kStage2Out;

// The GEMMs the pair kernel runs.  Forward: gate/up (A = x_d, B = interleaved gate / up halves,
// a = silu(g) u) and down (A = a, B = down, plain cast).  Expert backward (ruDNN user guide §12):
//   kDa   da = dy down_e          A = dy [rows, H], B = down_e [H, I] with N (= I) contiguous,
//                                 FP32 output
//   kGu   g, u = x_d gate_e^T, x_d up_e^T recomputed as in the forward; epilogue with da:
//                                 s = sigmoid(g), dg = da u s (1 + g (1 - s)), du = da g s,
//                                 a = g s u -> dg | du [rows, 2I] and a [rows, I]
//   kDin  dinput = [dg du] [gate_e; up_e]   A = dg | du [rows, 2I], B = gate_e / up_e [I, H] with
//                                 N (= H) contiguous (k < I from gate, else up), plain cast
// A B operand with N contiguous is loaded as two 64-column boxes per CTA half and described as an
// MN-major 128-byte-swizzled matrix (boxes 8 KB apart).
enum PairKind { kGateUp = 0, kDown = 1, kDa = 2, kGu = 3, kDin = 4 };

// Tile-id ring of the pair kernel (dynamic claims): slot q holds the id CTA 0's producer claimed.
constexpr int kRing = 8;
// GEMMs with at least this many 64-deep K blocks a tile claim their tiles dynamically.
constexpr int kDynamicMinKB = 64;
// 32-bit store into the shared memory of another CTA of the cluster (address from mapa).
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// try_wait with acquire at cluster scope: the phase was completed by another CTA's release.
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait_bounded_cl(uint32_t bar, uint32_t parity,
                                                volatile int* abort_f, unsigned* status) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if (*abort_f) return false;
    if (clock64() - t0 > kWaitLimit) {
      *abort_f = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

template <int KIND, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    moe_experts_tc2(const __grid_constant__ CUtensorMap mapA,
                    const __grid_constant__ CUtensorMap mapB0,
                    const __grid_constant__ CUtensorMap mapB1,
                    const __grid_constant__ CUtensorMap mapAh, const TcParams p) {
  constexpr bool GATEUP = KIND == kGateUp || KIND == kGu;  // B: interleaved gate / up halves
  constexpr bool B_MN = KIND == kDa || KIND == kDin;       // B stored with N contiguous
  constexpr int ES = KIND == kDa ? 4 : 2;                  // output element size
  extern __shared__ uint8_t tc_smem_raw[];
  const uint32_t raw = smem_u32(tc_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = tc_smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES2 * STAGE2_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES2 + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES2 + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES2 + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES2 + 4);
  auto rfull = [&](int q) { return bar0 + 8u * (2 * STAGES2 + 5 + q); };           // each CTA
  auto rempty = [&](int q) { return bar0 + 8u * (2 * STAGES2 + 5 + kRing + q); };  // CTA 0's
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES2 + 5 + 2 * kRing);
  volatile int* abort_f = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* rids = reinterpret_cast<volatile int*>(tmem_slot + 2);  // kRing tile ids
  int* pref = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + kBar2Bytes);
  int* offs = pref + (kMaxExperts + 4);  // a copy of offsets[0 .. E]
  // staging of the down epilogue, after the barriers, the prefix and the offsets
  const uint32_t stage_out = base + STAGES2 * STAGE2_BYTES + kBar2Bytes +
                             (uint32_t)(2 * (kMaxExperts + 4) * sizeof(int));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = (int)cluster_id_x(), npairs = (int)ncluster_x();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 8);
    }
    mbar_init(drain_bar, 1);
    for (int q = 0; q < kRing; ++q) {
      mbar_init(rfull(q), 1);
      // readers of every id: CTA 0's MMA thread and epilogue warps, CTA 1's producer and
      // epilogue warps
      mbar_init(rempty(q), 10);
    }
    *abort_f = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc2(smem_u32(tmem_slot), kTmemCols);
  if (warp == 2) build_mtile_prefix(p.offsets, p.E, BM2, pref, lane);
  if (warp == 3)
    for (int i = lane; i <= p.E; i += 32) offs[i] = __ldg(p.offsets + i);
  if (warp == 0 && lane == 0) {
    tma_prefetch(&mapA);
    tma_prefetch(&mapB0);
    if (GATEUP || KIND == kDin) tma_prefetch(&mapB1);
    tma_prefetch(&mapAh);
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs: barriers initialised, TMEM allocated, prefix built
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = pref[p.E] * p.NT;
  // Tile order.  Dynamic (p.tile_ctr set): a pair's first tile is tile `pair`, later ones are
  // claimed from the global counter by CTA 0's producer, which writes each id into both CTAs'
  // rings; every role of both CTAs reads the ids in order (so the pairs that finish early take
  // the last tiles).  Static: pair, pair + P, ...  Either way a role's tiles increase.
  const bool dyn = p.tile_ctr != nullptr;
  int rq = 0, st_t = -1;
  uint32_t rph = 0;
  auto claim = [&]() -> int {  // CTA 0's producer: the next tile, published to both CTAs
    if (!dyn) {
      st_t = st_t < 0 ? pair : st_t + npairs;
      return st_t < total ? st_t : -1;
    }
    if (!wait_bounded(rempty(rq), rph ^ 1u, abort_f, p.status)) return -2;
    int t = st_t < 0 ? pair : npairs + (int)atomicAdd(p.tile_ctr, 1u);
    st_t = t;
    if (t >= total) t = -1;
    rids[rq] = t;
    st_cluster_u32(map_to_rank(smem_u32((const void*)(rids + rq)), 1), (uint32_t)t);
    mbar_arrive(rfull(rq));
    mbar_arrive_cluster(map_to_rank(rfull(rq), 1));  // release: the store above lands first
    if (++rq == kRing) {
      rq = 0;
      rph ^= 1u;
    }
    return t;
  };
  // Every other role (one thread each: the producer of CTA 1, the MMA thread, lane 0 of each
  // epilogue warp): the next id (-1: none left, -2: a wait gave up).
  auto consume = [&](bool arrive) -> int {
    if (!dyn) {
      st_t = st_t < 0 ? pair : st_t + npairs;
      return st_t < total ? st_t : -1;
    }
    const bool ok = leader ? wait_bounded(rfull(rq), rph, abort_f, p.status)
                           : wait_bounded_cl(rfull(rq), rph, abort_f, p.status);
    if (!ok) return -2;
    const int t = rids[rq];
    if (arrive) {
      if (leader) mbar_arrive(rempty(rq));
      else mbar_arrive_cluster(map_to_rank(rempty(rq), 0));
    }
    if (++rq == kRing) {
      rq = 0;
      rph ^= 1u;
    }
    return t;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      int stage = 0, armed = 0;
      uint32_t phase = 0;
      bool stop = false;
      const uint64_t keep = policy_evict_last(), other = policy_evict_normal();
      TileCursor<BM2> cur(pref, p.E, p.NT, p.KB * BK);
      // CTA 0 claims and publishes the next tile before loading this one, so neither producer
      // waits for a claim's round trip at a tile boundary
      int t = leader ? claim() : consume(true);
      while (t >= 0 && !stop) {
        const int tn = leader ? claim() : 0;
        int e, m, n;
        const bool a_res = cur.next(t, e, m, n);
        const uint64_t pa = a_res ? keep : other, pb = a_res ? other : keep;
        const int r0 = offs[e] + m * BM2;
        const bool half = offs[e + 1] - r0 <= 128;
        const int a_row = r0 + (int)rank * (half ? 64 : 128);
        const int b_row = GATEUP ? e * p.b_rows + n * (BN / 2) + (int)rank * 64
                                 : e * p.b_rows + n * BN + (int)rank * 128;
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_f, p.status)) {
            stop = true;
            break;
          }
          const uint32_t sa = base + stage * STAGE2_BYTES, sb = sa + A2_BYTES;
          const uint32_t fb = map_to_rank(full_bar(stage), 0);
          // a half tile's CTA loads only its 64 A rows (the MMA reads no more of them)
          if (leader) mbar_expect_tx(full_bar(stage), 2 * (half ? STAGE2_BYTES - A2_BYTES / 2 : STAGE2_BYTES));
          tma_load_2d_pair(sa, half ? &mapAh : &mapA, fb, kb * BK, a_row, pa);
          if (GATEUP) {  // 64 gate rows, then the same 64 up rows
            tma_load_2d_pair(sb, &mapB0, fb, kb * BK, b_row, pb);
            tma_load_2d_pair(sb + B2_BYTES / 2, &mapB1, fb, kb * BK, b_row, pb);
          } else if (!B_MN) {
            tma_load_2d_pair(sb, &mapB0, fb, kb * BK, b_row, pb);
          } else {
            // this CTA's 128 output columns as two 64-column boxes of the 64 K rows of the stage:
            // down rows e H + k (kDa), or gate rows e I + k for k < I and up rows e I + k - I
            const CUtensorMap* mb = &mapB0;
            int kr = e * p.b_rows + kb * BK;
            if (KIND == kDin) {
              const int k0 = kb * BK;
              if (k0 >= p.I) mb = &mapB1;
              kr = e * p.I + (k0 >= p.I ? k0 - p.I : k0);
            }
            const int c0 = n * BN + (int)rank * 128;
            tma_load_2d_pair(sb, mb, fb, c0, kr, pb);
            tma_load_2d_pair(sb + B2_BYTES / 2, mb, fb, c0 + 64, kr, pb);
          }
          ++armed;
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
        }
        t = leader ? tn : consume(true);
      }
      if (*abort_f && leader) {  // let copies still in flight land before the pair exits
        for (int i = 0; i < min(armed, STAGES2); ++i) {
          if (stage == 0) {
            stage = STAGES2 - 1;
            phase ^= 1u;
          } else {
            --stage;
          }
          wait_drain(full_bar(stage), phase);
        }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ------------------------------------------------------------ MMA issuer (CTA 0 only)
      constexpr uint32_t bmn = B_MN ? 1u << 16 : 0u;  // instruction descriptor: B MN-major
      constexpr uint32_t idesc_full = make_idesc(BF16, BM2, BN) | bmn;
      constexpr uint32_t idesc_half = make_idesc(BF16, BM2 / 2, BN) | bmn;
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool stop = false;
      TileCursor<BM2> cur(pref, p.E, p.NT, p.KB * BK);
      for (int t = consume(true); t >= 0 && !stop; t = consume(true)) {
        int e, m, n;
        cur.next(t, e, m, n);
        const int r0 = offs[e] + m * BM2;
        const uint32_t idesc = offs[e + 1] - r0 <= 128 ? idesc_half : idesc_full;
        if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_f, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, abort_f, p.status)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + stage * STAGE2_BYTES, sb = sa + A2_BYTES;
          const uint64_t da = make_sdesc(sa);
          const uint64_t db = B_MN ? make_sdesc_mn_box(sb, B2_BYTES / 2) : make_sdesc(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // K = 16: 32 bytes (K-major) or 2 KB (MN-major)
            umma2_f16(d_tmem, da + 2u * kk, db + (B_MN ? 128u : 2u) * kk, idesc, (kb | kk) != 0);
          umma_commit2(empty_bar(stage), 0x3);
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
        umma_commit2(tfull_bar(acc), 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit2(drain_bar, 0x1);  // arrives once every MMA issued above has completed
      wait_drain(drain_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- epilogue (warps 2..5, both)
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    TileCursor<BM2> cur(pref, p.E, p.NT, p.KB * BK);
    while (true) {
      int t = 0;
      if (lane == 0) t = consume(true);  // one reader per warp; the id goes to every lane
      t = __shfl_sync(0xFFFFFFFFu, t, 0);
      if (t < 0) break;
      int e, m, n;
      cur.next(t, e, m, n);
      const bool ok = wait_bounded(tfull_bar(acc), acc_phase, abort_f, p.status);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      const int r0 = offs[e] + m * BM2;
      const int r_end = offs[e + 1];
      const bool half = r_end - r0 <= 128;
      // full tile: lane quarter q holds rows 128 rank + 32 q + lane over all N columns;
      // half tile: quarters 0-1 hold rows 64 rank + 32 q + lane for N columns 0-127, quarters 2-3
      // the same rows for N columns 128-255 (TMEM columns 0-127 in both cases)
      const int row =
          r0 + (half ? (int)rank * 64 + (q & 1) * 32 + lane : (int)rank * 128 + q * 32 + lane);
      const int nhalf = half ? (q >> 1) : 0;  // which half of N this warp holds (half tiles)
      const bool valid = row < r_end;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      uint8_t* orow = p.out + (size_t)row * p.N * ES;
      if (KIND == kGu) {
        // as the gate/up epilogue, with the SwiGLU gradient: dg | du and a for 32 columns at once
        const float* darow = p.da + (size_t)row * p.I;
        uint8_t* arow = p.out1 + (size_t)row * p.I * 2;
        uint8_t* dgrow = p.out + (size_t)row * 2 * p.I * 2;
#pragma unroll 1
        for (int j = 0; j < (half ? 2 : 4); ++j) {
          const int gc = half ? 32 * j : (j & 1) * 32 + (j >> 1) * 128;
          uint32_t g[32], u[32];
          tmem_ld32(taddr + gc, g);
          tmem_ld32(taddr + gc + 64, u);
          tmem_wait_ld();
          const int col0 = n * (BN / 2) + (half ? 64 * nhalf + 32 * j : 32 * j);
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (col0 + v * 8 < p.I) {
                float dv[8];
                *reinterpret_cast<uint4*>(dv) = ld_nc_v4(darow + col0 + v * 8);
                *reinterpret_cast<uint4*>(dv + 4) = ld_nc_v4(darow + col0 + v * 8 + 4);
                uint32_t pg[4], pu[4], pa[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  float dgv[2], duv[2], av[2];
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    const float gv = __uint_as_float(g[v * 8 + i * 2 + h]);
                    const float uv = __uint_as_float(u[v * 8 + i * 2 + h]);
                    const float sg = 1.f / (1.f + __expf(-gv));
                    const float act = gv * sg, d = dv[i * 2 + h];
                    dgv[h] = d * uv * sg * (1.f + gv * (1.f - sg));
                    duv[h] = d * act;
                    av[h] = act * uv;
                  }
                  pg[i] = pack2<BF16>(dgv[0], dgv[1]);
                  pu[i] = pack2<BF16>(duv[0], duv[1]);
                  pa[i] = pack2<BF16>(av[0], av[1]);
                }
                st_v4(dgrow + (size_t)(col0 + v * 8) * 2, make_uint4(pg[0], pg[1], pg[2], pg[3]));
                st_v4(dgrow + (size_t)(p.I + col0 + v * 8) * 2,
                      make_uint4(pu[0], pu[1], pu[2], pu[3]));
                st_v4(arow + (size_t)(col0 + v * 8) * 2, make_uint4(pa[0], pa[1], pa[2], pa[3]));
              }
            }
          }
        }
      } else if (KIND == kDa) {
        // FP32 output.  Full tile with all 32 rows of this warp in the expert: 32-column chunks
        // (128 bytes a row) staged through shared memory and written as whole 128-byte lines, as
        // below; otherwise this lane's row, 16 bytes at a time.
        const bool staged = !half && __all_sync(0xFFFFFFFFu, valid);
        const uint32_t buf = stage_out + (uint32_t)(q * kStage2Out);
        const int row0 = r0 + (int)rank * 128 + q * 32;
#pragma unroll 1
        for (int c = 0; c < (half ? 4 : 8); ++c) {
          uint32_t r[32];
          tmem_ld32(taddr + c * 32, r);
          tmem_wait_ld();
          const int col0 = n * BN + 128 * nhalf + c * 32;
          if (staged && col0 + 32 <= p.N) {
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), r[4 * j], r[4 * j + 1],
                           r[4 * j + 2], r[4 * j + 3]);
            __syncwarp();
#pragma unroll
            for (int pass = 0; pass < 8; ++pass) {
              const int rr = pass * 4 + (lane >> 3), ch = lane & 7;
              const uint4 v = ld_shared_v4(buf + rr * 128 + ((ch ^ (rr & 7)) << 4));
              st_v4(p.out + ((size_t)(row0 + rr) * p.N + col0 + ch * 4) * 4, v);
            }
          } else if (valid) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              if (col0 + v * 4 < p.N)
                st_v4(orow + (size_t)(col0 + v * 4) * 4,
                      make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]));
          }
        }
      } else if (GATEUP) {
        // output column group j (32 columns): gate at accumulator column gc, up at gc + 64;
        // full tile: j = 0..3, gc = (j & 1) * 32 + (j >> 1) * 128, outputs n*128 + 32 j;
        // half tile: j = 0..1, gc = 32 j, outputs n*128 + 64 nhalf + 32 j
#pragma unroll 1
        for (int j = 0; j < (half ? 2 : 4); ++j) {
          const int gc = half ? 32 * j : (j & 1) * 32 + (j >> 1) * 128;
          uint32_t g[32], u[32];
          tmem_ld32(taddr + gc, g);
          tmem_ld32(taddr + gc + 64, u);
          tmem_wait_ld();
          const int col0 = n * (BN / 2) + (half ? 64 * nhalf + 32 * j : 32 * j);
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (col0 + v * 8 < p.N) {
                uint32_t pk[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  float a2[2];
#pragma unroll
                  for (int h = 0; h < 2; ++h) {
                    const float gv = __uint_as_float(g[v * 8 + i * 2 + h]);
                    const float uv = __uint_as_float(u[v * 8 + i * 2 + h]);
                    a2[h] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                  }
                  pk[i] = pack2<BF16>(a2[0], a2[1]);
                }
                st_v4(orow + (size_t)(col0 + v * 8) * 2, make_uint4(pk[0], pk[1], pk[2], pk[3]));
              }
            }
          }
        }
      } else if (!half && __all_sync(0xFFFFFFFFu, valid)) {
        // full tile, all 32 rows of this warp in the expert: 64-column chunks staged through
        // shared memory (16-byte chunk j of row r at j ^ (r & 7)) and written as whole 128-byte
        // lines, 8 lanes per row, instead of one 16-byte piece of 32 different rows per store
        const uint32_t buf = stage_out + (uint32_t)(q * kStage2Out);
        const int row0 = r0 + (int)rank * 128 + q * 32;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32], r2[32];
          tmem_ld32(taddr + c * 64, r);
          tmem_ld32(taddr + c * 64 + 32, r2);
          tmem_wait_ld();
          const int col0 = n * BN + c * 64;
          if (col0 + 64 <= p.N) {
            __syncwarp();  // every lane is done reading the previous chunk out of `buf`
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t* src = j < 4 ? r + 8 * j : r2 + 8 * (j - 4);
              st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4),
                           pack2<BF16>(__uint_as_float(src[0]), __uint_as_float(src[1])),
                           pack2<BF16>(__uint_as_float(src[2]), __uint_as_float(src[3])),
                           pack2<BF16>(__uint_as_float(src[4]), __uint_as_float(src[5])),
                           pack2<BF16>(__uint_as_float(src[6]), __uint_as_float(src[7])));
            }
            __syncwarp();
#pragma unroll
            for (int pass = 0; pass < 8; ++pass) {
              const int rr = pass * 4 + (lane >> 3), ch = lane & 7;
              const uint4 v = ld_shared_v4(buf + rr * 128 + ((ch ^ (rr & 7)) << 4));
              st_v4(p.out + ((size_t)(row0 + rr) * p.N + col0 + ch * 8) * 2, v);
            }
          } else {  // ragged N: this lane's row, 16 bytes at a time
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const int cc = col0 + v * 8;
              if (cc < p.N) {
                const uint32_t* src = v < 4 ? r + 8 * v : r2 + 8 * (v - 4);
                st_v4(orow + (size_t)cc * 2,
                      make_uint4(pack2<BF16>(__uint_as_float(src[0]), __uint_as_float(src[1])),
                                 pack2<BF16>(__uint_as_float(src[2]), __uint_as_float(src[3])),
                                 pack2<BF16>(__uint_as_float(src[4]), __uint_as_float(src[5])),
                                 pack2<BF16>(__uint_as_float(src[6]), __uint_as_float(src[7]))));
              }
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < (half ? 4 : 8); ++c) {
          uint32_t r[32];
          tmem_ld32(taddr + c * 32, r);
          tmem_wait_ld();
          const int col0 = n * BN + 128 * nhalf + c * 32;
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (col0 + v * 8 < p.N) {
                uint32_t pk[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  pk[i] = pack2<BF16>(__uint_as_float(r[v * 8 + i * 2]),
                                      __uint_as_float(r[v * 8 + i * 2 + 1]));
                st_v4(orow + (size_t)(col0 + v * 8) * 2, make_uint4(pk[0], pk[1], pk[2], pk[3]));
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync_all();  // no CTA leaves while its pair may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
// 2-D K-major map over a [rows, K] 16-bit matrix, box = 64 (K) x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, bool bf16, int64_t K, int64_t rows, int box_rows) {
  return tc::make_map_2d(m, ptr, bf16, K, rows, BK, box_rows);
}

template <bool GATEUP, bool BF16>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                       const TcParams& p, int64_t rows, int sms, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(moe_experts_tc<GATEUP, BF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  const int64_t upper = ((rows + BM - 1) / BM + p.E) * (int64_t)p.NT;  // >= number of tiles
  const int grid = (int)(upper < sms ? upper : sms);
  moe_experts_tc<GATEUP, BF16><<<grid, kThreads, kSmemBytes, s>>>(a, b0, b1, p);
  return cudaGetLastError();
}

template <int KIND, bool BF16>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                        const CUtensorMap& ah, const TcParams& p, int64_t rows, int dev,
                        cudaStream_t s) {
  auto kern = moe_experts_tc2<KIND, BF16>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmem2Bytes);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem2Bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2);
  // co-resident pairs on this device (queried once per device)
  // (relaxed atomics: host threads may race on the first query; every one stores the same value)
  static std::atomic<int> max_pairs[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int mp = max_pairs[dev].load(std::memory_order_relaxed);
  if (mp == 0) {
    err = cudaOccupancyMaxActiveClusters(&mp, kern, &cfg);
    if (err != cudaSuccess) return err;
    if (mp < 1) return cudaErrorLaunchOutOfResources;
    max_pairs[dev].store(mp, std::memory_order_relaxed);
  }
  const int64_t upper = ((rows + BM2 - 1) / BM2 + p.E) * (int64_t)p.NT;  // >= number of tiles
  const int pairs = (int)(upper < mp ? upper : mp);
  cfg.gridDim = dim3(2 * pairs);
  // Dynamic tile claims pay where tiles are long (the tail they remove is about half a tile);
  // short ones keep the static order, whose tile boundaries hold no hand-off.
  TcParams q = p;
  if (q.KB < kDynamicMinKB) q.tile_ctr = nullptr;
  if (q.tile_ctr && (err = cudaMemsetAsync(q.tile_ctr, 0, sizeof(unsigned), s)) != cudaSuccess)
    return err;
  return cudaLaunchKernelEx(&cfg, kern, a, b0, b1, ah, q);
}

template <bool BF16>
cudaError_t launch_tc_t(const void* x_d, const int32_t* offsets, int64_t rows, const void* gate,
                        const void* up, const void* down, int E, int H, int I, void* y, void* a,
                        unsigned* status, cudaStream_t s, cudaEvent_t between) {
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;

  // CTA pairs (256-row tiles) when experts average at least 128 rows; below that the pair's
  // taller tiles mostly multiply padding and single CTAs stream the weights as well.
  const bool pair = rows >= (int64_t)128 * E;
  CUtensorMap mx, mg, mu, ma, md;
  if (!make_map(&mx, x_d, BF16, H, rows, BM) || !make_map(&mg, gate, BF16, H, (int64_t)E * I, BN / 2) ||
      !make_map(&mu, up, BF16, H, (int64_t)E * I, BN / 2) || !make_map(&ma, a, BF16, I, rows, BM) ||
      !make_map(&md, down, BF16, I, (int64_t)E * H, pair ? BN / 2 : BN))
    return cudaErrorInvalidValue;

  // the pair kernels' tile-claim counter: byte 192 of the caller's 256-byte workspace header
  unsigned* tile_ctr = status ? status + 48 : nullptr;
  TcParams p1{offsets, (uint8_t*)a, status, E, I, (H + BK - 1) / BK, (I + BN / 2 - 1) / (BN / 2), I};
  p1.tile_ctr = tile_ctr;
  CUtensorMap mxh, mah;  // the pair kernel's half tiles load 64 rows of x_d / a per CTA
  if (pair) {  // the pair kernel loads gate and up in 64-row boxes (interleaved B halves)
    if (!make_map(&mg, gate, BF16, H, (int64_t)E * I, BN / 4) ||
        !make_map(&mu, up, BF16, H, (int64_t)E * I, BN / 4) ||
        !make_map(&mxh, x_d, BF16, H, rows, BM / 2) || !make_map(&mah, a, BF16, I, rows, BM / 2))
      return cudaErrorInvalidValue;
  }
  err = pair ? launch_pair<kGateUp, BF16>(mx, mg, mu, mxh, p1, rows, dev, s)
             : launch_one<true, BF16>(mx, mg, mu, p1, rows, sms, s);
  if (err != cudaSuccess) return err;
  if (between && (err = cudaEventRecord(between, s)) != cudaSuccess) return err;
  TcParams p2{offsets, (uint8_t*)y, status, E, H, (I + BK - 1) / BK, (H + BN - 1) / BN, H};
  p2.tile_ctr = tile_ctr;
  return pair ? launch_pair<kDown, BF16>(ma, md, md, mah, p2, rows, dev, s)
              : launch_one<false, BF16>(ma, md, md, p2, rows, sms, s);
}

template <bool BF16>
cudaError_t bwd_pair_t(const void* x_d, const int32_t* offsets, int64_t rows, const void* gate,
                       const void* up, const void* down, int E, int H, int I, const void* dy,
                       float* da, void* dgdu, void* a, void* dinput, unsigned* status,
                       cudaStream_t s) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  CUtensorMap mA, mAh, mB0, mB1;
  // 1. da = dy down_e: down read as [E H, I] (N = I contiguous) in 64 x 64 boxes
  if (!make_map(&mA, dy, BF16, H, rows, BM) || !make_map(&mAh, dy, BF16, H, rows, BM / 2) ||
      !tc::make_map_2d(&mB0, down, BF16, I, (int64_t)E * H, 64, 64))
    return cudaErrorInvalidValue;
  unsigned* tile_ctr = status ? status + 48 : nullptr;  // byte 192 of the workspace header
  TcParams p1{offsets, (uint8_t*)da, status, E, I, (H + BK - 1) / BK, (I + BN - 1) / BN, H};
  p1.tile_ctr = tile_ctr;
  err = launch_pair<kDa, BF16>(mA, mB0, mB0, mAh, p1, rows, dev, s);
  if (err != cudaSuccess) return err;
  // 2. g, u recomputed (gate and up in 64-row K-major boxes, as the forward), SwiGLU gradient
  if (!make_map(&mA, x_d, BF16, H, rows, BM) || !make_map(&mAh, x_d, BF16, H, rows, BM / 2) ||
      !make_map(&mB0, gate, BF16, H, (int64_t)E * I, BN / 4) ||
      !make_map(&mB1, up, BF16, H, (int64_t)E * I, BN / 4))
    return cudaErrorInvalidValue;
  TcParams p2{offsets, (uint8_t*)dgdu, status, E, I, (H + BK - 1) / BK, (I + BN / 2 - 1) / (BN / 2), I};
  p2.da = da;
  p2.out1 = (uint8_t*)a;
  p2.I = I;
  p2.tile_ctr = tile_ctr;
  err = launch_pair<kGu, BF16>(mA, mB0, mB1, mAh, p2, rows, dev, s);
  if (err != cudaSuccess) return err;
  // 3. dinput = [dg du] [gate_e; up_e]: gate and up read as [E I, H] (N = H contiguous)
  if (!make_map(&mA, dgdu, BF16, 2 * (int64_t)I, rows, BM) ||
      !make_map(&mAh, dgdu, BF16, 2 * (int64_t)I, rows, BM / 2) ||
      !tc::make_map_2d(&mB0, gate, BF16, H, (int64_t)E * I, 64, 64) ||
      !tc::make_map_2d(&mB1, up, BF16, H, (int64_t)E * I, 64, 64))
    return cudaErrorInvalidValue;
  TcParams p3{offsets, (uint8_t*)dinput, status, E, H, 2 * I / BK, (H + BN - 1) / BN, I};
  p3.I = I;
  p3.tile_ctr = tile_ctr;
  return launch_pair<kDin, BF16>(mA, mB0, mB1, mAh, p3, rows, dev, s);
}

}  // namespace

cudaError_t launch_experts_bwd_pair(const void* x_d, const int32_t* offsets, int64_t rows,
                                    const void* gate, const void* up, const void* down, int wdt,
                                    int E, int H, int I, const void* dy, float* da, void* dgdu,
                                    void* a, void* dinput, unsigned* status, cudaStream_t s) {
  if (wdt == MOE_BF16)
    return bwd_pair_t<true>(x_d, offsets, rows, gate, up, down, E, H, I, dy, da, dgdu, a, dinput,
                            status, s);
  if (wdt == MOE_F16)
    return bwd_pair_t<false>(x_d, offsets, rows, gate, up, down, E, H, I, dy, da, dgdu, a,
                             dinput, status, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_experts_tc(const void* x_d, const int32_t* offsets, int64_t rows,
                              const void* gate, const void* up, const void* down, int wdt, int E,
                              int H, int I, void* y, void* a, unsigned* status, cudaStream_t s,
                              cudaEvent_t between) {
  if (wdt == MOE_BF16)
    return launch_tc_t<true>(x_d, offsets, rows, gate, up, down, E, H, I, y, a, status, s,
                             between);
  if (wdt == MOE_F16)
    return launch_tc_t<false>(x_d, offsets, rows, gate, up, down, E, H, I, y, a, status, s,
                              between);
  return cudaErrorInvalidValue;
}

}  // namespace moe
