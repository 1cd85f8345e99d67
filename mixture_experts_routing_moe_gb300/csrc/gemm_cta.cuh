// The single-CTA grouped GEMM of the SwiGLU experts (ruDNN user guide, §5 "Expertengewichte und
// Verteilung") as three warp roles that a persistent kernel runs over a tile list:
//   producer  (one thread)  TMA loads of a 128-row A tile and a 256-row B tile per 64-deep K slice
//                           into a 4-stage shared-memory ring (128-byte swizzle).  For gate/up
//                           the B tile is 128 rows of gate followed by the same 128 rows of up.
//   mma       (one thread)  tcgen05.mma kind::f16, M = 128, N = 256, K = 16, FP32 accumulators in
//                           TMEM, double-buffered (2 x 256 of 512 columns); commits free ring slots.
//   epilogue  (four warps)  tcgen05.ld of its 32-lane quarter, silu(g) * u (gate/up) or a plain
//                           cast (down), 16-byte stores masked to the expert's rows and columns.
// The ring, accumulator and phase state live in the role structs, so one kernel may run several
// GEMMs back to back over the same ring (the fused decode kernel does).  Every mbarrier wait is
// bounded; on expiry the role records the timeout and returns false.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tiles.cuh"

namespace moe {
namespace cta_gemm {
using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxExperts = 1024;
constexpr int kBarBytes = 256;  // ring + accumulator barriers, TMEM slot, abort flag
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + (size_t)STAGES * STAGE_BYTES +
                              kBarBytes + (kMaxExperts + 4) * sizeof(int);

// Tile t -> (expert e, m-tile m, n-tile n).  Inside an expert, the operand with fewer bytes
// (A: mt * 128 rows, B: NT * 256 rows, both K deep) is the one kept resident in L2 while the
// other streams through once: A resident -> n outer, m inner; B resident -> m outer, n inner.
// When the resident operand exceeds kResidentBytes it is cut into groups that do fit.
// Returns true when A is the resident operand.
constexpr long long kResidentBytes = 64ll << 20;
template <int TBM = BM>
__device__ __forceinline__ bool decode_tile(int t, const int* pref, int E, int NT, int K, int& e,
                                            int& m, int& n) {
  e = find_expert(pref, E, t / NT);
  const int local = t - pref[e] * NT;
  const int mt = pref[e + 1] - pref[e];
  const long long rows_fit = kResidentBytes / ((long long)K * 2);
  if ((long long)mt * TBM <= (long long)NT * BN) {
    const int g = (int)max(1ll, min((long long)mt, rows_fit / TBM));
    const int grp = local / (g * NT);
    const int gm = min(g, mt - grp * g);
    const int r = local - grp * g * NT;
    n = r / gm;
    m = grp * g + r % gm;
    return true;
  }
  const int g = (int)max(1ll, min((long long)NT, rows_fit / BN));
  const int grp = local / (g * mt);
  const int gn = min(g, NT - grp * g);
  const int r = local - grp * g * mt;
  m = r / gn;
  n = grp * g + r % gn;
  return false;
}

// The same decoding for one role's tiles, visited in increasing t (t, t + P, ...): the expert is
// found by scanning forward from the previous tile's (no binary search), and the L2 residency
// groups are sized once per launch, so the MMA issuer's step from one tile to the next is short.
template <int TBM>
struct TileCursor {
  const int* pref;
  int E, NT, fit_m, fit_n;  // m-tiles / n-tiles whose K-deep rows fit kResidentBytes
  int e;
  __device__ TileCursor(const int* pref_, int E_, int NT_, int K) : pref(pref_), E(E_), NT(NT_), e(0) {
    const long long rows_fit = kResidentBytes / ((long long)K * 2);
    fit_m = (int)max(1ll, min(rows_fit / TBM, 1ll << 30));
    fit_n = (int)max(1ll, min(rows_fit / BN, 1ll << 30));
  }
  // t -> (e, m, n) as decode_tile<TBM>; returns true when A is the resident operand.
  __device__ __forceinline__ bool next(int t, int& e_out, int& m, int& n) {
    const int j = t / NT;  // the tile's global m-tile
    while (e + 1 < E && pref[e + 1] <= j) ++e;
    e_out = e;
    const int local = t - pref[e] * NT;
    const int mt = pref[e + 1] - pref[e];
    if ((long long)mt * TBM <= (long long)NT * BN) {
      const int g = min(mt, fit_m);
      const int grp = local / (g * NT);
      const int gm = min(g, mt - grp * g);
      const int r = local - grp * g * NT;
      n = r / gm;
      m = grp * g + (r - n * gm);
      return true;
    }
    const int g = min(NT, fit_n);
    const int grp = local / (g * mt);
    const int gn = min(g, NT - grp * g);
    const int r = local - grp * g * mt;
    m = r / gn;
    n = grp * g + (r - m * gn);
    return false;
  }
};

struct TcParams {
  const int32_t* offsets;  // [E + 1] in global memory, or in shared memory when FUSED
  uint8_t* out;            // a [rows, N] (gate/up) or y [rows, N] (down), 16-bit elements
  unsigned* status;
  int E;
  int N;                   // valid output columns: I (gate/up) or H (down)
  int KB;                  // 64-deep K slices: ceil(H / 64) or ceil(I / 64)
  int NT;                  // n-tiles per expert: ceil(I / 128) or ceil(H / 256)
  int b_rows;              // rows of the B tensor per expert: I or H
  // Dataflow between two GEMMs of one launch (null when unused).  ready_signal: the epilogue
  // adds 1 per warp to ready_signal[global m-tile] once its rows of a tile are stored.
  // ready_wait: before the first A load of a tile the producer waits until
  // ready_wait[global m-tile] >= ready_target (0: the number of rows of that m-tile).  Global
  // m-tile = pref[e] + m.
  unsigned* ready_signal;
  const unsigned* ready_wait;
  unsigned ready_target;
  int signal_nt;  // > 0: ready_signal is per (m-tile, n-tile): index (pref[e] + m) * signal_nt + n
  // CTA-pair kernels of the expert backward: the FP32 da read by the SwiGLU-gradient epilogue,
  // its second output (a), and the intermediate size I
  const float* da;
  uint8_t* out1;
  int I;
  // CTA-pair kernels: tiles after each pair's first are claimed from this counter (zero at launch;
  // null: the static order pair, pair + P, ...)
  unsigned* tile_ctr;
};

__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Bounded wait until *cnt >= target (then the generic-proxy stores it counts are visible to TMA).
__device__ __forceinline__ bool wait_count(const unsigned* cnt, unsigned target,
                                           volatile int* abort_f, unsigned* status) {
  if (ld_acquire_gpu_u32(cnt) >= target) {
    fence_proxy_async_global();
    return true;
  }
  const long long t0 = clock64();
  while (ld_acquire_gpu_u32(cnt) < target) {
    if (*abort_f) return false;
    if (clock64() - t0 > kWaitLimit) {
      *abort_f = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
    __nanosleep(64);
  }
  fence_proxy_async_global();
  return true;
}

// offsets[e]: read-only path for a standalone launch, a plain load when FUSED (shared memory).
template <bool FUSED>
__device__ __forceinline__ int off_at(const int32_t* offsets, int e) {
  if constexpr (FUSED) return offsets[e];
  else return __ldg(offsets + e);
}

// Shared-memory ring and TMEM of one CTA.
struct Ring {
  uint32_t base;       // 1024-aligned start of the stages
  uint32_t bar0;       // first barrier
  uint32_t tmem_base;
  volatile int* abort_f;
  __device__ uint32_t full_bar(int s) const { return bar0 + 8u * s; }
  __device__ uint32_t empty_bar(int s) const { return bar0 + 8u * (STAGES + s); }
  __device__ uint32_t tfull_bar(int a) const { return bar0 + 8u * (2 * STAGES + a); }
  __device__ uint32_t tempty_bar(int a) const { return bar0 + 8u * (2 * STAGES + 2 + a); }
  __device__ uint32_t drain_bar() const { return bar0 + 8u * (2 * STAGES + 4); }
};

struct ProducerState {
  int stage = 0, armed = 0;
  uint32_t phase = 0;
};
struct MmaState {
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
};
struct EpilogueState {
  int acc = 0;
  uint32_t acc_phase = 0;
};

// Carves the ring out of dynamic shared memory; barrier i sits at 8 i after the stages, then the
// TMEM slot, the abort flag and, 16 bytes after the slot, room for kMaxExperts + 4 ints.
__device__ __forceinline__ Ring carve_ring(uint8_t* smem_raw, uint32_t** tmem_slot, int** pref) {
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + STAGES * STAGE_BYTES);
  *tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  *pref = reinterpret_cast<int*>(*tmem_slot + 4);
  Ring r;
  r.base = base;
  r.bar0 = smem_u32(bars);
  r.tmem_base = 0;
  r.abort_f = reinterpret_cast<volatile int*>(*tmem_slot + 1);
  return r;
}

// Thread 0: initialise the barriers and the abort flag.
__device__ __forceinline__ void init_ring(const Ring& r) {
  for (int s = 0; s < STAGES; ++s) {
    mbar_init(r.full_bar(s), 1);
    mbar_init(r.empty_bar(s), 1);
  }
  for (int a = 0; a < 2; ++a) {
    mbar_init(r.tfull_bar(a), 1);
    mbar_init(r.tempty_bar(a), 4);
  }
  mbar_init(r.drain_bar(), 1);
  *r.abort_f = 0;
  fence_mbar_init();
}

// ---------------------------------------------------------------- producer (one thread)
// All K slices of tile t.
template <bool GATEUP, bool FUSED>
__device__ __forceinline__ bool producer_tile(const CUtensorMap* mapA, const CUtensorMap* mapB0,
                                              const CUtensorMap* mapB1, const TcParams& p,
                                              const int* pref, const Ring& r, ProducerState& st,
                                              int t) {
  // The resident operand is marked evict_last.  The other one is NOT marked evict_first:
  // each of its tiles is still read by every CTA of the same m-row / n-column, shortly apart.
  const uint64_t keep = policy_evict_last(), other = policy_evict_normal();
  int e, m, n;
  const bool a_res = decode_tile(t, pref, p.E, p.NT, p.KB * BK, e, m, n);
  const uint64_t pa = a_res ? keep : other, pb = a_res ? other : keep;
  const int a_row = off_at<FUSED>(p.offsets, e) + m * BM;
  const int b_row = e * p.b_rows + n * (GATEUP ? BN / 2 : BN);
  for (int kb = 0; kb < p.KB; ++kb) {
    if (!wait_bounded(r.empty_bar(st.stage), st.phase ^ 1u, r.abort_f, p.status)) return false;
    const uint32_t sa = r.base + st.stage * STAGE_BYTES, sb = sa + A_BYTES;
    mbar_expect_tx(r.full_bar(st.stage), STAGE_BYTES);
    ++st.armed;
    if (GATEUP) {  // B first: it never waits for another tile
      tma_load_2d(sb, mapB0, r.full_bar(st.stage), kb * BK, b_row, pb);
      tma_load_2d(sb + B_BYTES / 2, mapB1, r.full_bar(st.stage), kb * BK, b_row, pb);
    } else {
      tma_load_2d(sb, mapB0, r.full_bar(st.stage), kb * BK, b_row, pb);
    }
    if (kb == 0 && p.ready_wait) {
      // ready_target 0: wait for one count per row of the m-tile
      const unsigned target =
          p.ready_target ? p.ready_target
                         : (unsigned)min(BM, off_at<FUSED>(p.offsets, e + 1) - a_row);
      if (!wait_count(p.ready_wait + pref[e] + m, target, r.abort_f, p.status)) return false;
    }
    tma_load_2d(sa, mapA, r.full_bar(st.stage), kb * BK, a_row, pa);
    if (++st.stage == STAGES) {
      st.stage = 0;
      st.phase ^= 1u;
    }
  }
  return true;
}

// Tiles blockIdx.x, blockIdx.x + gridDim.x, ... of the tile list.
template <bool GATEUP, bool FUSED>
__device__ __forceinline__ bool producer(const CUtensorMap* mapA, const CUtensorMap* mapB0,
                                         const CUtensorMap* mapB1, const TcParams& p,
                                         const int* pref, const Ring& r, ProducerState& st) {
  const int total = pref[p.E] * p.NT;
  for (int t = blockIdx.x; t < total; t += gridDim.x)
    if (!producer_tile<GATEUP, FUSED>(mapA, mapB0, mapB1, p, pref, r, st, t)) return false;
  return true;
}

// After an abort: let the copies still in flight land before the CTA exits.
__device__ __forceinline__ void producer_drain(const Ring& r, ProducerState& st) {
  for (int i = 0; i < min(st.armed, STAGES); ++i) {
    if (st.stage == 0) {
      st.stage = STAGES - 1;
      st.phase ^= 1u;
    } else {
      --st.stage;
    }
    wait_drain(r.full_bar(st.stage), st.phase);
  }
}

// ---------------------------------------------------------------- MMA issuer (one thread)
// One tile: all K slices into the next TMEM accumulator.
template <bool BF16>
__device__ __forceinline__ bool mma_tile(const TcParams& p, const Ring& r, MmaState& st) {
  constexpr uint32_t idesc = make_idesc(BF16, BM, BN);
  if (!wait_bounded(r.tempty_bar(st.acc), st.acc_phase ^ 1u, r.abort_f, p.status)) return false;
  tc_fence_after();
  const uint32_t d_tmem = r.tmem_base + (uint32_t)(st.acc * BN);
  for (int kb = 0; kb < p.KB; ++kb) {
    if (!wait_bounded(r.full_bar(st.stage), st.phase, r.abort_f, p.status)) return false;
    tc_fence_after();
    const uint32_t sa = r.base + st.stage * STAGE_BYTES, sb = sa + A_BYTES;
    const uint64_t da = make_sdesc(sa), db = make_sdesc(sb);
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk)  // advance 16 elements = 32 bytes along K
      umma_f16(d_tmem, da + 2u * kk, db + 2u * kk, idesc, (kb | kk) != 0);
    umma_commit(r.empty_bar(st.stage));
    if (++st.stage == STAGES) {
      st.stage = 0;
      st.phase ^= 1u;
    }
  }
  umma_commit(r.tfull_bar(st.acc));
  st.acc ^= 1;
  if (st.acc == 0) st.acc_phase ^= 1u;
  return true;
}

template <bool BF16>
__device__ __forceinline__ bool mma(const TcParams& p, const int* pref, const Ring& r,
                                    MmaState& st) {
  const int total = pref[p.E] * p.NT;
  for (int t = blockIdx.x; t < total; t += gridDim.x)
    if (!mma_tile<BF16>(p, r, st)) return false;
  return true;
}

// Wait until every MMA issued by this thread has completed (before TMEM is freed).
__device__ __forceinline__ void mma_drain(const Ring& r) {
  umma_commit(r.drain_bar());
  wait_drain(r.drain_bar(), 0);
}

// ---------------------------------------------------------------- epilogue (warps 2..5)
// One tile: this warp's 32 rows of the accumulator.
template <bool GATEUP, bool BF16, bool FUSED>
__device__ __forceinline__ bool epilogue_tile(const TcParams& p, const int* pref, const Ring& r,
                                              EpilogueState& st, int t, int warp, int lane) {
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  {
    int e, m, n;
    decode_tile(t, pref, p.E, p.NT, p.KB * BK, e, m, n);
    const bool ok = wait_bounded(r.tfull_bar(st.acc), st.acc_phase, r.abort_f, p.status);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    tc_fence_after();
    const int row = off_at<FUSED>(p.offsets, e) + m * BM + q * 32 + lane;
    const bool valid = row < off_at<FUSED>(p.offsets, e + 1);
    const uint32_t taddr = r.tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(st.acc * BN);
    uint8_t* orow = p.out + (size_t)row * p.N * 2;
    if (GATEUP) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t g[32], u[32];
        tmem_ld32(taddr + c * 32, g);
        tmem_ld32(taddr + BN / 2 + c * 32, u);
        tmem_wait_ld();
        const int col0 = n * (BN / 2) + c * 32;
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
    } else {
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t rr[32];
        tmem_ld32(taddr + c * 32, rr);
        tmem_wait_ld();
        const int col0 = n * BN + c * 32;
        if (valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            if (col0 + v * 8 < p.N) {
              uint32_t pk[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                pk[i] = pack2<BF16>(__uint_as_float(rr[v * 8 + i * 2]),
                                    __uint_as_float(rr[v * 8 + i * 2 + 1]));
              st_v4(orow + (size_t)(col0 + v * 8) * 2, make_uint4(pk[0], pk[1], pk[2], pk[3]));
            }
          }
        }
      }
    }
    tc_fence_before();
    if (p.ready_signal) fence_proxy_async_global();  // this lane's rows are read by TMA later
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(r.tempty_bar(st.acc));
      if (p.ready_signal) {
        __threadfence();
        const int gm = pref[e] + m;
        atomicAdd(p.ready_signal + (p.signal_nt > 0 ? gm * p.signal_nt + n : gm), 1u);
      }
    }
    st.acc ^= 1;
    if (st.acc == 0) st.acc_phase ^= 1u;
  }
  return true;
}

template <bool GATEUP, bool BF16, bool FUSED>
__device__ __forceinline__ bool epilogue(const TcParams& p, const int* pref, const Ring& r,
                                         EpilogueState& st, int warp, int lane) {
  const int total = pref[p.E] * p.NT;
  for (int t = blockIdx.x; t < total; t += gridDim.x)
    if (!epilogue_tile<GATEUP, BF16, FUSED>(p, pref, r, st, t, warp, lane)) return false;
  return true;
}

}  // namespace cta_gemm
}  // namespace moe
