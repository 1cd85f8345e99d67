// Expert backward on 5th-generation tensor cores for bf16 / f16 layers (ruDNN user guide, §12
// "MoE-Training erster Ordnung", cache.backward(dexpert)).  Per expert e and its dispatched rows:
//   DA    da  = dy down_e                       (FP32 [rows, I]; down_e read N-major)
//   GU    g, u = x gate_e^T, x up_e^T recomputed; epilogue with da:
//           s = sigmoid(g), dg = da u s (1 + g (1 - s)), du = da g s, a = g s u
//           -> dgdu [rows, 2I] (dg | du) and a [rows, I], both in the layer dtype
//   DIN   dinput = [dg du] [gate_e; up_e]       (layer dtype [rows, H]; K = 2I, B read N-major)
//   WG    dgate_e = dg^T x, dup_e = du^T x, ddown_e = dy^T a   (FP32; both operands M/N-major,
//         the contraction runs over the expert's rows)
// Persistent clusters of two CTAs (one per SM), the warp roles of the forward kernel (TMA
// producer, MMA issuer, four epilogue warps), 128 x 256 tiles, 4 x 48 KB stages, FP32
// accumulators in TMEM.  The two CTAs of a cluster take two tiles of the same expert that share
// an operand: two m-tiles of one n-tile, or, on an expert's odd last m-tile, two n-tiles of it.
// Each CTA loads all of its own operands (plain TMA loads into its own shared memory); the pair
// reads the shared operand at about the same time, so the second read is served by L2.  An
// operand whose contiguous dimension is M or N is loaded as 64-column boxes and described as an
// MN-major 128-byte-swizzled matrix (boxes 8 KB apart, 8-row groups 1 KB apart).  In WG the last
// 64-row K block of an expert would run into the next expert's rows: the MMA warp zeroes those
// rows in shared memory before the MMAs read them.  WG epilogue warps stage each 32 x 32 FP32
// chunk in shared memory (128-byte swizzle) and write it with a TMA tensor store through a
// [E][M][N] map, so every store moves whole 128-byte lines and never crosses into the next
// expert's slice.  All waits are bounded as in the forward.
#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tiles.cuh"

namespace moe {
namespace {
using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BOX_BYTES = 64 * 128;  // one 64-row x 64-column box
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxExperts = 1024;
constexpr int kChunkBytes = 32 * 32 * 4;             // one 32-row x 32-column FP32 store box
// Epilogue warps (a multiple of 4: each TMEM lane quarter is read by n/4 warps that split the
// columns) and ring stages per mode.  Eight WG epilogue warps with a 3-stage ring measured slower
// on GB300 than four warps with four stages, so every mode uses four and four.
template <int MODE> constexpr int n_epi_warps() { return 4; }
template <int MODE> constexpr int n_stages() { return 4; }
template <int MODE> constexpr int n_threads() { return 64 + 32 * n_epi_warps<MODE>(); }
// WG store buffers per epilogue warp.  Four (with a 3-stage ring to make room) measured slower
// than two with four stages.
constexpr int kStoreBufs = 2;
template <int MODE> constexpr int staging_bytes() { return MODE == 3 ? n_epi_warps<MODE>() * kStoreBufs * kChunkBytes : 0; }

enum Mode { DA = 0, GU = 1, DIN = 2, WG = 3 };

// WG: stages | store buffers | barriers.  Others: stages | barriers | m-tile prefix.
template <int MODE>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)n_stages<MODE>() * STAGE_BYTES + staging_bytes<MODE>() + 256 +
         (MODE == WG ? 0 : (kMaxExperts + 4) * sizeof(int));
}
static_assert(WG == 3, "n_epi_warps / n_stages key on the WG mode number");
static_assert(smem_bytes<WG>() <= 232448 && smem_bytes<DA>() <= 232448, "shared memory");

// MN-major 128-byte-swizzled operand: 64-column boxes BOX_BYTES apart, 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t make_sdesc_mn(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(BOX_BYTES >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16 instruction descriptor with operand majors (bit 15: A MN-major, bit 16: B MN-major)
__host__ __device__ constexpr uint32_t idesc_majors(bool bf16, int M, int N, bool a_mn, bool b_mn) {
  return make_idesc(bf16, M, N) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16);
}

struct BwdParams {
  const int32_t* offsets;
  int E, H, I;
  int KB;           // K blocks (DA: H/64, GU: H/64, DIN: 2I/64); WG: per expert
  int NT;           // n-tiles per expert
  int MP;           // WG: m-tile pairs per expert
  int M, N;         // WG: output matrix of each expert is M x N
  int a_col0;       // WG: first column of A inside its source matrix (du starts at I)
  int split;        // WG: rows of C below this go to the map `mapX`, the others (row - split)
                    // to `mapB1` (dgate | dup in one launch: split = I)
  const int* order; // WG: experts by descending row count (ties: lower id first)
  const float* da;  // GU: da [rows, I] FP32
  void* out0;       // DA: da FP32; GU: dgdu; DIN: dinput; WG: C [E, M, N] FP32
  void* out1;       // GU: a
  unsigned* status;
};

// Pair tile t -> expert e (rows r0 .. r1-1), this CTA's m-tile and n-tile, and which operand the
// pair shares.  WG: m-tiles 2 mp + rank of the expert's output share B.  Other modes: an expert
// with mt m-tiles has floor(mt / 2) * NT "m-pairs" (m-tiles 2 mp + rank, one n-tile, B shared)
// and, when mt is odd, ceil(NT / 2) "n-pairs" on its last m-tile (n-tiles 2 q + rank, A shared),
// so no pair computes a whole m-tile of rows that are not the expert's.  A tile past the
// expert's last m-tile or n-tile is computed on rows or columns of no interest and not stored.
template <int MODE>
__device__ __forceinline__ void decode(int t, const int* pref, const BwdParams& p, uint32_t rank,
                                       int& e, int& r0, int& r1, int& m, int& n) {
  if (MODE == WG) {  // t: position in the tile list of the experts sorted by rows
    const int per = p.MP * p.NT;
    const int sidx = t / per;
    e = __ldg(p.order + sidx);
    const int r = t - sidx * per;
    const int mp = r / p.NT;
    n = r - mp * p.NT;
    m = 2 * mp + (int)rank;
    r0 = __ldg(p.offsets + e);
    r1 = __ldg(p.offsets + e + 1);
  } else {
    e = find_expert(pref, p.E, t);
    r0 = __ldg(p.offsets + e);
    r1 = __ldg(p.offsets + e + 1);
    const int local = t - pref[e];
    const int mt = (r1 - r0 + BM - 1) / BM, full = (mt >> 1) * p.NT;
    if (local < full) {  // n inner: clusters in flight share the A tiles
      const int mp = local / p.NT;
      n = local - mp * p.NT;
      m = 2 * mp + (int)rank;
    } else {
      m = mt - 1;
      n = 2 * (local - full) + (int)rank;
    }
  }
}

// The j-th tile of pair `pair` (of P), or -1 when the pair has no more.  Other modes: tiles
// pair, pair + P, ... of the list.  WG: the list holds the experts' tiles in descending order of
// their rows, so its head is compute-bound (long contractions) and its tail store-bound (the FP32
// gradient of a short one, or zeros); each pair alternates between the two ends (pair q of the
// head, then pair q of the tail, ...), even pairs starting at the head and odd pairs at the tail,
// so at any time about half the pairs keep the tensor pipe busy while the others write.
template <int MODE>
__device__ __forceinline__ int tile_at(int j, int pair, int P, int N) {
  if (MODE != WG) {
    const long long t = pair + (long long)j * P;
    return t < N ? (int)t : -1;
  }
  const int Hh = (N + 1) / 2, Lh = N / 2;  // head positions [0, Hh), tail positions [Hh, N)
  const int nf = pair < Hh ? (Hh - pair + P - 1) / P : 0;
  const int nb = pair < Lh ? (Lh - pair + P - 1) / P : 0;
  const int both = min(nf, nb);
  bool head;
  int i;
  if (j < 2 * both) {
    head = ((j & 1) == 0) == ((pair & 1) == 0);
    i = j >> 1;
  } else {
    i = both + (j - 2 * both);
    head = nf > nb;
    if (i >= (head ? nf : nb)) return -1;
  }
  const int q = pair + i * P;
  return head ? q : N - 1 - q;
}

// Experts by descending row count, ties to the lower id (one block, E <= 1024): the order the WG
// tile list follows.  order[E] = the number of experts with rows (they come first).
__global__ void __launch_bounds__(1024) moe_expert_order(const int32_t* __restrict__ offsets, int E,
                                                         int* __restrict__ order) {
  __shared__ int n_active;
  if (threadIdx.x == 0) n_active = 0;
  __syncthreads();
  int mine = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) mine += offsets[i + 1] > offsets[i];
  if (mine) atomicAdd(&n_active, mine);
  __shared__ unsigned long long key[1024];
  int n = 1;
  while (n < E) n <<= 1;
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    key[i] = i < E ? ((unsigned long long)(uint32_t)(offsets[i + 1] - offsets[i]) << 32) |
                         (0xFFFFFFFFu - (uint32_t)i)
                   : 0ull;
  __syncthreads();
  for (int k = 2; k <= n; k <<= 1) {  // bitonic sort, descending
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ jj;
        if (ixj > i) {
          const unsigned long long a = key[i], b = key[ixj];
          if (((i & k) == 0) ? (a < b) : (a > b)) {
            key[i] = b;
            key[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    order[i] = (int)(0xFFFFFFFFu - (uint32_t)(key[i] & 0xFFFFFFFFull));
  if (threadIdx.x == 0) order[E] = n_active;
}

// The weight gradients of experts without rows are zero: written here with 16-byte streaming
// stores (evict-first in L2, so that the zeros do not push the GEMMs' operands out), instead of
// as GEMM tiles.  Every block walks the idle experts and stores its grid-stride share of their
// three matrices (dgate, dup, ddown) in batches of four stores a thread, so any grid size covers
// them.  With window_ns > 0 the fill runs beside GEMMs that take about that long and use part
// of HBM themselves: a burst of stores at the full write rate delays their operand loads by more
// than it saves, so each block pauses after every batch, long enough to spread its share over
// half the window (at most 2 us a batch; about 0.3 us of each batch goes to the stores).
__global__ void __launch_bounds__(256)
    moe_zero_idle_grads(const int32_t* __restrict__ offsets, int E, float* __restrict__ g0,
                        float* __restrict__ g1, float* __restrict__ g2, int64_t per_expert,
                        int64_t window_ns) {
  const int64_t n4 = per_expert / 4;  // per_expert = I * H, a multiple of 64
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  unsigned pause_ns = 0;
  if (window_ns > 0) {
    int idle = 0;
    for (int e = 0; e < E; ++e) idle += offsets[e + 1] > offsets[e] ? 0 : 1;
    const int64_t batches = ((int64_t)idle * 3 * n4 + 4 * stride - 1) / (4 * stride);
    if (batches > 0) {
      const int64_t p = window_ns / 2 / batches - 300;
      pause_ns = p <= 0 ? 0u : p >= 2000 ? 2000u : (unsigned)p;
    }
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int e = 0; e < E; ++e) {
    if (offsets[e + 1] > offsets[e]) continue;
#pragma unroll 1
    for (int m = 0; m < 3; ++m) {
      float4* v = reinterpret_cast<float4*>((m == 0 ? g0 : m == 1 ? g1 : g2) +
                                            (size_t)e * per_expert);
      for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += 4 * stride) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (i + u * stride < n4) __stcs(v + i + u * stride, z);
        if (pause_ns) __nanosleep(pause_ns);
      }
    }
  }
}

// The fill above, run beside the tensor-core GEMMs of steps 1-3 of the backward, which use about
// half of HBM's bandwidth: on a second stream of this device's context (created on first use),
// forked from the caller's stream before the first GEMM and joined back before the weight
// gradients, with one block per SM, so that every SM keeps room for a GEMM CTA next to it (the
// fill holds no shared memory and prefers the largest shared-memory carveout), paced over half
// the GEMMs' time.  While the caller's stream is being captured into a graph the fill runs on
// that stream itself, in order, at full width.
class IdleGradFill {
 public:
  IdleGradFill(cudaStream_t s) : s_(s) {}
  ~IdleGradFill() { join(); }
  // Before the first GEMM is enqueued: the fill depends on nothing enqueued after this.
  cudaError_t fork() {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s_, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
      return cudaSuccess;  // in order on s_
    cudaError_t err = side_stream(&s2_);
    if (err != cudaSuccess || !s2_) return err;
    if ((err = cudaEventCreateWithFlags(&fork_, cudaEventDisableTiming)) != cudaSuccess ||
        (err = cudaEventCreateWithFlags(&join_, cudaEventDisableTiming)) != cudaSuccess)
      return err;
    return cudaEventRecord(fork_, s_);
  }
  // After the first GEMM is enqueued, so that its CTAs are placed first.  window_ns: about how
  // long the GEMMs beside the fill take.
  cudaError_t launch(const int32_t* offsets, int E, float* g0, float* g1, float* g2,
                     int64_t per_expert, int sms, int64_t window_ns) {
    cudaError_t err = cudaFuncSetAttribute(moe_zero_idle_grads,
                                           cudaFuncAttributePreferredSharedMemoryCarveout,
                                           (int)cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    if (!fork_) {
      moe_zero_idle_grads<<<4 * sms, 256, 0, s_>>>(offsets, E, g0, g1, g2, per_expert, 0);
      return cudaGetLastError();
    }
    if ((err = cudaStreamWaitEvent(s2_, fork_, 0)) != cudaSuccess) return err;
    moe_zero_idle_grads<<<sms, 256, 0, s2_>>>(offsets, E, g0, g1, g2, per_expert, window_ns);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    err = cudaEventRecord(join_, s2_);
    if (err == cudaSuccess) recorded_ = true;
    return err;
  }
  // The caller's stream waits for the fill (also on every early return, through the destructor).
  cudaError_t join() {
    cudaError_t err = cudaSuccess;
    if (recorded_) err = cudaStreamWaitEvent(s_, join_, 0);
    recorded_ = false;
    if (fork_) cudaEventDestroy(fork_);
    if (join_) cudaEventDestroy(join_);
    fork_ = join_ = nullptr;
    return err;
  }

 private:
  // The second stream of the current device and context (null, and the fill in order, when
  // the context cannot be identified).
  static cudaError_t side_stream(cudaStream_t* out) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static cudaStream_t st[kMaxDevices] = {};
    static unsigned long long ctx_of[kMaxDevices] = {};
    *out = nullptr;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (ctx == 0) return cudaSuccess;
    if (!st[dev] || ctx != ctx_of[dev]) {  // a new context: the old stream went with the old one
      cudaStream_t s2 = nullptr;
      if ((err = cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking)) != cudaSuccess) return err;
      st[dev] = s2;
      ctx_of[dev] = ctx;
    }
    *out = st[dev];
    return cudaSuccess;
  }
  cudaStream_t s_, s2_ = nullptr;
  cudaEvent_t fork_ = nullptr, join_ = nullptr;
  bool recorded_ = false;
};

// Pair tiles of an expert with n rows (modes other than WG).
struct PairTiles {
  int NT;
  __device__ int operator()(int n) const {
    const int mt = (n + BM - 1) / BM;
    return (mt >> 1) * NT + (mt & 1) * ((NT + 1) >> 1);
  }
};

template <int MODE, bool BF16>
__global__ void __launch_bounds__(n_threads<MODE>(), 1)
    moe_experts_bwd_tc(const __grid_constant__ CUtensorMap mapA,
                       const __grid_constant__ CUtensorMap mapB0,
                       const __grid_constant__ CUtensorMap mapB1,
                       const __grid_constant__ CUtensorMap mapX, const BwdParams p) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int NST = n_stages<MODE>();
  constexpr bool A_MN = MODE == WG, B_MN = MODE != GU;
  extern __shared__ uint8_t tcb_smem_raw[];
  const uint32_t raw = smem_u32(tcb_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = tcb_smem_raw + (base - raw);
  const uint32_t staging = base + NST * STAGE_BYTES;  // WG store buffers (1 KB aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + NST * STAGE_BYTES + staging_bytes<MODE>());
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (NST + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * NST + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * NST + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * NST + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * NST + 5);
  volatile int* abort_f = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* pref = reinterpret_cast<int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = (int)cluster_id_x(), npairs = (int)ncluster_x();
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);  // this CTA's MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), n_epi_warps<MODE>());
    }
    mbar_init(drain_bar, 1);
    *abort_f = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  if (warp == 2 && MODE != WG) build_expert_prefix(p.offsets, p.E, PairTiles{p.NT}, pref, lane);
  if (warp == 0 && lane == 0) {
    tma_prefetch(&mapA);
    tma_prefetch(&mapB0);
    tma_prefetch(&mapB1);
    if (MODE == WG) tma_prefetch(&mapX);
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs started (the tile list is split by cluster rank)
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // WG: the experts with rows only (order[E] of them, first in the order); the others' gradients
  // are zeroed by moe_zero_idle_grads
  const int total = MODE == WG ? __ldg(p.order + p.E) * p.MP * p.NT : pref[p.E];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0, armed = 0;
      uint32_t phase = 0;
      bool stop = false;
      const uint64_t pol = policy_evict_normal();
      for (int j = 0; !stop; ++j) {
        const int t = tile_at<MODE>(j, pair, npairs, total);
        if (t < 0) break;
        int e, r0, r1, m, n;
        decode<MODE>(t, pref, p, rank, e, r0, r1, m, n);
        const int KB = MODE == WG ? (r1 - r0 + BK - 1) / BK : p.KB;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_f, p.status)) {
            stop = true;
            break;
          }
          const uint32_t sa = base + stage * STAGE_BYTES, sb = sa + A_BYTES;
          mbar_expect_tx(full_bar(stage), STAGE_BYTES);
          if (MODE == WG) {  // A: rows r0 + 64 kb, columns a_col0 + 128 m (two 64-column boxes)
            const int y = r0 + kb * BK;
            for (int j = 0; j < 2; ++j)
              tma_load_2d(sa + j * BOX_BYTES, &mapA, full_bar(stage), p.a_col0 + m * BM + 64 * j, y, pol);
            for (int j = 0; j < 4; ++j)  // B: columns n * BN .. + 255 (four 64-column boxes)
              tma_load_2d(sb + j * BOX_BYTES, &mapB0, full_bar(stage), n * BN + 64 * j, y, pol);
          } else {
            tma_load_2d(sa, &mapA, full_bar(stage), kb * BK, r0 + m * BM, pol);
            if (MODE == GU) {  // K-major: 128 gate rows then the same 128 up rows
              const int br = e * p.I + n * (BN / 2);
              tma_load_2d(sb, &mapB0, full_bar(stage), kb * BK, br, pol);
              tma_load_2d(sb + B_BYTES / 2, &mapB1, full_bar(stage), kb * BK, br, pol);
            } else {
              // N-major B: rows are K.  DA: down [E*H, I];  DIN: gate (k < I) / up (k >= I)
              const CUtensorMap* mb = &mapB0;
              int kr;
              if (MODE == DA) {
                kr = e * p.H + kb * BK;
              } else {
                const int k0 = kb * BK;
                if (k0 >= p.I) mb = &mapB1;
                kr = e * p.I + (k0 >= p.I ? k0 - p.I : k0);
              }
              for (int j = 0; j < 4; ++j)
                tma_load_2d(sb + j * BOX_BYTES, mb, full_bar(stage), n * BN + 64 * j, kr, pol);
            }
          }
          ++armed;
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_f) {
        for (int i = 0; i < min(armed, NST); ++i) {
          if (stage == 0) {
            stage = NST - 1;
            phase ^= 1u;
          } else {
            --stage;
          }
          wait_drain(full_bar(stage), phase);
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA warp (lane 0 issues)
    constexpr uint32_t idesc = idesc_majors(BF16, BM, BN, A_MN, B_MN);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool stop = false;
    for (int j = 0; !stop; ++j) {
      const int t = tile_at<MODE>(j, pair, npairs, total);
      if (t < 0) break;
      int e, r0, r1, m, n;
      decode<MODE>(t, pref, p, rank, e, r0, r1, m, n);
      const int KB = MODE == WG ? (r1 - r0 + BK - 1) / BK : p.KB;
      bool ok = lane != 0 || wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_f, p.status);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < KB; ++kb) {
        ok = wait_bounded(full_bar(stage), phase, abort_f, p.status);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          stop = true;
          break;
        }
        const uint32_t sa = base + stage * STAGE_BYTES, sb = sa + A_BYTES;
        int nkk = BK / 16;  // K = 16 steps of this stage that hold the expert's rows
        if (MODE == WG) {
          const int valid = r1 - (r0 + kb * BK);
          if (valid < BK) {
            // the last stage of an expert: only ceil(valid / 16) K steps are issued, and the rows
            // between the expert's end and that step's end (they belong to the next expert) are
            // zeroed in both operands
            nkk = (valid + 15) / 16;
            const int nz = (nkk * 16 - valid) * 6 * 8;  // rows x (2 A + 4 B boxes) x 8 chunks
            uint8_t* g0 = gbase + stage * STAGE_BYTES;
            for (int i = lane; i < nz; i += 32) {
              const int row = valid + i / 48, rem = i % 48, box = rem / 8, ch = rem % 8;
              uint8_t* dst = g0 + (box < 2 ? box * BOX_BYTES : A_BYTES + (box - 2) * BOX_BYTES) +
                             row * 128 + ch * 16;
              *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
          }
        }
        if (lane == 0) {
          tc_fence_after();
          const uint64_t da = A_MN ? make_sdesc_mn(sa) : make_sdesc(sa);
          const uint64_t db = B_MN ? make_sdesc_mn(sb) : make_sdesc(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // 16 K: 32 bytes (K-major) or 2 KB (MN-major)
            if (kk < nkk)
              umma_f16(d_tmem, da + (A_MN ? 128u : 2u) * kk, db + (B_MN ? 128u : 2u) * kk, idesc,
                       (kb | kk) != 0);
          umma_commit(empty_bar(stage));  // frees the stage once its MMAs complete
        }
        __syncwarp();
        if (++stage == NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (stop) break;
      if (lane == 0) umma_commit(tfull_bar(acc));
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) {
      umma_commit(drain_bar);
      wait_drain(drain_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0, slot = 0;
    uint32_t acc_phase = 0;
    for (int j = 0;; ++j) {
      const int t = tile_at<MODE>(j, pair, npairs, total);
      if (t < 0) break;
      int e, r0, r1, m, n;
      decode<MODE>(t, pref, p, rank, e, r0, r1, m, n);
      const bool ok = wait_bounded(tfull_bar(acc), acc_phase, abort_f, p.status);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (MODE == WG) {
        // rows m*BM + q*32 .. +31 of C_e; chunk c covers columns n*BN + 32c .. +31
        const int row0 = m * BM + q * 32;
        const bool empty = r1 == r0;  // no rows: the gradient is zero
        if (row0 < p.M) {
#pragma unroll 1
          // warps 2-5 take column chunks 0-3, warps 6-9 chunks 4-7 (WG has eight epilogue warps)
          constexpr int kCpw = 8 / (n_epi_warps<MODE>() / 4);
          const int c0 = ((warp - 2) >> 2) * kCpw;
          for (int c = c0; c < c0 + kCpw; ++c) {
            const int col0 = n * BN + c * 32;
            if (col0 >= p.N) break;
            uint32_t r[32];
            tmem_ld32(taddr + c * 32, r);
            tmem_wait_ld();
            const uint32_t buf =
                staging + (uint32_t)(((warp - 2) * kStoreBufs + slot) * kChunkBytes);
            if (lane == 0) bulk_wait_read<kStoreBufs - 1>();  // the store that last read `buf` is done
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // 16-byte chunk j of this lane's row, 128-byte swizzle
              const uint32_t dst = buf + lane * 128 + ((j ^ (lane & 7)) << 4);
              if (empty)
                st_shared_v4(dst, 0u, 0u, 0u, 0u);
              else
                st_shared_v4(dst, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (row0 < p.split)  // a 32-row chunk never straddles split (a multiple of 64)
                tma_store_3d(&mapX, buf, col0, row0, e);
              else
                tma_store_3d(&mapB1, buf, col0, row0 - p.split, e);
              bulk_commit();
            }
            slot = slot + 1 == kStoreBufs ? 0 : slot + 1;
          }
        }
      } else {
        const int row = r0 + m * BM + q * 32 + lane;
        const bool valid = row < r1;
        if (MODE == GU) {
          const float* darow = p.da + (size_t)row * p.I;
          T* dg_row = reinterpret_cast<T*>(p.out0) + (size_t)row * 2 * p.I;
          T* a_row = reinterpret_cast<T*>(p.out1) + (size_t)row * p.I;
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
                if (col0 + v * 8 < p.I) {
                  float dv[8];
                  *reinterpret_cast<float4*>(dv) = *reinterpret_cast<const float4*>(darow + col0 + v * 8);
                  *reinterpret_cast<float4*>(dv + 4) = *reinterpret_cast<const float4*>(darow + col0 + v * 8 + 4);
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
                  st_v4(dg_row + col0 + v * 8, make_uint4(pg[0], pg[1], pg[2], pg[3]));
                  st_v4(dg_row + p.I + col0 + v * 8, make_uint4(pu[0], pu[1], pu[2], pu[3]));
                  st_v4(a_row + col0 + v * 8, make_uint4(pa[0], pa[1], pa[2], pa[3]));
                }
              }
            }
          }
        } else {  // DA (FP32 out, N = I) or DIN (layer dtype out, N = H)
          const int Nout = MODE == DA ? p.I : p.H;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r[32];
            tmem_ld32(taddr + c * 32, r);
            tmem_wait_ld();
            const int col0 = n * BN + c * 32;
            if (valid) {
              if (MODE == DA) {
                float* o = reinterpret_cast<float*>(p.out0) + (size_t)row * Nout;
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  if (col0 + v * 4 < Nout)
                    st_v4(o + col0 + v * 4, make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]));
              } else {
                T* o = reinterpret_cast<T*>(p.out0) + (size_t)row * Nout;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                  if (col0 + v * 8 < Nout) {
                    uint32_t pk[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                      pk[i] = pack2<BF16>(__uint_as_float(r[v * 8 + i * 2]),
                                          __uint_as_float(r[v * 8 + i * 2 + 1]));
                    st_v4(o + col0 + v * 8, make_uint4(pk[0], pk[1], pk[2], pk[3]));
                  }
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (MODE == WG && lane == 0) bulk_wait_all();  // stores done before shared memory goes away
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Launches clusters of two CTAs, at most as many as can be resident at once (queried once per
// device and mode); `upper_pairs` bounds the number of pair tiles.  `c` is the TMA store map of
// the weight gradient (WG; other modes do not read it).
template <int MODE, bool BF16>
cudaError_t launch_mode(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                        const CUtensorMap& c, const BwdParams& p, int64_t upper_pairs, int dev,
                        cudaStream_t s) {
  auto kern = moe_experts_bwd_tc<MODE, BF16>;
  constexpr size_t smem = smem_bytes<MODE>();
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(n_threads<MODE>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2);
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
  const int pairs = (int)(upper_pairs < mp ? upper_pairs : mp);
  if (pairs < 1) return cudaSuccess;
  cfg.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&cfg, kern, a, b0, b1, c, p);
}

template <bool BF16>
cudaError_t bwd_tc_t(const void* x_d, const int32_t* offsets, int64_t rows, const void* gate,
                     const void* up, const void* down, int E, int H, int I, const void* dy,
                     void* dinput, float* dgate, float* dup, float* ddown, void* scratch,
                     unsigned* status, cudaStream_t s) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  // scratch: da FP32 [rows, I] | dgdu [rows, 2I] | a [rows, I] (layer dtype)
  float* da = (float*)scratch;
  uint8_t* dgdu = (uint8_t*)scratch + align_up((size_t)rows * I * 4, 256);
  uint8_t* abuf = dgdu + align_up((size_t)rows * 2 * I * 2, 256);
  int* order = (int*)(abuf + align_up((size_t)rows * I * 2, 256));  // [E + 1] for the WG tile order
  const int64_t mt_upper = (rows + BM - 1) / BM + E;  // >= m-tiles; pair tiles <= mt * ceil(NT/2)
  CUtensorMap mA, mB0, mB1;
  BwdParams p{};
  p.offsets = offsets;
  p.E = E;
  p.H = H;
  p.I = I;
  p.status = status;

  int sms = 0;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return err;
  // the zero gradients of experts without rows, beside steps 1-3
  IdleGradFill fill(s);
  if ((err = fill.fork()) != cudaSuccess) return err;

  // 1-3 on CTA pairs (256-row tiles) when the experts average at least 128 rows, as the forward
  if (rows >= (int64_t)128 * E) {
    err = launch_experts_bwd_pair(x_d, offsets, rows, gate, up, down, BF16 ? MOE_BF16 : MOE_F16, E,
                                  H, I, dy, da, dgdu, abuf, dinput, status, s);
    if (err != cudaSuccess) return err;
  } else {
  // 1. da = dy down_e
  if (!make_map_2d(&mA, dy, BF16, H, rows, BK, BM) ||
      !make_map_2d(&mB0, down, BF16, I, (int64_t)E * H, 64, 64))
    return cudaErrorInvalidValue;
  p.KB = (H + BK - 1) / BK;
  p.NT = (I + BN - 1) / BN;
  p.out0 = da;
  err = launch_mode<DA, BF16>(mA, mB0, mB0, mA, p, mt_upper * ((p.NT + 1) / 2), dev, s);
  if (err != cudaSuccess) return err;

  // 2. g, u recomputed; epilogue -> dg | du, a
  if (!make_map_2d(&mA, x_d, BF16, H, rows, BK, BM) ||
      !make_map_2d(&mB0, gate, BF16, H, (int64_t)E * I, BK, BN / 2) ||
      !make_map_2d(&mB1, up, BF16, H, (int64_t)E * I, BK, BN / 2))
    return cudaErrorInvalidValue;
  p.KB = (H + BK - 1) / BK;
  p.NT = (I + BN / 2 - 1) / (BN / 2);
  p.da = da;
  p.out0 = dgdu;
  p.out1 = abuf;
  err = launch_mode<GU, BF16>(mA, mB0, mB1, mA, p, mt_upper * ((p.NT + 1) / 2), dev, s);
  if (err != cudaSuccess) return err;

  // 3. dinput = [dg du] [gate_e; up_e]
  if (!make_map_2d(&mA, dgdu, BF16, 2 * (int64_t)I, rows, BK, BM) ||
      !make_map_2d(&mB0, gate, BF16, H, (int64_t)E * I, 64, 64) ||
      !make_map_2d(&mB1, up, BF16, H, (int64_t)E * I, 64, 64))
    return cudaErrorInvalidValue;
  p.KB = 2 * I / BK;
  p.NT = (H + BN - 1) / BN;
  p.out0 = dinput;
  err = launch_mode<DIN, BF16>(mA, mB0, mB1, mA, p, mt_upper * ((p.NT + 1) / 2), dev, s);
  if (err != cudaSuccess) return err;
  }
  // steps 1-3: 10 R H I FLOPs, at about 1.4 PFLOP/s on the skewed layer's shapes
  const int64_t window_ns = (int64_t)(10.0 * (double)rows * H * I / 1.4e6);
  if ((err = fill.launch(offsets, E, dgate, dup, ddown, (int64_t)I * H, sms, window_ns)) !=
          cudaSuccess ||
      (err = fill.join()) != cudaSuccess)
    return err;

  // 4. weight gradients of the experts with rows, contracted over each expert's rows, experts
  // ordered by row count
  moe_expert_order<<<1, 1024, 0, s>>>(offsets, E, order);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  p.order = order;
  // dgate and dup in one launch: [dg du]^T x_d is a [2I, H] matrix per expert, whose rows below
  // I are dgate's and the others dup's
  CUtensorMap mX, mC, mC2;
  if (!make_map_2d(&mA, dgdu, BF16, 2 * (int64_t)I, rows, 64, 64) ||
      !make_map_2d(&mX, x_d, BF16, H, rows, 64, 64) ||
      !make_map_3d_f32(&mC, dgate, H, I, E, 32, 32) || !make_map_3d_f32(&mC2, dup, H, I, E, 32, 32))
    return cudaErrorInvalidValue;
  p.M = 2 * I;
  p.split = I;
  p.N = H;
  p.MP = (2 * I + 2 * BM - 1) / (2 * BM);
  p.NT = (H + BN - 1) / BN;
  p.out0 = dgate;
  p.a_col0 = 0;
  err = launch_mode<WG, BF16>(mA, mX, mC2, mC, p, (int64_t)E * p.MP * p.NT, dev, s);
  if (err != cudaSuccess) return err;
  CUtensorMap mY, mAct;
  if (!make_map_2d(&mY, dy, BF16, H, rows, 64, 64) ||
      !make_map_2d(&mAct, abuf, BF16, I, rows, 64, 64) ||
      !make_map_3d_f32(&mC, ddown, I, H, E, 32, 32))
    return cudaErrorInvalidValue;
  p.M = H;
  p.split = H;
  p.N = I;
  p.MP = (H + 2 * BM - 1) / (2 * BM);
  p.NT = (I + BN - 1) / BN;
  p.out0 = ddown;
  p.a_col0 = 0;
  return launch_mode<WG, BF16>(mY, mAct, mAct, mC, p, (int64_t)E * p.MP * p.NT, dev, s);
}

}  // namespace

size_t experts_backward_tc_scratch_bytes(int64_t rows, int64_t I) {
  return align_up((size_t)rows * I * 4, 256) + align_up((size_t)rows * 2 * I * 2, 256) +
         align_up((size_t)rows * I * 2, 256) + (1024 + 1) * sizeof(int);
}

cudaError_t launch_experts_backward_tc(const void* x_d, const int32_t* offsets, int64_t rows,
                                       const void* gate, const void* up, const void* down,
                                       int wdt, int E, int H, int I, const void* dy, void* dinput,
                                       float* dgate, float* dup, float* ddown, void* scratch,
                                       unsigned* status, cudaStream_t s) {
  if (wdt == MOE_BF16)
    return bwd_tc_t<true>(x_d, offsets, rows, gate, up, down, E, H, I, dy, dinput, dgate, dup,
                          ddown, scratch, status, s);
  if (wdt == MOE_F16)
    return bwd_tc_t<false>(x_d, offsets, rows, gate, up, down, E, H, I, dy, dinput, dgate, dup,
                           ddown, scratch, status, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
