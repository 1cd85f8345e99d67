// Group-limited sigmoid routing: route_sigmoid_grouped of the ruDNN user guide, §10
// "Gruppenbeschränktes Sigmoid-MoE-Routing".
//
// s = sigmoid(logit); c = s + bias (bias optional, FP32, selection only).  Experts form `groups`
// contiguous groups of gs = E / groups; a group scores its largest c, or the sum of its two largest
// with group_top_two.  The `selected_groups` best groups (ties: lower group id) are kept, then the
// top_k experts inside them by c (ties: lower id), slots in that order.  Weights are s of the
// chosen experts, divided by their sum when renormalising, times scale, rounded to the logits
// dtype.  Rows whose corrected scores hold a NaN get NaN weights and ids 0..k-1.
//
// The selection (sigmoid, correction, group scores, ranking) is the decision float64 arithmetic
// makes, as in the float64 reference.  One warp owns a row: lane i holds experts i, i + 32, ...;
// the group and expert choices are rounds of warp argmax over (score, -id) pairs.  Each row is
// first decided in FP32 (accurate expf, IEEE division): with the FP32 error of every corrected
// score bounded by E_c = 5e-7 + 1.2e-7 max|c| (expf within 2 ulp, the division and the additions
// rounded once each), the FP32 choice is the float64 choice whenever every margin it rests on --
// last chosen group vs the best other group, each chosen expert vs the next one, the k-th vs the
// best unchosen candidate -- exceeds twice the bound on the two scores compared.  Those rows take
// their k weights from float64 sigmoids of the chosen experts; every other row (a near or exact
// tie, a NaN or infinite score) is decided again entirely in float64.  Either way the indices
// and weights are the float64 path's.
//
// Rows of E = L * EPL experts (E a power of two up to 512, EPL = 8 or 16, groups of whole lanes,
// k <= L, 16-byte aligned rows) take a faster form of the same FP32 attempt, with a row held by L
// consecutive lanes instead of a warp: lane l owns experts l EPL .. l EPL + EPL - 1 (16-byte
// loads), a group's top-two is merged across its gs / EPL lanes by shuffles, and the G group
// scores are ranked by G shuffles.  The top_k experts of the chosen groups come from the few
// candidates near the k-th score, compacted into shared memory and ranked by counting (see
// sigmoid_row_sub).  Where a margin fails, float64 scores are computed only where they can change
// the answer: for the groups in the run of close group scores across the boundary, and for the
// run of close candidates that reaches the k-th (a row whose close run outgrows the sub-warp
// takes the float64 decision of the whole selection).  Rows with a non-finite score are handed
// to the warp-wide routine by the whole warp.
#include "common.cuh"
#include "launch.h"
#include "route_sigmoid_core.cuh"

namespace moe {
namespace {

constexpr int kSigWarps = 4;

template <typename T, int C>
__global__ void __launch_bounds__(kSigWarps * 32)
    moe_route_sigmoid_kernel(const T* __restrict__ logits, const float* __restrict__ bias,
                             int64_t T_, int E, int k, int G, int SG, int top_two, int renorm,
                             float scale, uint32_t* __restrict__ idx_out, T* __restrict__ w_out) {
  extern __shared__ double sig_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * kSigWarps + warp;
  if (row >= T_) return;  // whole warp leaves together
  sigmoid_route_row<T, C>(logits + row * (int64_t)E, bias, row, E, k, G, SG, top_two, renorm,
                          scale, sig_smem + (size_t)warp * (E + 128 + 64 + 32), lane, idx_out,
                          w_out);
}

// Order-preserving map of a double to 64 bits (larger double -> larger key; -0 below +0 does not
// matter: equal scores compare equal through their values before the keys are formed).
__device__ __forceinline__ unsigned long long dkey(double d) {
  const unsigned long long u = (unsigned long long)__double_as_longlong(d);
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double dkey_value(unsigned long long k) {
  return __longlong_as_double((long long)((k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k));
}
__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned mask, unsigned long long v,
                                                            int o, int w) {
  const unsigned lo = __shfl_xor_sync(mask, (unsigned)v, o, w);
  const unsigned hi = __shfl_xor_sync(mask, (unsigned)(v >> 32), o, w);
  return ((unsigned long long)hi << 32) | lo;
}
__device__ __forceinline__ unsigned long long shfl_u64(unsigned mask, unsigned long long v, int src,
                                                       int w) {
  const unsigned lo = __shfl_sync(mask, (unsigned)v, src, w);
  const unsigned hi = __shfl_sync(mask, (unsigned)(v >> 32), src, w);
  return ((unsigned long long)hi << 32) | lo;
}
// The logits and corrections of experts e0 .. e0 + EPL - 1 (16-byte loads; 16-byte aligned).
template <typename T, int EPL>
__device__ __forceinline__ void sub_load(const T* __restrict__ src, const float* __restrict__ bias,
                                         int e0, float* x, float* b) {
  constexpr int PER = 16 / (int)sizeof(T);  // elements per 16-byte load
#pragma unroll
  for (int v = 0; v < EPL / PER; ++v) {
    Vec16<T> q;
    q.u = ld_nc_v4(src + e0 + v * PER);
    q.to_float(x + v * PER);
  }
#pragma unroll
  for (int v = 0; v < EPL / 4; ++v) {
    const float4 q = bias ? __ldg(reinterpret_cast<const float4*>(bias + e0) + v)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    b[4 * v] = q.x;
    b[4 * v + 1] = q.y;
    b[4 * v + 2] = q.z;
    b[4 * v + 3] = q.w;
  }
}
// 64-bit key of a finite FP32 score and its expert: a larger score gives a larger key, and equal
// scores (-0 and +0 included) prefer the lower id.
__device__ __forceinline__ unsigned long long skey(float v, int id) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  const uint32_t m = (u >> 31) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)m << 32) | (0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ float skey_score(unsigned long long key) {
  const uint32_t m = (uint32_t)(key >> 32);
  return __uint_as_float((m >> 31) ? (m & 0x7FFFFFFFu) : ~m);
}
__device__ __forceinline__ int skey_id(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)key);
}

// float64 score of an expert, as the float64 decision computes it
__device__ __forceinline__ double sig_score64(float x, float b) {
  return 1.0 / (1.0 + exp(-(double)x)) + (double)b;
}

// The float64 decision of a row whose FP32 attempt could not prove its choice, computing float64
// scores only where they can change it: every score is within ec of its FP32 value, so an expert
// below its group's FP32 second-best (best, without top_two) by more than 2 ec cannot be in the
// group's float64 top two, and a candidate below the FP32 (k+1)-th best candidate of the chosen
// groups by more than 2 ec cannot be in the float64 top k.  Group scores and the ranking use
// float64 values compared as 64-bit keys (ties: lower group id, lower expert id).  Out of line:
// rows get here rarely.
template <typename T, int L, int EPL>
__device__ __noinline__ void sigmoid_row_sub_f64(const T* __restrict__ src,
                                                    const float* __restrict__ bias, const float* c,
                                                    float ec, float t2f, int64_t row, int k, int G,
                                                    int SG, int top_two, int renorm, float scale,
                                                    int sl, unsigned mask, int sub0,
                                                    uint32_t* __restrict__ idx_out,
                                                    T* __restrict__ w_out) {
  constexpr int E = L * EPL;
  const int gs = E / G, lpg = gs / EPL;
  float x[EPL], b[EPL];
  sub_load<T, EPL>(src, bias, sl * EPL, x, b);
  // float64 scores of the experts a group's top two may contain
  unsigned long long key[EPL];
  unsigned have = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) key[j] = 0ull;
  unsigned need = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) need |= (c[j] >= t2f - 2.f * ec ? 1u : 0u) << j;
  auto fill = [&](unsigned want) {  // float64 keys of the experts in `want` not computed yet
    want &= ~have;
    while (__any_sync(mask, want != 0)) {
      const int j = want ? __ffs(want) - 1 : -1;
      float xj = 0.f, bj = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        xj = (i == j) ? x[i] : xj;
        bj = (i == j) ? b[i] : bj;
      }
      const unsigned long long kj = j >= 0 ? dkey(sig_score64(xj, bj)) : 0ull;
#pragma unroll
      for (int i = 0; i < EPL; ++i) key[i] = (i == j) ? kj : key[i];
      if (j >= 0) {
        want &= want - 1;
        have |= 1u << j;
      }
    }
  };
  fill(need);
  // the group's float64 top two (duplicates count), merged over its lanes
  unsigned long long k1 = 0, k2 = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    if (!((need >> j) & 1u)) continue;
    if (key[j] > k1) {
      k2 = k1;
      k1 = key[j];
    } else if (key[j] > k2) {
      k2 = key[j];
    }
  }
  for (int o = 1; o < lpg; o <<= 1) {
    const unsigned long long o1 = shfl_xor_u64(mask, k1, o, L), o2 = shfl_xor_u64(mask, k2, o, L);
    const unsigned long long n1 = k1 > o1 ? k1 : o1;
    const unsigned long long lo = k1 > o1 ? o1 : k1, hi2 = k2 > o2 ? k2 : o2;
    k2 = lo > hi2 ? lo : hi2;
    k1 = n1;
  }
  const double gsc = top_two ? dkey_value(k1) + dkey_value(k2) : dkey_value(k1);
  const unsigned long long gk = shfl_u64(mask, dkey(gsc), (sl < G ? sl : 0) * lpg, L);
  int rank = 0;
  for (int g = 0; g < G; ++g) {
    const unsigned long long o = shfl_u64(mask, gk, g, L);
    rank += (o > gk) || (o == gk && g < sl);
  }
  const unsigned chosen = (__ballot_sync(mask, sl < G && rank < SG) >> sub0);
  const bool mine = (chosen >> (sl / lpg)) & 1u;
  // the FP32 (k+1)-th best candidate bounds the experts the float64 top k may contain
  const int cand = SG * gs;
  unsigned cmask = mine ? (1u << EPL) - 1u : 0u;
  float vk1 = -INFINITY;
  if (cand > k) {
    unsigned avail = cmask;
    for (int r = 0; r <= k; ++r) {
      float bv = -INFINITY;
      int bj = -1;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (((avail >> j) & 1u) && (bj < 0 || c[j] > bv)) {
          bv = c[j];
          bj = j;
        }
      float m = bv;
#pragma unroll
      for (int o = 1; o < L; o <<= 1) m = fmaxf(m, __shfl_xor_sync(mask, m, o, L));
      const int wl = __ffs((__ballot_sync(mask, bj >= 0 && bv == m) >> sub0)) - 1;
      const int wj = __shfl_sync(mask, bj, wl, L);
      if (sl == wl) avail &= ~(1u << wj);
      vk1 = m;
    }
  }
  unsigned rel = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) rel |= (((cmask >> j) & 1u) && c[j] >= vk1 - 2.f * ec ? 1u : 0u) << j;
  fill(rel);
  // the top k of the relevant candidates by float64 score, ties to the lower id
  float my_x = 0.f;
  int my_id = -1;
  for (int r = 0; r < k; ++r) {
    unsigned long long bk = 0;
    int bj = -1;
#pragma unroll
    for (int j = 0; j < EPL; ++j)
      if (((rel >> j) & 1u) && (bj < 0 || key[j] > bk)) {
        bk = key[j];
        bj = j;
      }
    unsigned long long mk = bk;
#pragma unroll
    for (int o = 1; o < L; o <<= 1) {
      const unsigned long long ok = shfl_xor_u64(mask, mk, o, L);
      mk = ok > mk ? ok : mk;
    }
    const int wl = __ffs((__ballot_sync(mask, bj >= 0 && bk == mk) >> sub0)) - 1;
    const int wj = __shfl_sync(mask, bj, wl, L);
    float wx = 0.f;
#pragma unroll
    for (int j = 0; j < EPL; ++j) wx = (j == wj) ? x[j] : wx;
    wx = __shfl_sync(mask, wx, wl, L);
    if (sl == wl) rel &= ~(1u << wj);
    if (sl == r) {
      my_id = wl * EPL + wj;
      my_x = wx;
    }
  }
  // weights: the float64 path's arithmetic
  double sv = 0.0;
  if (sl < k) sv = 1.0 / (1.0 + exp(-(double)my_x));
  double sel = 0.0;
  for (int j = 0; j < k; ++j) sel += __shfl_sync(mask, sv, j, L);
  double w = sv;
  if (renorm) w = w / sel;
  w *= (double)scale;
  if (sl < k) {
    idx_out[row * k + sl] = (uint32_t)my_id;
    w_out[row * k + sl] = Dt<T>::from_f((float)w);
  }
}

// The chosen groups when the last chosen group and the best other one are closer than the FP32
// margin.  The groups sorted by FP32 score split into runs whose neighbours are within 2 E_g of
// each other; every group score is within E_g of its float64 value, so groups above the run that
// crosses the boundary stay chosen, groups below it stay out, and only that run needs float64
// group scores: the float64 top two (or best) of each of its groups, computed only for experts
// within 2 E_c of the group's FP32 second best (best), ranked by 64-bit keys (ties: lower group
// id).  gv, rank: group sl's FP32 score and rank in lanes sl < G; tq: this lane's group's FP32
// second best (best).  Returns the chosen groups, bit g for group g.  Out of line: rare.
template <typename T, int L, int EPL>
__device__ __noinline__ unsigned refine_groups(const T* __restrict__ src,
                                               const float* __restrict__ bias, const float* c,
                                               float ec, float eg, float tq, float gv, int rank,
                                               int G, int SG, int top_two, int sl, unsigned mask,
                                               int sub0) {
  constexpr int E = L * EPL;
  const int gs = E / G, lpg = gs / EPL;
  const unsigned lanes = L == 32 ? 0xFFFFFFFFu : (1u << L) - 1u;
  const bool glane = sl < G;
  float below = -INFINITY;  // the FP32 score of the group ranked just below group sl
  for (int g = 0; g < G; ++g) {
    const float o = __shfl_sync(mask, gv, g, L);
    const int orank = __shfl_sync(mask, rank, g, L);
    if (glane && orank == rank + 1) below = o;
  }
  const unsigned link = glane && rank + 1 < G && !(gv - below > 2.f * eg) ? 1u << rank : 0u;
  const unsigned links = __reduce_or_sync(mask, link);  // bit p: positions p, p+1 one run
  const unsigned starts = ~(links << 1);
  const int r0 = 31 - __clz(starts & ((2u << (SG - 1)) - 1u));  // the run's first position
  const int r1 = __ffs(~links & ~((1u << (SG - 1)) - 1u)) - 1;    // and its last (>= SG)
  const int grank = __shfl_sync(mask, rank, (sl / lpg) & 31, L);  // FP32 rank of sl's group
  const bool in_run = grank >= r0 && grank <= r1;
  float x[EPL], b[EPL];
  sub_load<T, EPL>(src, bias, sl * EPL, x, b);
  unsigned long long key[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) key[j] = 0ull;
  unsigned want = 0;
  if (in_run) {
#pragma unroll
    for (int j = 0; j < EPL; ++j) want |= (c[j] >= tq - 2.f * ec ? 1u : 0u) << j;
  }
  const unsigned need = want;
  while (__any_sync(mask, want != 0)) {  // one float64 score per lane and pass
    const int j = want ? __ffs(want) - 1 : -1;
    float xj = 0.f, bj = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      xj = (i == j) ? x[i] : xj;
      bj = (i == j) ? b[i] : bj;
    }
    const unsigned long long kj = j >= 0 ? dkey(sig_score64(xj, bj)) : 0ull;
#pragma unroll
    for (int i = 0; i < EPL; ++i) key[i] = (i == j) ? kj : key[i];
    if (j >= 0) want &= want - 1;
  }
  // the group's float64 top two (duplicates count), merged over its lanes
  unsigned long long k1 = 0, k2 = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    if (!((need >> j) & 1u)) continue;
    if (key[j] > k1) {
      k2 = k1;
      k1 = key[j];
    } else if (key[j] > k2) {
      k2 = key[j];
    }
  }
  for (int o = 1; o < lpg; o <<= 1) {
    const unsigned long long o1 = shfl_xor_u64(mask, k1, o, L), o2 = shfl_xor_u64(mask, k2, o, L);
    const unsigned long long n1 = k1 > o1 ? k1 : o1;
    const unsigned long long lo = k1 > o1 ? o1 : k1, hi2 = k2 > o2 ? k2 : o2;
    k2 = lo > hi2 ? lo : hi2;
    k1 = n1;
  }
  const double gsc = top_two ? dkey_value(k1) + dkey_value(k2) : dkey_value(k1);
  const unsigned long long gk = shfl_u64(mask, dkey(gsc), (glane ? sl : 0) * lpg, L);
  const bool grun = glane && rank >= r0 && rank <= r1;
  int rr = 0;  // rank inside the run by float64 score
  for (int g = 0; g < G; ++g) {
    const unsigned long long og = shfl_u64(mask, gk, g, L);
    const int orank = __shfl_sync(mask, rank, g, L);
    if (grun && orank >= r0 && orank <= r1 && (og > gk || (og == gk && g < sl))) ++rr;
  }
  const bool pick = glane && (rank < r0 || (grun && rr < SG - r0));
  return (__ballot_sync(mask, pick) >> sub0) & lanes;
}

// The float64 order of a row's best candidates when some of them lie closer than the FP32
// margin.  Lane r holds the r-th candidate by FP32 score (cur) and sees the next one (nxt); the
// sorted list splits into runs whose neighbours are within 2 E_c of each other.  Every score is
// within E_c of its float64 value, so candidates in different runs keep their FP32 order, and only
// the runs up to the one holding the top_k-th candidate need float64 scores: one per lane, ranked
// inside each run by 64-bit keys (ties: lower id).  Returns false, in every lane of the row, when
// that run reaches past the row's lanes (the caller then takes the full float64 decision);
// otherwise slot lanes (sl < k) get their expert in *id.  Out of line: rows get here rarely.
template <typename T, int L>
__device__ __noinline__ bool refine_runs(const T* __restrict__ src, const float* __restrict__ bias,
                                         unsigned long long cur, unsigned long long nxt, int n,
                                         int k, float ec, int sl, unsigned mask, int sub0,
                                         int* id) {
  const unsigned lanes = L == 32 ? 0xFFFFFFFFu : (1u << L) - 1u;
  const bool link = sl + 1 < n && !(skey_score(cur) - skey_score(nxt) > 2.f * ec);
  const unsigned links = (__ballot_sync(mask, link) >> sub0) & lanes;  // bit r: r, r+1 one run
  // e: the last position of the run holding position k - 1
  const unsigned open = ~links & lanes & ~((1u << (k - 1)) - 1u);
  if (open == 0) return false;
  const int e = __ffs(open) - 1;
  const unsigned starts = ~(links << 1);                               // bit r: a run starts at r
  const int r0 = 31 - __clz(starts & (sl == 31 ? 0xFFFFFFFFu : (2u << sl) - 1u));
  const int me = skey_id(cur);
  unsigned long long key = 0ull;
  if (sl <= e) key = dkey(sig_score64(Dt<T>::to_f(src[me]), bias ? bias[me] : 0.f));
  // rank inside the run, then the new position's expert
  int pos = r0;
  for (int j = 0; j <= e; ++j) {
    const unsigned long long kj = shfl_u64(mask, key, j, L);
    const int ij = __shfl_sync(mask, me, j, L);
    const int sj = __shfl_sync(mask, r0, j, L);
    if (sl <= e && sj == r0 && (kj > key || (kj == key && ij < me))) ++pos;
  }
  for (int j = 0; j <= e; ++j) {
    const int pj = __shfl_sync(mask, pos, j, L);
    const int ij = __shfl_sync(mask, me, j, L);
    if (pj == sl && sl < k) *id = ij;
  }
  return true;
}

// One row held by the L lanes of a sub-warp (see the file comment).  Returns true when it wrote
// the row's ids and weights (from the FP32 attempt, or when that cannot prove its choice, from
// the float64 decision above); false leaves the row (a non-finite score) to the warp-wide
// routine.  sl: lane in the row; scr: 2 L keys of shared memory owned by the row.
//
// The top_k experts of the chosen groups.  Each chosen group's two best experts are candidates,
// so when top_k <= 2 SG the top_k-th best candidate scores at least tau, the smallest second-best
// of the chosen groups; a candidate below tau - 3 E_c can then neither be chosen nor come within
// the margin of a chosen one.  The candidates at or above that line (about ten a row on the
// skewed layer's logits) are compacted into shared memory as 64-bit keys and ranked by counting;
// slot r takes the r-th key.  Rows with more than 2 L such candidates, or top_k > 2 SG, take
// top_k (+1) rounds of sub-warp argmax instead.
template <typename T, int L, int EPL>
__device__ __forceinline__ bool sigmoid_row_sub(const T* __restrict__ src,
                                                const float* __restrict__ bias, int64_t row, int k,
                                                int G, int SG, int top_two, int renorm,
                                                float scale, int sl, unsigned mask,
                                                unsigned long long* scr,
                                                uint32_t* __restrict__ idx_out,
                                                T* __restrict__ w_out) {
  constexpr int E = L * EPL;
  const int gs = E / G, lpg = gs / EPL;  // experts and lanes per group
  const int e0 = sl * EPL;
  float c[EPL];
  {
    float x[EPL], b[EPL];
    sub_load<T, EPL>(src, bias, e0, x, b);
#pragma unroll
    for (int j = 0; j < EPL; ++j) c[j] = 1.0f / (1.0f + expf(-x[j])) + b[j];
  }
  float amax = 0.f;
  bool finite = true;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    finite &= isfinite(c[j]);
    amax = fmaxf(amax, fabsf(c[j]));
  }
  if (!__all_sync(mask, finite)) return false;
#pragma unroll
  for (int o = 1; o < L; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(mask, amax, o, L));
  const float ec = 5e-7f + 1.2e-7f * amax;                     // bound on |c32 - c64|
  const float eg = (top_two ? 2.f * ec : ec) + 2.4e-7f * amax;  // bound on a group score
  // the top two of this lane's experts, merged over the group's lanes
  float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    if (c[j] > t1) {
      t2 = t1;
      t1 = c[j];
    } else if (c[j] > t2) {
      t2 = c[j];
    }
  }
  for (int o = 1; o < lpg; o <<= 1) {
    const float o1 = __shfl_xor_sync(mask, t1, o, L), o2 = __shfl_xor_sync(mask, t2, o, L);
    const float n1 = fmaxf(t1, o1);
    t2 = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
    t1 = n1;
  }
  const float gscore = top_two ? t1 + t2 : t1;
  // rank the G groups: lane g (< G) takes group g's score and counts the better ones
  const float gv = __shfl_sync(mask, gscore, (sl < G ? sl : 0) * lpg, L);
  int rank = 0;
  for (int g = 0; g < G; ++g) {
    const float o = __shfl_sync(mask, gv, g, L);
    rank += (o > gv) || (o == gv && g < sl);
  }
  const int sub0 = (threadIdx.x & 31) & ~(L - 1);  // first lane of this row in the warp
  unsigned chosen = (__ballot_sync(mask, sl < G && rank < SG) >> sub0) & (L == 32 ? 0xFFFFFFFFu : (1u << L) - 1u);
  if (SG < G) {  // the last chosen group must beat the best other group by the error margin
    const int l_last = __ffs((__ballot_sync(mask, sl < G && rank == SG - 1) >> sub0)) - 1;
    const int l_next = __ffs((__ballot_sync(mask, sl < G && rank == SG) >> sub0)) - 1;
    const float v_last = __shfl_sync(mask, gv, l_last, L);
    const float v_next = __shfl_sync(mask, gv, l_next, L);
    if (!(v_last - v_next > 2.f * eg))
      chosen = refine_groups<T, L, EPL>(src, bias, c, ec, eg, top_two ? t2 : t1, gv, rank, G, SG,
                                        top_two, sl, mask, sub0);
  }
  const bool mine = (chosen >> (sl / lpg)) & 1u;
  const int cand = SG * gs;
  int my_id = -1;
  bool decided = false;
  if (k <= 2 * SG) {
    float tau = mine ? t2 : INFINITY;
#pragma unroll
    for (int o = 1; o < L; o <<= 1) tau = fminf(tau, __shfl_xor_sync(mask, tau, o, L));
    const float line = tau - 3.f * ec;
    unsigned fm = 0;
    if (mine) {
#pragma unroll
      for (int j = 0; j < EPL; ++j) fm |= (c[j] >= line ? 1u : 0u) << j;
    }
    const int cnt = __popc(fm);
    int incl = cnt;  // inclusive prefix of the counts over the row's lanes
#pragma unroll
    for (int o = 1; o < L; o <<= 1) {
      const int y = __shfl_up_sync(mask, incl, o, L);
      if (sl >= o) incl += y;
    }
    const int n = __shfl_sync(mask, incl, L - 1, L);
    if (n <= 2 * L && n >= k) {  // n >= 2 SG >= top_k always holds; kept as a guard
      int pos = incl - cnt;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if ((fm >> j) & 1u) scr[pos++] = skey(c[j], e0 + j);
      __syncwarp(mask);
      const unsigned long long q0 = sl < n ? scr[sl] : 0ull;
      const unsigned long long q1 = sl + L < n ? scr[sl + L] : 0ull;
      int r0 = 0, r1 = 0;
      for (int i = 0; i < n; ++i) {
        const unsigned long long o = scr[i];
        r0 += o > q0 ? 1 : 0;
        r1 += o > q1 ? 1 : 0;
      }
      __syncwarp(mask);
      if (sl < n) scr[r0] = q0;  // keys are distinct: the ranks are a permutation of 0 .. n-1
      if (sl + L < n) scr[r1] = q1;
      __syncwarp(mask);
      const unsigned long long cur = sl < n ? scr[sl] : 0ull;
      const unsigned long long nxt = sl + 1 < n ? scr[sl + 1] : 0ull;
      __syncwarp(mask);  // scr is written again by the row's next use
      // slot r (< top_k) must beat the next candidate by the margin, unless the two have the same
      // logit and the same correction (the same score in any precision: the lower id first)
      const float vc = skey_score(cur), vn = skey_score(nxt);
      bool ok = !(sl < k && sl + 1 < n) || vc - vn > 2.f * ec, refined = false;
      if (!__all_sync(mask, ok)) {
        if (!ok) {
          const int ia = skey_id(cur), ib = skey_id(nxt);
          ok = vc == vn && Dt<T>::to_f(src[ia]) == Dt<T>::to_f(src[ib]) &&
               (bias == nullptr || bias[ia] == bias[ib]);
        }
        if (!__all_sync(mask, ok)) {
          if (!refine_runs<T, L>(src, bias, cur, nxt, n, k, ec, sl, mask, sub0, &my_id)) {
            sigmoid_row_sub_f64<T, L, EPL>(src, bias, c, ec, top_two ? t2 : t1, row, k, G, SG,
                                           top_two, renorm, scale, sl, mask, sub0, idx_out,
                                           w_out);
            return true;
          }
          refined = true;
        }
      }
      if (sl < k && !refined) my_id = skey_id(cur);
      decided = true;
    }
  }
  if (!decided) {
    // top_k (+1) rounds of sub-warp argmax over the chosen groups' experts; slot r kept in lane r
    float x[EPL], b[EPL];
    sub_load<T, EPL>(src, bias, e0, x, b);
    unsigned avail = mine ? (EPL == 32 ? 0xFFFFFFFFu : (1u << EPL) - 1u) : 0u;
    float prev = 0.f, px = 0.f, pb = 0.f;
    for (int r = 0; r < k + (k < cand ? 1 : 0); ++r) {
      float bv = -INFINITY;
      int bj = -1;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (((avail >> j) & 1u) && (bj < 0 || c[j] > bv)) {
          bv = c[j];
          bj = j;
        }
      float m = bv;
#pragma unroll
      for (int o = 1; o < L; o <<= 1) m = fmaxf(m, __shfl_xor_sync(mask, m, o, L));
      // the winner: the lowest lane holding the maximum, its lowest such expert
      const int wl = __ffs((__ballot_sync(mask, bj >= 0 && bv == m) >> sub0)) - 1;
      const int wj = __shfl_sync(mask, bj, wl, L);
      float wx = 0.f, wb = 0.f;
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        wx = (j == wj) ? x[j] : wx;
        wb = (j == wj) ? b[j] : wb;
      }
      wx = __shfl_sync(mask, wx, wl, L);
      wb = __shfl_sync(mask, wb, wl, L);
      if (r > 0 && !(prev - m > 2.f * ec) && !(m == prev && wx == px && wb == pb)) {
        sigmoid_row_sub_f64<T, L, EPL>(src, bias, c, ec, top_two ? t2 : t1, row, k, G, SG,
                                       top_two, renorm, scale, sl, mask, sub0, idx_out, w_out);
        return true;
      }
      if (r == k) break;
      prev = m;
      px = wx;
      pb = wb;
      if (sl == wl) avail &= ~(1u << wj);
      if (sl == r) my_id = wl * EPL + wj;
    }
  }
  // weights, as in the warp-wide attempt
  const float my_x = sl < k ? Dt<T>::to_f(src[my_id]) : 0.f;
  float w32 = 0.f;
  if (sl < k) w32 = 1.0f / (1.0f + expf(-my_x));
  float sel32 = 0.f;
  for (int j = 0; j < k; ++j) sel32 += __shfl_sync(mask, w32, j, L);
  bool exact = sizeof(T) == 2;
  T wout = Dt<T>::from_f(0.f);
  if (exact && sl < k) {
    constexpr float kWeightErr = 4e-6f;
    const float w = (renorm ? w32 / sel32 : w32) * scale;
    wout = Dt<T>::from_f(w);
    const T lo = Dt<T>::from_f(w * (1.f - kWeightErr)), hi = Dt<T>::from_f(w * (1.f + kWeightErr));
    exact = Dt<T>::to_f(lo) == Dt<T>::to_f(wout) && Dt<T>::to_f(hi) == Dt<T>::to_f(wout);
  }
  if (!__all_sync(mask, exact)) {
    double sv = 0.0;
    if (sl < k) sv = 1.0 / (1.0 + exp(-(double)my_x));
    double sel = 0.0;
    for (int j = 0; j < k; ++j) sel += __shfl_sync(mask, sv, j, L);
    double w = sv;
    if (renorm) w = w / sel;
    w *= (double)scale;
    wout = Dt<T>::from_f((float)w);
  }
  if (sl < k) {
    idx_out[row * k + sl] = (uint32_t)my_id;
    w_out[row * k + sl] = wout;
  }
  return true;
}

constexpr int kSubWarps = 8;

template <typename T, int L, int EPL>
__global__ void __launch_bounds__(kSubWarps * 32, 4)
    moe_route_sigmoid_sub(const T* __restrict__ logits, const float* __restrict__ bias,
                          int64_t T_, int k, int G, int SG, int top_two, int renorm, float scale,
                          uint32_t* __restrict__ idx_out, T* __restrict__ w_out) {
  constexpr int E = L * EPL, RPW = 32 / L, C = (E + 31) / 32;
  extern __shared__ double sig_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sl = lane & (L - 1);
  const unsigned mask = L == 32 ? 0xFFFFFFFFu : ((1u << L) - 1u) << (lane & ~(L - 1));
  // candidate keys of the sub-warp rows: 2 L per row, 64 per warp, after the warp-wide scratch
  unsigned long long* scr = reinterpret_cast<unsigned long long*>(
                                sig_smem + (size_t)kSubWarps * (E + 128 + 64 + 32)) +
                            warp * 64 + (lane / L) * 2 * L;
  const int64_t stride = (int64_t)gridDim.x * kSubWarps * RPW;
  for (int64_t base = ((int64_t)blockIdx.x * kSubWarps + warp) * RPW; base < T_; base += stride) {
    const int64_t row = base + lane / L;
    bool fallback = false;
    if (row < T_)
      fallback = !sigmoid_row_sub<T, L, EPL>(logits + row * E, bias, row, k, G, SG, top_two,
                                             renorm, scale, sl, mask, scr, idx_out, w_out);
    // rows the sub-warp attempt could not prove: the whole warp, one row at a time
    unsigned todo = __ballot_sync(0xFFFFFFFFu, fallback && sl == 0);
    while (todo) {
      const int l0 = __ffs(todo) - 1;
      todo &= todo - 1;
      const int64_t frow = base + l0 / L;
      sigmoid_route_row<T, C>(logits + frow * E, bias, frow, E, k, G, SG, top_two, renorm, scale,
                              sig_smem + (size_t)warp * (E + 128 + 64 + 32), lane, idx_out, w_out);
    }
  }
}

template <typename T, int L, int EPL>
cudaError_t launch_sig_sub(const void* logits, const float* bias, int64_t T_, int k, int G, int SG,
                           int top_two, int renorm, float scale, uint32_t* idx, void* w,
                           cudaStream_t s) {
  constexpr int E = L * EPL;
  const size_t smem = (size_t)kSubWarps * (E + 128 + 64 + 32 + 64) * sizeof(double);
  cudaError_t err = cudaFuncSetAttribute(moe_route_sigmoid_sub<T, L, EPL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t rows_per_block = (int64_t)kSubWarps * (32 / L);
  int64_t blocks = (T_ + rows_per_block - 1) / rows_per_block;
  if (blocks > 65535) blocks = 65535;
  if (blocks < 1) return cudaSuccess;
  moe_route_sigmoid_sub<T, L, EPL><<<(unsigned)blocks, kSubWarps * 32, smem, s>>>(
      (const T*)logits, bias, T_, k, G, SG, top_two, renorm, scale, idx, (T*)w);
  return cudaGetLastError();
}

// The sub-warp kernel for this shape, if it has one (returns cudaErrorNotSupported otherwise).
template <typename T>
cudaError_t launch_sig_sub_t(const void* logits, const float* bias, int64_t T_, int E, int k,
                             int G, int SG, int top_two, int renorm, float scale, uint32_t* idx,
                             void* w, cudaStream_t s) {
  if (((uintptr_t)logits & 15u) != 0 || (bias && ((uintptr_t)bias & 15u) != 0))
    return cudaErrorNotSupported;
  const int gs = E / G;
  for (int epl = 16; epl >= 8; epl /= 2) {
    const int L = E / epl;
    if (E % epl != 0 || gs % epl != 0 || L < 1 || L > 32 || (L & (L - 1)) != 0 || k > L) continue;
#define MOE_SIG_SUB(LL, EE)                                                                   \
  if (L == LL && epl == EE)                                                                   \
    return launch_sig_sub<T, LL, EE>(logits, bias, T_, k, G, SG, top_two, renorm, scale, idx, \
                                     w, s);
    MOE_SIG_SUB(32, 16) MOE_SIG_SUB(16, 16) MOE_SIG_SUB(8, 16) MOE_SIG_SUB(4, 16)
    MOE_SIG_SUB(2, 16) MOE_SIG_SUB(1, 16) MOE_SIG_SUB(32, 8) MOE_SIG_SUB(16, 8)
    MOE_SIG_SUB(8, 8) MOE_SIG_SUB(4, 8) MOE_SIG_SUB(2, 8) MOE_SIG_SUB(1, 8)
#undef MOE_SIG_SUB
  }
  return cudaErrorNotSupported;
}

template <typename T, int C>
cudaError_t launch_sig_c(const void* logits, const float* bias, int64_t T_, int E, int k, int G,
                         int SG, int top_two, int renorm, float scale, uint32_t* idx, void* w,
                         cudaStream_t s) {
  const size_t smem = (size_t)kSigWarps * (E + 128 + 64 + 32) * sizeof(double);
  cudaError_t err = cudaFuncSetAttribute(moe_route_sigmoid_kernel<T, C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const unsigned blocks = (unsigned)((T_ + kSigWarps - 1) / kSigWarps);
  moe_route_sigmoid_kernel<T, C><<<blocks, kSigWarps * 32, smem, s>>>(
      (const T*)logits, bias, T_, E, k, G, SG, top_two, renorm, scale, idx, (T*)w);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_sig_t(const void* logits, const float* bias, int64_t T_, int E, int k, int G,
                         int SG, int top_two, int renorm, float scale, uint32_t* idx, void* w,
                         cudaStream_t s) {
  const cudaError_t sub = launch_sig_sub_t<T>(logits, bias, T_, E, k, G, SG, top_two, renorm,
                                              scale, idx, w, s);
  if (sub != cudaErrorNotSupported) return sub;
#define MOE_SIG(CC)                                                                        \
  if (E <= 32 * CC)                                                                        \
    return launch_sig_c<T, CC>(logits, bias, T_, E, k, G, SG, top_two, renorm, scale, idx, \
                               w, s);
  MOE_SIG(1) MOE_SIG(2) MOE_SIG(4) MOE_SIG(8) MOE_SIG(16) MOE_SIG(32)
#undef MOE_SIG
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_route_sigmoid(const void* logits, int ldt, const float* bias, int64_t T_, int E,
                                 int k, int G, int SG, int top_two, int renorm, float scale,
                                 uint32_t* idx, void* w, cudaStream_t s) {
  switch (ldt) {
    case MOE_F32:
      return launch_sig_t<float>(logits, bias, T_, E, k, G, SG, top_two, renorm, scale, idx, w, s);
    case MOE_F16:
      return launch_sig_t<__half>(logits, bias, T_, E, k, G, SG, top_two, renorm, scale, idx, w, s);
    case MOE_BF16:
      return launch_sig_t<__nv_bfloat16>(logits, bias, T_, E, k, G, SG, top_two, renorm, scale,
                                         idx, w, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
