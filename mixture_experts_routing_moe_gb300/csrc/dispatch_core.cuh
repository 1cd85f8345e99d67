// Dispatch of a short batch by one block (ruDNN user guide, §5 "Expertengewichte und
// Verteilung"): count, scan and stable scatter of R <= a few thousand slots with the histograms in
// shared memory.  Warp w of `nwarps` owns the contiguous slot chunk [w*CH, w*CH + CH) (CH a
// multiple of 32, nwarps * CH >= R); inside a chunk, lanes with the same expert are ranked by
// lane with a per-bit ballot mask.  Rows of expert e keep ascending slot order s = t*k + j, whatever nwarps
// is.  Shared by the dispatch kernel for short batches and the fused decode kernel.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace moe {

// Lanes of the warp whose `key` equals this lane's (the mask __match_any_sync would give), from
// one ballot per key bit: valid keys are < 2^nbits, invalid lanes pass valid = false and match
// only each other.  Cheaper than match.any for the few bits of an expert id.
__device__ __forceinline__ unsigned same_key_lanes(uint32_t key, bool valid, int nbits) {
  unsigned m = __ballot_sync(0xFFFFFFFFu, valid);
  if (!valid) m = ~m;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (key >> b) & 1u;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, bit);
    m &= bit ? bal : ~bal;
  }
  return m;
}

// hist: shared [nwarps * E]; off: shared [E + 1], left holding the offsets.  offsets_out and
// row_of_slot may be null (not written); token_of_row may point to shared or global memory.
// IDX_SMEM: idx is in shared memory (plain loads); otherwise it is read with __ldg.  Expert ids
// >= E are not dispatched: their row_of_slot is kInvalidRow and the status word gets the index bit.
// dispatch_count: histograms, offsets (off, offsets_out) and each chunk's starting rows in hist.
template <bool IDX_SMEM>
__device__ __forceinline__ void dispatch_count(const uint32_t* __restrict__ idx, int64_t R, int E,
                                               int nwarps, int CH, int32_t* hist, int32_t* off,
                                               int32_t* offsets_out, unsigned* status) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < nwarps * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t s0 = (int64_t)warp * CH, s1 = (R < s0 + CH) ? R : s0 + CH;
  int32_t* h = hist + warp * E;
  const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;  // bits of an expert id
  bool bad = false;
  for (int64_t base = s0; base < s1; base += 32) {  // counts: order does not matter
    const int64_t s = base + lane;
    const bool act = s < s1;
    const uint32_t e = act ? (IDX_SMEM ? idx[s] : __ldg(idx + s)) : 0xFFFFFFFFu;
    const bool valid = act && e < (uint32_t)E;
    bad |= act && !valid;
    if (valid) atomicAdd(&h[e], 1);
  }
  __syncwarp();
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && status) atomicOr(status, kStatusIndex);
  __syncthreads();
  // per expert: exclusive prefix over the chunks, and the expert's total
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int32_t c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    off[e] = run;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the totals -> offsets
    int32_t carry = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int32_t c = e < E ? off[e] : 0;
      int32_t x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      if (e < E) {
        off[e] = carry + x - c;
        if (offsets_out) offsets_out[e] = carry + x - c;
      }
      carry += __shfl_sync(0xFFFFFFFFu, x, 31);
    }
    if (lane == 0) {
      off[E] = carry;
      if (offsets_out) offsets_out[E] = carry;
    }
  }
  __syncthreads();
  if (warp < nwarps) {
    for (int e = lane; e < E; e += 32) h[e] += off[e];  // running row of each expert in this chunk
  }
  __syncwarp();
}

// Second half of dispatch_block (same arguments; hist and off as left by dispatch_count).  Only
// warps 0 .. nwarps-1 take part, so other warps of the block may do something else meanwhile.
template <bool IDX_SMEM>
__device__ __forceinline__ void dispatch_scatter(const uint32_t* __restrict__ idx, int64_t R, int E,
                                                 int k, int CH, int32_t* hist,
                                                 uint32_t* token_of_row, uint32_t* row_of_slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t s0 = (int64_t)warp * CH, s1 = (R < s0 + CH) ? R : s0 + CH;
  int32_t* h = hist + warp * E;
  const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;  // bits of an expert id
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t base = s0; base < s1; base += 32) {
    const int64_t s = base + lane;
    const bool act = s < s1;
    const uint32_t e = act ? (IDX_SMEM ? idx[s] : __ldg(idx + s)) : 0xFFFFFFFFu;
    const bool valid = act && e < (uint32_t)E;
    const unsigned peers = same_key_lanes(e, valid, nbits);
    if (valid) {
      const uint32_t row = (uint32_t)(h[e] + __popc(peers & lt));
      if (row_of_slot) row_of_slot[s] = row;
      token_of_row[row] = (uint32_t)s / (uint32_t)k;  // s < 2^31
    } else if (act && row_of_slot) {
      row_of_slot[s] = kInvalidRow;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) h[e] += __popc(peers);
    __syncwarp();
  }
}

template <bool IDX_SMEM>
__device__ __forceinline__ void dispatch_block(const uint32_t* __restrict__ idx, int64_t R, int E,
                                               int k, int nwarps, int CH, int32_t* hist,
                                               int32_t* off, int32_t* offsets_out,
                                               uint32_t* token_of_row, uint32_t* row_of_slot,
                                               unsigned* status) {
  dispatch_count<IDX_SMEM>(idx, R, E, nwarps, CH, hist, off, offsets_out, status);
  if ((int)(threadIdx.x >> 5) < nwarps)
    dispatch_scatter<IDX_SMEM>(idx, R, E, k, CH, hist, token_of_row, row_of_slot);
}

}  // namespace moe
