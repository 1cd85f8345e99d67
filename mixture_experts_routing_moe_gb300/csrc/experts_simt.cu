// f32 SwiGLU experts on CUDA cores: SwiGluExperts::forward_dispatched of the ruDNN user guide,
// §5 "Expertengewichte und Verteilung" (gate/up [E, I, H], down [E, H, I], no bias).
//
// Two ragged grouped GEMMs over the dispatched rows of each expert, FP32 FMA throughout:
//   kernel 1:  a[r, i] = silu(x_d[r] . gate[e, i]) * (x_d[r] . up[e, i])
//   kernel 2:  y[r, h] = a[r] . down[e, h]
// Block tiles are 64 rows x 64 columns with 16-deep K slices in shared memory; a block finds its
// expert from the m-tile prefix of the device-side offsets, so the launch needs no host sync.
// Used for f32 layers, where tensor-core rates do not apply.
#include "common.cuh"
#include "launch.h"
#include "tiles.cuh"

namespace moe {
namespace {

constexpr int SB = 64, SK = 16;

template <bool GATEUP>
__global__ void __launch_bounds__(256)
    moe_experts_simt(const float* __restrict__ A, const int32_t* __restrict__ offsets, int E,
                     int K, int N, const float* __restrict__ B0, const float* __restrict__ B1,
                     float* __restrict__ C) {
  __shared__ int pref[1025];
  __shared__ float As[SK][SB + 4];
  __shared__ float Bs0[SK][SB + 4];
  __shared__ float Bs1[GATEUP ? SK : 1][SB + 4];
  const int tid = threadIdx.x;
  if (tid < 32) build_mtile_prefix(offsets, E, SB, pref, tid);
  __syncthreads();
  const int j = blockIdx.x;
  if (j >= pref[E]) return;
  const int e = find_expert(pref, E, j);
  const int row0 = offsets[e] + (j - pref[e]) * SB;
  const int row_end = offsets[e + 1];
  const int n0 = blockIdx.y * SB;
  const float* b0 = B0 + (int64_t)e * N * K;
  const float* b1 = GATEUP ? B1 + (int64_t)e * N * K : nullptr;

  const int tx = tid & 15, ty = tid >> 4;
  float acc0[4][4] = {}, acc1[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += SK) {
    // 64 x 16 slices: each thread loads 4 elements of A and of each B (transposed into smem)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int li = tid + q * 256;
      const int r = li / SK, kk = li % SK;
      const int gk = k0 + kk;
      const int ar = row0 + r;
      As[kk][r] = (ar < row_end && gk < K) ? A[(int64_t)ar * K + gk] : 0.f;
      const int bn = n0 + r;
      Bs0[kk][r] = (bn < N && gk < K) ? b0[(int64_t)bn * K + gk] : 0.f;
      if (GATEUP) Bs1[kk][r] = (bn < N && gk < K) ? b1[(int64_t)bn * K + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SK; ++kk) {
      float a[4], b[4], c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs0[kk][tx * 4 + i];
        if (GATEUP) c[i] = Bs1[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc0[i][q] = fmaf(a[i], b[q], acc0[i][q]);
          if (GATEUP) acc1[i][q] = fmaf(a[i], c[q], acc1[i][q]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= row_end) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + tx * 4 + q;
      if (n >= N) continue;
      float v = acc0[i][q];
      if (GATEUP) v = v / (1.f + expf(-v)) * acc1[i][q];
      C[(int64_t)r * N + n] = v;
    }
  }
}

}  // namespace

cudaError_t launch_experts_simt(const float* x_d, const int32_t* offsets, int64_t rows,
                                const float* gate, const float* up, const float* down, int E,
                                int H, int I, float* y, float* a, cudaStream_t s,
                                cudaEvent_t between) {
  const int64_t mtiles = (rows + SB - 1) / SB + E;  // upper bound of sum_e ceil(n_e / 64)
  dim3 g1((unsigned)mtiles, (unsigned)((I + SB - 1) / SB));
  moe_experts_simt<true><<<g1, 256, 0, s>>>(x_d, offsets, E, H, I, gate, up, a);
  if (between) {
    const cudaError_t err = cudaEventRecord(between, s);
    if (err != cudaSuccess) return err;
  }
  dim3 g2((unsigned)mtiles, (unsigned)((H + SB - 1) / SB));
  moe_experts_simt<false><<<g2, 256, 0, s>>>(a, offsets, E, I, H, down, nullptr, y);
  return cudaGetLastError();
}

}  // namespace moe
