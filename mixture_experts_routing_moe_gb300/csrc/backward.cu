// Backward chain of the local MoE layer: combine_backward, the expert backward and
// dispatch_backward of the ruDNN user guide, §12 "MoE-Training erster Ordnung".
//
//   combine_backward:  dexpert[row(t, j)] = w[t, j] * dout[t]          (y dtype)
//                      dweights[t, j]     = <dout[t], y[row(t, j)]>    (FP32)
//   expert backward (per expert e, its dispatched rows r; g = x gate_e^T, u = x up_e^T recomputed):
//                      da = dy down_e;  s = sigmoid(g);  du = da * g s;  dg = da * u * s (1 + g (1 - s))
//                      dx = dg gate_e + du up_e                        (layer dtype)
//                      ddown_e = dy^T a (a = g s u);  dgate_e = dg^T x;  dup_e = du^T x   (FP32)
//   dispatch_backward: dx[t] = sum_j dinput[row(t, j)]                 (no routing weights)
//
// The expert backward runs on CUDA cores in FP32: 64 x 64 tiles, 16-deep K slices in shared
// memory, ragged per-expert row groups found from the device-side offsets (rows for the
// activation GEMMs, the contraction dimension for the weight gradients).  Sums over slots are
// in slot order and sums inside a tile in a fixed order, so results are run-to-run identical.
#include "combine_core.cuh"
#include "common.cuh"
#include "launch.h"
#include "tiles.cuh"

namespace moe {
namespace {

constexpr int TB = 64, TK = 16;

template <typename T>
__device__ __forceinline__ float ldf(const T* p) {
  return Dt<T>::to_f(*p);
}

// ------------------------------------------------------------------ combine / dispatch backward
template <typename TY, typename TW>
__global__ void __launch_bounds__(256)
    moe_combine_bwd_kernel(const TY* __restrict__ y, const uint32_t* __restrict__ row_of_slot,
                           const TW* __restrict__ w, const TY* __restrict__ dout, int64_t T_,
                           int64_t H, int k, TY* __restrict__ dexpert,
                           float* __restrict__ dweights) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T_) return;
  const TY* go = dout + t * H;
  for (int j = 0; j < k; ++j) {
    const uint32_t r = row_of_slot[t * k + j];
    const float wj = Dt<TW>::to_f(w[t * k + j]);
    float dot = 0.f;
    if (r != kInvalidRow) {
      const TY* yr = y + (int64_t)r * H;
      TY* dr = dexpert + (int64_t)r * H;
      for (int64_t h = lane; h < H; h += 32) {
        const float g = ldf(go + h);
        dot = fmaf(g, ldf(yr + h), dot);
        dr[h] = Dt<TY>::from_f(wj * g);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
    if (lane == 0) dweights[t * k + j] = r == kInvalidRow ? __int_as_float(0x7FC00000) : dot;
  }
}

// Vectorised combine backward for top_k <= 8 and 16-byte rows: one warp per token, lanes over
// 16-byte column chunks; per chunk the k rows of y are loaded together, dexpert = w dout is
// written (the same values as the scalar kernel) and the k dot products accumulate in a fixed
// order (chunk by chunk, then a xor tree), so the result is the same on every run.
template <typename TY, typename TW>
__global__ void __launch_bounds__(256)
    moe_combine_bwd_vec(const TY* __restrict__ y, const uint32_t* __restrict__ row_of_slot,
                        const TW* __restrict__ w, const TY* __restrict__ dout, int64_t T_,
                        int64_t H, int k, TY* __restrict__ dexpert, float* __restrict__ dweights) {
  constexpr int VW = 16 / (int)sizeof(TY);
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T_) return;
  uint32_t r[8];
  float wj[8], dot[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    r[j] = j < k ? row_of_slot[t * k + j] : kInvalidRow;
    wj[j] = j < k ? Dt<TW>::to_f(w[t * k + j]) : 0.f;
    dot[j] = 0.f;
  }
  const int64_t chunks = H / VW;
  for (int64_t c = lane; c < chunks; c += 32) {
    Vec16<TY> g;
    g.u = ld_nc_v4(dout + t * H + c * VW);
    float gf[VW];
    g.to_float(gf);
    uint4 yv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (r[j] != kInvalidRow) yv[j] = ld_nc_v4(y + (int64_t)r[j] * H + c * VW);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (r[j] != kInvalidRow) {
        Vec16<TY> q;
        q.u = yv[j];
        float yf[VW], of[VW];
        q.to_float(yf);
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < VW; ++i) {
          d = fmaf(gf[i], yf[i], d);
          of[i] = wj[j] * gf[i];
        }
        dot[j] += d;
        Vec16<TY> o;
        o.from_float(of);
        st_v4(dexpert + (int64_t)r[j] * H + c * VW, o.u);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot[j] += __shfl_xor_sync(0xFFFFFFFFu, dot[j], o);
    if (lane == 0 && j < k)
      dweights[t * k + j] = r[j] == kInvalidRow ? __int_as_float(0x7FC00000) : dot[j];
  }
}

// Rows of dexpert that no slot maps to.  moe_dispatch gives the n valid slots the rows 0 .. n-1
// (a bijection), so the rows it leaves unused are the last R - n, one per slot with row
// 0xFFFFFFFF; they exist only when some expert ids were invalid.  One block counts those slots
// and zeroes that many trailing rows, so dexpert is fully defined whatever the buffer held.
template <typename TY>
__global__ void __launch_bounds__(1024)
    moe_combine_bwd_zero_tail(const uint32_t* __restrict__ row_of_slot, int64_t R, int64_t H,
                              TY* __restrict__ dexpert) {
  __shared__ unsigned long long n_bad;
  if (threadIdx.x == 0) n_bad = 0;
  __syncthreads();
  unsigned long long c = 0;
  for (int64_t s = threadIdx.x; s < R; s += blockDim.x) c += row_of_slot[s] == kInvalidRow;
  if (c) atomicAdd(&n_bad, c);
  __syncthreads();
  const int64_t first = R - (int64_t)n_bad;  // the first unused row
  if (first >= R) return;
  const int64_t n = (R - first) * H;
  TY* d = dexpert + first * H;
  const TY z = Dt<TY>::from_f(0.f);
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = z;
}

template <typename T>
__global__ void __launch_bounds__(256)
    moe_dispatch_bwd_kernel(const T* __restrict__ dinput, const uint32_t* __restrict__ row_of_slot,
                            int64_t T_, int64_t H, int k, T* __restrict__ dx) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T_) return;
  for (int64_t h = lane; h < H; h += 32) {
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
      const uint32_t r = row_of_slot[t * k + j];
      acc += r == kInvalidRow ? __int_as_float(0x7FC00000) : ldf(dinput + (int64_t)r * H + h);
    }
    dx[t * H + h] = Dt<T>::from_f(acc);
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
    moe_dispatch_bwd_vec(const T* __restrict__ dinput, const uint32_t* __restrict__ row_of_slot,
                         int64_t T_, int64_t H, int k, int64_t wpt, T* __restrict__ dx) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t t = gw / wpt;
  if (t >= T_) return;
  combine_warp<T, float, true, false, 1>(dinput, row_of_slot, nullptr, t, H, k, gw - t * wpt, dx,
                                         lane);
}

// ------------------------------------------------------------------ ragged row GEMMs
// C[r, n] = sum_k A[r, k] * B_e(k, n) for the rows r of expert e, with
//   BMODE 0: B_e(k, n) = W0_e[n * K + k]          (x W^T, W_e stored [N, K])
//   BMODE 1: B_e(k, n) = W0_e[k * N + n]          (dy W, W_e stored [K, N])
//   BMODE 2: B_e(k, n) = k < K/2 ? W0_e[k * N + n] : W1_e[(k - K/2) * N + n]   ([dg du] [gate; up])
// Epilogues: EPI 0 store FP32; EPI 1 the da epilogue (reads g, u; writes dg, du, a);
//            EPI 2 store in TO (rounded once).
enum { EPI_F32 = 0, EPI_DGDU = 1, EPI_OUT = 2 };

template <typename TA, typename TWt, int BMODE, int EPI, typename TO>
__global__ void __launch_bounds__(256)
    moe_bwd_rowgemm(const TA* __restrict__ A, int lda, const int32_t* __restrict__ offsets, int E,
                    int K, int N, const TWt* __restrict__ W0, const TWt* __restrict__ W1,
                    int64_t wstride, float* __restrict__ Cf, TO* __restrict__ Co, int ldc,
                    const float* __restrict__ gbuf, const float* __restrict__ ubuf,
                    float* __restrict__ dgdu, float* __restrict__ abuf) {
  __shared__ int pref[1025];
  __shared__ float As[TK][TB + 4];
  __shared__ float Bs[TK][TB + 4];
  const int tid = threadIdx.x;
  if (tid < 32) build_mtile_prefix(offsets, E, TB, pref, tid);
  __syncthreads();
  const int j = blockIdx.x;
  if (j >= pref[E]) return;
  const int e = find_expert(pref, E, j);
  const int row0 = offsets[e] + (j - pref[e]) * TB;
  const int row_end = offsets[e + 1];
  const int n0 = blockIdx.y * TB;
  const TWt* w0 = W0 + (int64_t)e * wstride;
  const TWt* w1 = BMODE == 2 ? W1 + (int64_t)e * wstride : nullptr;
  const int tx = tid & 15, ty = tid >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int li = tid + q * 256;
      const int rr = li / TK, kk = li % TK;   // A: 64 rows x 16 k
      const int gk = k0 + kk, ar = row0 + rr;
      As[kk][rr] = (ar < row_end && gk < K) ? ldf(A + (int64_t)ar * lda + gk) : 0.f;
      // B: 16 k x 64 n; for BMODE 0 walk k fastest (contiguous in W), else n fastest
      int bk, bn;
      if (BMODE == 0) {
        bn = li / TK;
        bk = li % TK;
      } else {
        bk = li / TB;
        bn = li % TB;
      }
      const int gk2 = k0 + bk, gn = n0 + bn;
      float bv = 0.f;
      if (gk2 < K && gn < N) {
        if (BMODE == 0) bv = ldf(w0 + (int64_t)gn * K + gk2);
        else if (BMODE == 1) bv = ldf(w0 + (int64_t)gk2 * N + gn);
        else {
          const int half = K / 2;
          bv = gk2 < half ? ldf(w0 + (int64_t)gk2 * N + gn) : ldf(w1 + (int64_t)(gk2 - half) * N + gn);
        }
      }
      Bs[bk][bn] = bv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(a[i], b[q], acc[i][q]);
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
      const float v = acc[i][q];
      if (EPI == EPI_F32) {
        Cf[(int64_t)r * ldc + n] = v;
      } else if (EPI == EPI_OUT) {
        Co[(int64_t)r * ldc + n] = Dt<TO>::from_f(v);
      } else {  // da epilogue: N = I
        const float g = gbuf[(int64_t)r * N + n], u = ubuf[(int64_t)r * N + n];
        const float s = 1.f / (1.f + expf(-g));
        const float act = g * s;
        dgdu[(int64_t)r * 2 * N + n] = v * u * s * (1.f + g * (1.f - s));
        dgdu[(int64_t)r * 2 * N + N + n] = v * act;
        abuf[(int64_t)r * N + n] = act * u;
      }
    }
  }
}

// ------------------------------------------------------------------ weight gradients
// C_e[m, n] = sum over the rows r of expert e of A[r, m] * B[r, n]; C is [E, M, N] FP32.
template <typename TA, typename TBt>
__global__ void __launch_bounds__(256)
    moe_bwd_wgrad(const TA* __restrict__ A, int lda, const TBt* __restrict__ B, int ldb,
                  const int32_t* __restrict__ offsets, int M, int N, float* __restrict__ C) {
  __shared__ float As[TK][TB + 4];
  __shared__ float Bs[TK][TB + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int e = blockIdx.z, m0 = blockIdx.y * TB, n0 = blockIdx.x * TB;
  const int lo = offsets[e], hi = offsets[e + 1];
  float acc[4][4] = {};
  for (int r0 = lo; r0 < hi; r0 += TK) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int li = tid + q * 256;
      const int kk = li / TB, c = li % TB;    // 16 rows x 64 columns, columns contiguous
      const int r = r0 + kk;
      As[kk][c] = (r < hi && m0 + c < M) ? ldf(A + (int64_t)r * lda + m0 + c) : 0.f;
      Bs[kk][c] = (r < hi && n0 + c < N) ? ldf(B + (int64_t)r * ldb + n0 + c) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(a[i], b[q], acc[i][q]);
    }
    __syncthreads();
  }
  float* Ce = C + (int64_t)e * M * N;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int n = n0 + tx * 4 + q;
      if (n < N) Ce[(int64_t)m * N + n] = acc[i][q];
    }
  }
}

template <typename T>
cudaError_t experts_bwd_t(const void* x_d, const int32_t* offsets, int64_t rows, const void* gate,
                          const void* up, const void* down, int E, int H, int I, const void* dy,
                          void* dinput, float* dgate, float* dup, float* ddown, float* ws,
                          cudaStream_t s) {
  float* g = ws;
  float* u = g + (size_t)rows * I;
  float* a = u + (size_t)rows * I;
  float* dgdu = a + (size_t)rows * I;  // [rows, 2I]
  const int64_t mt = (rows + TB - 1) / TB + E;  // >= sum_e ceil(n_e / 64)
  const T *X = (const T*)x_d, *G = (const T*)gate, *U = (const T*)up, *D = (const T*)down,
          *DY = (const T*)dy;
  const dim3 gI((unsigned)mt, (unsigned)((I + TB - 1) / TB)), gH((unsigned)mt, (unsigned)((H + TB - 1) / TB));
  const int64_t ws_ih = (int64_t)I * H;
  // g = x gate^T, u = x up^T
  moe_bwd_rowgemm<T, T, 0, EPI_F32, float><<<gI, 256, 0, s>>>(X, H, offsets, E, H, I, G, nullptr,
                                                              ws_ih, g, nullptr, I, nullptr,
                                                              nullptr, nullptr, nullptr);
  moe_bwd_rowgemm<T, T, 0, EPI_F32, float><<<gI, 256, 0, s>>>(X, H, offsets, E, H, I, U, nullptr,
                                                              ws_ih, u, nullptr, I, nullptr,
                                                              nullptr, nullptr, nullptr);
  // da = dy down_e (down_e [H, I] = [K, N]); epilogue: dg, du, a
  moe_bwd_rowgemm<T, T, 1, EPI_DGDU, float><<<gI, 256, 0, s>>>(DY, H, offsets, E, H, I, D, nullptr,
                                                               ws_ih, nullptr, nullptr, I, g, u,
                                                               dgdu, a);
  // dx = [dg du] [gate_e; up_e]  (K = 2I, gate_e / up_e [I, H] = [K/2, N])
  moe_bwd_rowgemm<float, T, 2, EPI_OUT, T><<<gH, 256, 0, s>>>(dgdu, 2 * I, offsets, E, 2 * I, H, G,
                                                              U, ws_ih, nullptr, (T*)dinput, H,
                                                              nullptr, nullptr, nullptr, nullptr);
  // weight gradients, contracted over each expert's rows
  const dim3 gD((unsigned)((I + TB - 1) / TB), (unsigned)((H + TB - 1) / TB), (unsigned)E);
  moe_bwd_wgrad<T, float><<<gD, 256, 0, s>>>(DY, H, a, I, offsets, H, I, ddown);
  const dim3 gG((unsigned)((H + TB - 1) / TB), (unsigned)((I + TB - 1) / TB), (unsigned)E);
  moe_bwd_wgrad<float, T><<<gG, 256, 0, s>>>(dgdu, 2 * I, X, H, offsets, I, H, dgate);
  moe_bwd_wgrad<float, T><<<gG, 256, 0, s>>>(dgdu + I, 2 * I, X, H, offsets, I, H, dup);
  return cudaGetLastError();
}

template <typename TY, typename TW>
cudaError_t combine_bwd_tw(const void* y, const uint32_t* ros, const void* w, const void* dout,
                           int64_t T_, int64_t H, int k, void* dexpert, float* dweights,
                           cudaStream_t s) {
  const bool vec = k <= 8 && (H * (int64_t)sizeof(TY)) % 16 == 0 && (uintptr_t)y % 16 == 0 &&
                   (uintptr_t)dout % 16 == 0 && (uintptr_t)dexpert % 16 == 0;
  if (vec)
    moe_combine_bwd_vec<TY, TW><<<(unsigned)((T_ + 7) / 8), 256, 0, s>>>(
        (const TY*)y, ros, (const TW*)w, (const TY*)dout, T_, H, k, (TY*)dexpert, dweights);
  else
    moe_combine_bwd_kernel<TY, TW><<<(unsigned)((T_ + 7) / 8), 256, 0, s>>>(
        (const TY*)y, ros, (const TW*)w, (const TY*)dout, T_, H, k, (TY*)dexpert, dweights);
  return cudaGetLastError();
}
template <typename TY>
cudaError_t combine_bwd_t(const void* y, const uint32_t* ros, const void* w, int wdt,
                          const void* dout, int64_t T_, int64_t H, int k, void* dexpert,
                          float* dweights, cudaStream_t s) {
  // the unused trailing rows first: a valid slot that maps into them (a row map not made by
  // moe_dispatch) is then still written by the kernel below
  moe_combine_bwd_zero_tail<TY><<<1, 1024, 0, s>>>(ros, T_ * k, H, (TY*)dexpert);
  cudaError_t err = cudaErrorInvalidValue;
  switch (wdt) {
    case MOE_F32:
      err = combine_bwd_tw<TY, float>(y, ros, w, dout, T_, H, k, dexpert, dweights, s);
      break;
    case MOE_F16:
      err = combine_bwd_tw<TY, __half>(y, ros, w, dout, T_, H, k, dexpert, dweights, s);
      break;
    case MOE_BF16:
      err = combine_bwd_tw<TY, __nv_bfloat16>(y, ros, w, dout, T_, H, k, dexpert, dweights, s);
      break;
  }
  return err;
}

}  // namespace

size_t experts_backward_scratch_bytes(int64_t rows, int64_t I) {
  return (size_t)rows * (size_t)I * 5 * sizeof(float);
}

cudaError_t launch_experts_backward(const void* x_d, const int32_t* offsets, int64_t rows,
                                    const void* gate, const void* up, const void* down, int wdt,
                                    int E, int H, int I, const void* dy, void* dinput,
                                    float* dgate, float* dup, float* ddown, float* scratch,
                                    cudaStream_t s) {
  switch (wdt) {
    case MOE_F32:
      return experts_bwd_t<float>(x_d, offsets, rows, gate, up, down, E, H, I, dy, dinput, dgate,
                                  dup, ddown, scratch, s);
    case MOE_F16:
      return experts_bwd_t<__half>(x_d, offsets, rows, gate, up, down, E, H, I, dy, dinput, dgate,
                                   dup, ddown, scratch, s);
    case MOE_BF16:
      return experts_bwd_t<__nv_bfloat16>(x_d, offsets, rows, gate, up, down, E, H, I, dy, dinput,
                                          dgate, dup, ddown, scratch, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine_backward(const void* y, int ydt, const uint32_t* ros, const void* w,
                                    int wdt, const void* dout, int64_t T_, int64_t H, int k,
                                    void* dexpert, float* dweights, cudaStream_t s) {
  switch (ydt) {
    case MOE_F32:
      return combine_bwd_t<float>(y, ros, w, wdt, dout, T_, H, k, dexpert, dweights, s);
    case MOE_F16:
      return combine_bwd_t<__half>(y, ros, w, wdt, dout, T_, H, k, dexpert, dweights, s);
    case MOE_BF16:
      return combine_bwd_t<__nv_bfloat16>(y, ros, w, wdt, dout, T_, H, k, dexpert, dweights, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_dispatch_backward(const void* dinput, int dt, const uint32_t* ros, int64_t T_,
                                     int64_t H, int k, void* dx, cudaStream_t s) {
  // 16-byte rows: the combine's warp routine with unit weights (a token spread over
  // ceil(H / (32 x 16 B)) warps, FP32 slot-order sums, NaN for a slot without a row)
  const int es = dt == MOE_F32 ? 4 : 2;
  if ((H * es) % 16 == 0 && (uintptr_t)dinput % 16 == 0 && (uintptr_t)dx % 16 == 0 &&
      (dt == MOE_F32 || dt == MOE_F16 || dt == MOE_BF16)) {
    const int64_t chunks = H * es / 16, wpt = (chunks + 31) / 32;
    const unsigned nb = (unsigned)((T_ * wpt + 7) / 8);
    switch (dt) {
      case MOE_F32:
        moe_dispatch_bwd_vec<float><<<nb, 256, 0, s>>>((const float*)dinput, ros, T_, H, k, wpt,
                                                        (float*)dx);
        break;
      case MOE_F16:
        moe_dispatch_bwd_vec<__half><<<nb, 256, 0, s>>>((const __half*)dinput, ros, T_, H, k, wpt,
                                                         (__half*)dx);
        break;
      default:
        moe_dispatch_bwd_vec<__nv_bfloat16><<<nb, 256, 0, s>>>(
            (const __nv_bfloat16*)dinput, ros, T_, H, k, wpt, (__nv_bfloat16*)dx);
    }
    return cudaGetLastError();
  }
  const unsigned blocks = (unsigned)((T_ + 7) / 8);
  switch (dt) {
    case MOE_F32:
      moe_dispatch_bwd_kernel<float><<<blocks, 256, 0, s>>>((const float*)dinput, ros, T_, H, k,
                                                             (float*)dx);
      break;
    case MOE_F16:
      moe_dispatch_bwd_kernel<__half><<<blocks, 256, 0, s>>>((const __half*)dinput, ros, T_, H, k,
                                                              (__half*)dx);
      break;
    case MOE_BF16:
      moe_dispatch_bwd_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
          (const __nv_bfloat16*)dinput, ros, T_, H, k, (__nv_bfloat16*)dx);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace moe
