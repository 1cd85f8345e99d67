// Shared device helpers of libmoe: dtype traits, 16-byte vector access, the workspace layout.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr uint32_t kInvalidRow = 0xFFFFFFFFu;
// The first 256 bytes of every workspace hold the device status word (and padding).
constexpr size_t kWsHeader = 256;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

template <typename T> struct Dt;
template <> struct Dt<float> {
  static constexpr int code = MOE_F32;
  __device__ static float to_f(float v) { return v; }
  __device__ static float from_f(float v) { return v; }
};
template <> struct Dt<__half> {
  static constexpr int code = MOE_F16;
  __device__ static float to_f(__half v) { return __half2float(v); }
  __device__ static __half from_f(float v) { return __float2half_rn(v); }
};
template <> struct Dt<__nv_bfloat16> {
  static constexpr int code = MOE_BF16;
  __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Eight (or four, for f32) elements of a 16-byte vector as floats.
template <typename T> struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  union {
    uint4 u;
    T e[N];
  };
  __device__ void to_float(float* f) const {
#pragma unroll
    for (int i = 0; i < N; ++i) f[i] = Dt<T>::to_f(e[i]);
  }
  __device__ void from_float(const float* f) {
#pragma unroll
    for (int i = 0; i < N; ++i) e[i] = Dt<T>::from_f(f[i]);
  }
};

__device__ inline uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ inline void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
// Streaming store: the written lines are not re-read by this kernel.
__device__ inline void st_cs_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Loads cached in L2 only: coherent with stores that other CTAs of the same launch made visible
// (through a fence and a grid barrier) before this thread loads; never served from a stale L1.
__device__ inline uint4 ld_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}
__device__ inline uint32_t ld_cg_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
  return r;
}
__device__ inline uint16_t ld_cg_u16(const void* p) {
  uint16_t r;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(r) : "l"(p) : "memory");
  return r;
}
// One element of type T; COHERENT selects an L2-only load over the read-only (nc) path.
template <bool COHERENT, typename T>
__device__ inline T ld_elem(const T* p) {
  if constexpr (!COHERENT) {
    return __ldg(p);
  } else if constexpr (sizeof(T) == 4) {
    const uint32_t u = ld_cg_u32(p);
    return *reinterpret_cast<const T*>(&u);
  } else {
    static_assert(sizeof(T) == 2, "2- or 4-byte elements");
    const uint16_t u = ld_cg_u16(p);
    return *reinterpret_cast<const T*>(&u);
  }
}
template <bool COHERENT>
__device__ inline uint4 ld_v4(const void* p) {
  if constexpr (COHERENT) return ld_cg_v4(p);
  else return ld_nc_v4(p);
}

}  // namespace moe
