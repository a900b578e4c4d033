// ckv_device.cuh -- device helpers shared by the CUDA kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ckv.h"

namespace ckv {

constexpr float kLog2e = 1.4426950408889634f;
// Finite stand-in for "no token yet" in a running max: differences of two
// sentinels are 0 (weight 1 times a zero sum), never NaN.
constexpr float kNegBig = -3.402823466e38f;

__device__ __forceinline__ void flag_error(int32_t* err, uint32_t bit) {
  if (err) atomicOr(reinterpret_cast<unsigned int*>(err), bit);
}

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// e^(a - b) for b >= a (both finite); the difference is formed first.
__device__ __forceinline__ float exp_diff(float a, float b) { return fast_exp2((a - b) * kLog2e); }

// ---- bf16 <-> fp32 (bf16 is the top half of an fp32 word) ----------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// ---- memory access with cache hints ---------------------------------------
// Streaming, read-only data (read once): do not allocate it in L1.
__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
  float4 v;
  asm("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}
// Read-only data shared by many CTAs (bias tables): normal caching.
__device__ __forceinline__ float4 ld_shared_ro_f4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

// ---- programmatic dependent launch ----------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Four consecutive channels of an input row, widened to fp32.
template <typename InT>
struct In4;
template <>
struct In4<float> {
  static __device__ __forceinline__ float4 load(const float* row, int c) {
    return ld_stream_f4(row + c);
  }
};
template <>
struct In4<__nv_bfloat16> {
  static __device__ __forceinline__ float4 load(const __nv_bfloat16* row, int c) {
    uint2 w = ld_stream_u2(row + c);
    return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
  }
};

__device__ __forceinline__ float get(const float4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__device__ __forceinline__ void set(float4& v, int i, float x) {
  if (i == 0) v.x = x;
  else if (i == 1) v.y = x;
  else if (i == 2) v.z = x;
  else v.w = x;
}

}  // namespace ckv
