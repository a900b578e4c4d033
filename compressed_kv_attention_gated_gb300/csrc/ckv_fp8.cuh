// ckv_fp8.cuh -- the pooled path's output stage for one 128-channel vector
// held by a warp (lane l owns channels 4l..4l+3): bf16 rounding, the
// Hadamard-128 rotation, bf16 rounding, absmax FP8-e4m3 quantisation (vLLM
// page "vllm.models.glm5next.amd.ops.kpool_compress",
// _kpool_softmax_rotate_write_cache_kernel), and the paged FP8 cache store.
#pragma once

#include <cstdint>

#include "ckv_device.cuh"

namespace ckv {

// Largest of the 32 lanes' non-negative values in one warp reduction: a
// non-negative float orders like its bit pattern, so the unsigned max of the
// bits is the float max (exact).  A NaN counts as 0, as fmaxf ignores it.
__device__ __forceinline__ float warp_absmax(float am) {
  uint32_t u = __float_as_uint(am);
  u = u > 0x7F800000u ? 0u : u;
  return __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, u));
}

// x (fp32) -> bf16 -> Hadamard-128 (fp32) -> bf16 -> absmax FP8-e4m3 + scale.
// The rotation is the orthonormal Sylvester Hadamard matrix: butterfly spans
// 1, 2, 4, ..., 64 in ascending order, each (u + v, u - v) in fp32, then one
// multiply by fp32(1/sqrt(128)).
template <bool kRound>
__device__ __forceinline__ void rotate_quantize(const float (&x)[4], int lane, uint32_t& codes,
                                                float& scale, float (&xb)[4], float (&yb)[4]) {
  float a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    xb[i] = round_bf16(x[i]);
    a[i] = xb[i];
  }
  {  // span 1: channel pairs (0,1), (2,3) of the lane
    const float u0 = a[0], v0 = a[1], u1 = a[2], v1 = a[3];
    a[0] = u0 + v0;
    a[1] = u0 - v0;
    a[2] = u1 + v1;
    a[3] = u1 - v1;
  }
  {  // span 2: pairs (0,2), (1,3)
    const float u0 = a[0], v0 = a[2], u1 = a[1], v1 = a[3];
    a[0] = u0 + v0;
    a[2] = u0 - v0;
    a[1] = u1 + v1;
    a[3] = u1 - v1;
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {  // spans 4, 8, 16, 32, 64: partner lane l ^ m
    // lower lane: a + o; upper lane: o - a.  fma(a, -1, o) rounds o - a once,
    // exactly like a subtraction, so one FMA serves both halves.
    const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float o = __shfl_xor_sync(0xFFFFFFFFu, a[i], m);
      a[i] = fmaf(a[i], sgn, o);
    }
  }
  const float c = __uint_as_float(0x3DB504F3u);  // fp32(1/sqrt(128))
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    yb[i] = round_bf16(a[i] * c);
    am = fmaxf(am, fabsf(yb[i]));
  }
  am = warp_absmax(am);
  am = fmaxf(am, 1e-4f);
  const float v = am * __uint_as_float(0x3B124925u);  // absmax * fp32(1/448)
  float q[4];
  if (kRound) {
    // smallest power of two >= v (v is a positive normal number); dividing by a
    // power of two is exact, so multiplying by its (exact) reciprocal is the same
    // IEEE quotient
    const uint32_t bits = __float_as_uint(v);
    const uint32_t e = (bits & 0x007FFFFFu) ? (bits & 0x7F800000u) + 0x00800000u : (bits & 0x7F800000u);
    scale = __uint_as_float(e);
    const float inv = __uint_as_float((254u << 23) - e);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = fminf(fmaxf(yb[i] * inv, -448.f), 448.f);
  } else {
    scale = v;
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = fminf(fmaxf(__fdiv_rn(yb[i], scale), -448.f), 448.f);
  }
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(q[0], q[1]), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(q[2], q[3]), __NV_SATFINITE, __NV_E4M3);
  codes = (lo & 0xFFFFu) | (hi << 16);
}

// Paged FP8 cache whose rows hold `blocks` 128-channel blocks: per page,
// page_size rows of 128 * blocks FP8 bytes, then page_size * blocks fp32
// scales (scale of block j of row r at r * blocks + j).  With blocks == 1 this
// is the pooled cache layout.  Stores block j of the row at location loc
// (lane l: the codes of channels 4l..4l+3; lane 0: the scale).
__device__ __forceinline__ void cache_write_block(uint8_t* cache, int64_t page_size, int64_t loc, int blocks,
                                                  int j, int lane, uint32_t codes, float scale) {
  const int64_t row_bytes = 128 * static_cast<int64_t>(blocks);
  const int64_t page = loc / page_size, tok = loc - page * page_size;
  uint8_t* base = cache + page * page_size * (row_bytes + 4 * blocks);
  reinterpret_cast<uint32_t*>(base + tok * row_bytes + 128 * j)[lane] = codes;
  if (lane == 0) reinterpret_cast<float*>(base + page_size * row_bytes)[tok * blocks + j] = scale;
}

// One warp stores block j of an fp32 row into the paged FP8 cache (bf16 ->
// Hadamard-128 -> bf16 -> absmax FP8, one scale per block); lane l passes
// channels 4l..4l+3 of the block.
__device__ __forceinline__ void fp8_block_store(float4 v, uint8_t* cache, int64_t page_size, int64_t loc,
                                                int blocks, int j, int lane, bool round_scale) {
  const float x[4] = {v.x, v.y, v.z, v.w};
  float xb[4], yb[4], scale;
  uint32_t codes;
  if (round_scale) rotate_quantize<true>(x, lane, codes, scale, xb, yb);
  else rotate_quantize<false>(x, lane, codes, scale, xb, yb);
  cache_write_block(cache, page_size, loc, blocks, j, lane, codes, scale);
}

// The same for a row staged in memory (128 channels from row128).
__device__ __forceinline__ void fp8_block_store(const float* row128, uint8_t* cache, int64_t page_size,
                                                int64_t loc, int blocks, int j, int lane, bool round_scale) {
  fp8_block_store(*reinterpret_cast<const float4*>(row128 + 4 * lane), cache, page_size, loc, blocks, j, lane,
                  round_scale);
}

}  // namespace ckv
