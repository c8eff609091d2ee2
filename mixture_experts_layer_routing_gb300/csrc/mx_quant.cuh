// OCP MX v1.0 quantiser for E4M3 elements with one E8M0 scale per 32 values,
// shared by the MXFP8 GEMM path and the MXFP8 decode kernels.
//   scale exponent X = floor(log2(amax of the block)) - 8 (E4M3's largest
//   exponent), clamped to [-127, 127], stored as X + 127; elements are
//   round-to-nearest-even E4M3 of v * 2^-X, saturated at +-448.
#pragma once
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ int mx_exponent(float amax) {
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xff);
  if (e == 0) return -127;                       // zero or below the normal range
  const int X = e - 127 - 8;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}
// 32 values -> 32 E4M3 codes (two uint4) and the E8M0 byte.
__device__ __forceinline__ uint8_t quant32(const float* v, uint4& lo, uint4& hi) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int X = mx_exponent(amax);
  const float inv = __uint_as_float((uint32_t)(127 - X) << 23);   // 2^-X, X <= 126 for finite bf16 input
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i] * inv, v[4 * i + 1] * inv), __NV_SATFINITE,
                                                 __NV_E4M3);
    const uint32_t b = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i + 2] * inv, v[4 * i + 3] * inv), __NV_SATFINITE,
                                                 __NV_E4M3);
    w[i] = a | (b << 16);
  }
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
  return (uint8_t)(X + 127);
}


}  // namespace
}  // namespace moe
