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
// Block-scale layout of every MXFP8 operand: "atoms" of 512 bytes, one per 128 operand rows (or
// columns, MN-major) and 128-element K block, each in the order in which tcgen05.cp.32x128b.warpx4
// moves it to TMEM for the MMA (row r of the 128 at byte 16 (r mod 32) + 4 (r / 32), the four
// 32-element sub-blocks of the K block in its four bytes). A GEMM stage then loads each operand's
// scales with one 512-byte bulk copy.
// K-major operand whose 128-row tiles start at multiples of 128 (the packed weights): byte of
// (row, 32-block b) for reduction length K.
__host__ __device__ __forceinline__ long atom_k(long row, long b, long K) {
  return (((row >> 7) * (K >> 7) + (b >> 2)) << 9) + ((row & 31) << 4) + (((row >> 5) & 3) << 2) + (b & 3);
}
// K-major operand in 128-row tiles numbered mt (the expert-sorted activations: tile mt of expert e
// covers its rows m*128 .. m*128+127, mt = tile prefix of e + m): byte of (tile mt, row r < 128, b).
__host__ __device__ __forceinline__ long atom_tile(long mt, int r, long b, long K) {
  return ((mt * (K >> 7) + (b >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (b & 3);
}
// MN-major operand [Krows][W] quantised along Krows in 32-row blocks rb: byte of (rb, column c).
__host__ __device__ __forceinline__ long atom_mn(long rb, long c, long W) {
  return (((rb >> 2) * (W >> 7) + (c >> 7)) << 9) + ((c & 31) << 4) + (((c >> 5) & 3) << 2) + (rb & 3);
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
