// e4m3 "pieces" of fp32 values for the tensor-core decode operands.
//
// A value y (already scaled by a power of two sigma) is written as
// y ~= sum_i p_i 16^-i with p_i = rn_e4m3(r_i), r_0 = y, r_{i+1} = 16 (r_i - p_i):
// each piece carries about four more bits than the last, and every product
// p_i * (+-1) is exact in an fp8 MMA with fp32 accumulation.  Operand bytes
// are laid out along K in the order the sign-plane operand uses (k_position).
#pragma once

#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace tq {

// Position along K of coordinate (or token) i inside a 128-element block: the
// e4m3 operand byte built from bit i sits at 32 (i/32) + 4 (i%8) + (i%32)/8,
// because one 32-bit register is built from bits i, i+8, i+16, i+24 of a word.
__device__ __forceinline__ int k_position(int i) { return 32 * (i >> 5) + 4 * (i & 7) + ((i & 31) >> 3); }

__device__ __forceinline__ uint8_t to_e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float from_e4m3(uint8_t b) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

// The bit-plane operand stores bit i of a 32-bit word (coordinate or token i
// of a 32-element group) as an e4m3 byte that is 0 or a power of two beta_j,
// j = i % 8: bits 0-2 as the mantissa bits of a subnormal (2^-9, 2^-8, 2^-7),
// bits 3-7 moved down by three (2^-9, 2^-8, 2^-7, then the lowest two
// exponent bits: 2^-6, 2^-5).  The other operand carries 1 / beta_j; the
// classes span a factor of 16, so the pieces of every class keep their bits.
__host__ __device__ constexpr float bit_inv_scale(int j) {
  return (j & 7) == 0 || (j & 7) == 3 ? 512.f : (j & 7) == 1 || (j & 7) == 4 ? 256.f
       : (j & 7) == 2 || (j & 7) == 5 ? 128.f : (j & 7) == 6 ? 64.f : 32.f;
}
constexpr float kMaxBitInvScale = 512.f;

// Power of two sigma with sigma * maxabs <= 200 (so every piece stays below
// the format's 448 limit), 1 when maxabs is 0.
__device__ __forceinline__ float piece_scale(float maxabs) {
  if (!(maxabs > 0.f)) return 1.f;
  return exp2f(floorf(log2f(200.f / maxabs)));
}

// 16^-i for the piece index i (an exact power of two built from its exponent
// field, so no call is left for the compiler to make).
__device__ __forceinline__ float inv16_pow(int i) { return __int_as_float((127 - 4 * i) << 23); }

// Pieces of y into byte `kpos` of N consecutive 128-byte rows starting at `rows`.
template <int N>
__device__ __forceinline__ void write_pieces_rows(uint8_t* rows, int kpos, float y) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint8_t p = to_e4m3(y);
    rows[i * 128 + kpos] = p;
    y = (y - from_e4m3(p)) * 16.f;
  }
}

// As write_pieces_rows for two values at once (rows_a gets ya's pieces,
// rows_b yb's): one paired conversion, and the residual of both in one paired
// FMA and multiply (the same pieces, bit for bit).
template <int N>
__device__ __forceinline__ void write_pieces_rows2(uint8_t* rows_a, uint8_t* rows_b, int kpos, float ya, float yb) {
  float2 y = make_float2(ya, yb);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);   // (x in the low byte)
    rows_a[i * 128 + kpos] = static_cast<uint8_t>(p & 0xff);
    rows_b[i * 128 + kpos] = static_cast<uint8_t>(p >> 8);
    const float2 b = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(p, __NV_E4M3)));
    y = __fmul2_rn(__ffma2_rn(b, make_float2(-1.f, -1.f), y), make_float2(16.f, 16.f));
  }
}

}  // namespace tq
