// PolarQuant record helpers shared by the quantize kernels (polar.cu and the
// tile quantizer's PolarQuant epilogue).  The intelliparadigm.com page,
// §2.1.1 step 2: pairs become (radius, angle), the angle is rounded to a
// multiple of pi/12.  Record of a head vector (64 bytes, one little-endian
// bit stream): the 64 level-1 codes (0..23) x 5 bits, then the 63 codes of
// levels 2..7 (0..6) x 3 bits.
#pragma once

#include <cstdint>

namespace tq {

constexpr int kPolarRecordWords = 16;       // 64-byte record
constexpr int kPolarUpperBit = 320;         // first bit of the level-2..7 codes

// Index of the first level-L code (L = 2..7) among the 63 upper codes.
__host__ __device__ constexpr int polar_upper_offset(int level) { return 64 - (128 >> (level - 1)); }

// Rounded multiple of pi/12 of the angle of (first, second); level 1 angles
// span (-pi, pi] and are taken modulo 24, upper levels lie in [0, pi/2].
__device__ __forceinline__ int polar_angle_code(float second, float first, bool level1) {
  const int k = __float2int_rn(atan2f(second, first) * 3.8197186342054881f);   // (times 12/pi, half to even)
  return level1 ? (k + 24) % 24 : k;
}

// Word wd (bits 32 wd .. 32 wd + 31) of a record from its codes: c1 the 64
// level-1 codes, cu the 63 upper codes (bytes).  Every code whose bits
// overlap the word is ORed in (a code cut by the word's first bit contributes
// its top bits).
__device__ __forceinline__ uint32_t polar_record_word(const uint8_t* c1, const uint8_t* cu, int wd) {
  const int lo = 32 * wd;
  uint32_t word = 0;
  for (int c = lo / 5; c < 64 && 5 * c < lo + 32; ++c) {
    const int sh = 5 * c - lo;
    const uint32_t code = c1[c];
    word |= sh >= 0 ? code << sh : code >> -sh;
  }
  for (int k = lo > kPolarUpperBit ? (lo - kPolarUpperBit) / 3 : 0; k < 63 && kPolarUpperBit + 3 * k < lo + 32; ++k) {
    const int sh = kPolarUpperBit + 3 * k - lo;
    const uint32_t code = cu[k];
    word |= sh >= 0 ? code << sh : code >> -sh;
  }
  return word;
}

}  // namespace tq
