// Weight quantisers shared by the host packer (packer.cpp) and the device packer (pack.cu).
//
// FP8: e4m3fn codes of a row divided by its scale s = amax / 448 (Ling-3.0-flash on DGX Spark,
// section "optimisation 2: online FP8 LM head": the bf16 head is quantised at load time).
// MXFP4: OCP Microscaling v1.0 FP4 (e2m1) elements, one E8M0 scale per 32 weights of a row, the
// scale exponent floor(log2 amax) - 2 (emax of e2m1 is 2). Both round to nearest with ties to
// the even code and saturate to the largest finite code. Every decision is taken on integer
// bits or in exact / correctly rounded IEEE arithmetic, so the host and the device give the same
// bytes.
#pragma once

#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#define DECQ_HD __host__ __device__ __forceinline__
#else
#define DECQ_HD inline
#endif

namespace decq {

DECQ_HD uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

DECQ_HD float bf16_to_f32(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

// Round the integer sig * 2^-shift to nearest, ties to even (shift in [1, 63]).
DECQ_HD uint64_t rne_shift(uint64_t sig, int shift) {
  const uint64_t q = sig >> shift;
  const uint64_t rem = sig & ((1ull << shift) - 1ull);
  const uint64_t half = 1ull << (shift - 1);
  return (rem > half || (rem == half && (q & 1ull))) ? q + 1ull : q;
}

// e4m3fn magnitude code of y (y >= 0 or NaN-free), ties to even, saturated to 448 (0x7E).
// e4m3fn: exponent bias 7, 3 mantissa bits, subnormals in units of 2^-9, no infinities.
DECQ_HD uint8_t e4m3_magnitude(float y) {
  if (!(y > 0.f)) return 0;
  if (y >= 448.f) return 0x7E;
  const uint32_t u = f32_bits(y);
  const int ef = (int)((u >> 23) & 0xFF);
  if (ef == 0) return 0;  // below 2^-126: far under half of the smallest subnormal 2^-9
  const int E = ef - 127;                                  // y = sig * 2^(E - 23)
  const uint64_t sig = (uint64_t)((u & 0x7FFFFFu) | 0x800000u);
  if (E < -6) {
    // subnormal: the code is round(y / 2^-9) = round(sig * 2^(E - 14)); 8 is the smallest normal
    const int shift = 14 - E;  // > 20
    if (shift > 40) return 0;
    return (uint8_t)rne_shift(sig, shift);
  }
  uint64_t q = rne_shift(sig, 20);  // 1.mmm with 3 mantissa bits: q in [8, 16]
  int e = E;
  if (q == 16) {
    q = 8;
    ++e;
  }
  const int code = ((e + 7) << 3) | (int)(q & 7u);
  return (uint8_t)(code > 0x7E ? 0x7E : code);
}

// e2m1 magnitude code of a (a >= 0): nearest of {0, .5, 1, 1.5, 2, 3, 4, 6}; a tie goes to the
// even code; values above 6 saturate.
DECQ_HD uint8_t e2m1_magnitude(double a) {
  if (a <= 0.25) return 0;
  if (a < 0.75) return 1;
  if (a <= 1.25) return 2;
  if (a < 1.75) return 3;
  if (a <= 2.5) return 4;
  if (a < 3.5) return 5;
  if (a <= 5.0) return 6;
  return 7;
}

// 2^k as a double, k in [-1022, 1023] (exact, built from the exponent bits).
DECQ_HD double pow2_f64(int k) {
  const uint64_t b = (uint64_t)(k + 1023) << 52;
  double d;
  memcpy(&d, &b, 8);
  return d;
}

// floor(log2 |v|) of a non-zero bf16 value, exactly, from its bits.
DECQ_HD int bf16_floor_log2(uint16_t b) {
  const int ex = (b >> 7) & 0xFF;
  const int m = b & 0x7F;
  if (ex) return ex - 127;
  int hb = 6;  // subnormal: value = m * 2^-133
  while (hb > 0 && !(m >> hb)) --hb;
  return hb - 133;
}

// Largest magnitude of n bf16 values, as bf16 bits (magnitudes order like their bit patterns;
// NaNs are skipped).
DECQ_HD uint16_t amax_bits(const uint16_t* v, int n) {
  uint16_t amax = 0;
  for (int i = 0; i < n; ++i) {
    const uint16_t a = (uint16_t)(v[i] & 0x7FFFu);
    if (a > amax && a <= 0x7F80u) amax = a;
  }
  return amax;
}

// E8M0 exponent of one block of 32 bf16 weights: clamp(floor(log2 amax) - 2 + 127, 0, 254);
// an all-zero block takes 0.
DECQ_HD int mxfp4_block_exponent(const uint16_t* blk) {
  const uint16_t amax = amax_bits(blk, 32);
  if (amax == 0) return 0;
  int e = bf16_floor_log2(amax) - 2 + 127;
  return e < 0 ? 0 : (e > 254 ? 254 : e);
}

// e2m1 code (sign in bit 3) of one bf16 weight under block exponent e: |v| / 2^(e - 127) is
// exact in double.
DECQ_HD uint8_t mxfp4_code(uint16_t v, int e) {
  const double y = (double)bf16_to_f32((uint16_t)(v & 0x7FFFu)) * pow2_f64(127 - e);
  return (uint8_t)(e2m1_magnitude(y) | ((v & 0x8000u) ? 0x8 : 0));
}

// Row scale of the FP8 encoding: amax / 448 in correctly rounded fp32; an all-zero row takes 1.
DECQ_HD float fp8_row_scale(float amax) { return amax > 0.f ? amax / 448.0f : 1.0f; }

// e4m3fn code (sign in bit 7) of one bf16 weight of a row with scale s: v / s in correctly
// rounded fp32.
DECQ_HD uint8_t fp8_code(uint16_t v, float s) {
  const float y = bf16_to_f32((uint16_t)(v & 0x7FFFu)) / s;
  return (uint8_t)(e4m3_magnitude(y) | ((v & 0x8000u) ? 0x80 : 0));
}

}  // namespace decq
