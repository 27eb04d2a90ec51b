/*
 * The counter-based generator's definition, shared by the host library (gen.c, C11) and the
 * device library (gen_dev.cu, CUDA). Input generation only: nothing of the decode step.
 *
 *   SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *   generators", OOPSLA 2014): gamma = 0x9E3779B97F4A7C15 and the 64-bit
 *   finaliser mix64(z) = z3 where z1 = (z ^ z>>30) * 0xBF58476D1CE4E5B9,
 *   z2 = (z1 ^ z1>>27) * 0x94D049BB133111EB, z3 = z2 ^ z2>>31.
 *   stream key   K(seed, tid) = mix64(mix64(seed + gamma) ^ tid)
 *   i-th draw    B(K, i)      = mix64(K + (i + 1) * gamma)       (mod 2^64)
 *   Box-Muller (Box & Muller 1958) on draws 2p and 2p+1:
 *     u1 = ((B(K,2p)   >> 11) + 1) * 2^-53   in (0, 1]
 *     u2 =  (B(K,2p+1) >> 11)      * 2^-53   in [0, 1)
 *     r  = sqrt(-2 ln u1);  z[2p] = r cos(2 pi u2);  z[2p+1] = r sin(2 pi u2)
 *   value = mean + std * z  (fp64, no fused multiply-add), then rounded to bfloat16 with
 *   round-to-nearest-even directly from the fp64 bits (no fp32 step).
 *
 * ln, sqrt, cos and sin are the platform's: libm on the host, CUDA's on the device. They may
 * differ in the last bits of a double, which changes a bf16 result only when the value lies
 * within a few ulps of a rounding midpoint (odds of order 1e-13 per value).
 */
#ifndef SYNTH_GEN_CORE_H
#define SYNTH_GEN_CORE_H

#include <math.h>
#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define SYNTH_HD static __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

#define SM_GAMMA 0x9E3779B97F4A7C15ULL

SYNTH_HD uint64_t sg_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SYNTH_HD uint64_t sg_stream_key(uint64_t seed, uint64_t tid) { return sg_mix64(sg_mix64(seed + SM_GAMMA) ^ tid); }

SYNTH_HD uint64_t sg_draw(uint64_t key, uint64_t i) { return sg_mix64(key + (i + 1) * SM_GAMMA); }

/* Round an IEEE double to bfloat16 bits, nearest-even, NaN kept quiet. */
SYNTH_HD uint16_t sg_f64_to_bf16(double v) {
  uint64_t b;
  memcpy(&b, &v, 8);
  uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
  uint64_t mag = b & 0x7FFFFFFFFFFFFFFFULL;
  if (mag > 0x7FF0000000000000ULL) return (uint16_t)(sign | 0x7FC0u); /* NaN */
  if (mag == 0x7FF0000000000000ULL) return (uint16_t)(sign | 0x7F80u); /* inf */
  int e = (int)(mag >> 52);           /* biased fp64 exponent */
  uint64_t m = mag & ((1ULL << 52) - 1);
  int E = e - 1023;                   /* unbiased */
  /* bf16: 8 exponent bits (bias 127), 7 mantissa bits, subnormals below 2^-126 */
  if (e == 0) return sign;            /* fp64 subnormals are far below bf16's range */
  uint64_t sig = m | (1ULL << 52);    /* 53-bit significand, value = sig * 2^(E-52) */
  int shift;                          /* bits to drop from sig */
  uint32_t out_exp;
  if (E >= -126) {
    shift = 52 - 7;
    out_exp = (uint32_t)(E + 127);
  } else {
    /* subnormal bf16: value = q * 2^-133, q = sig * 2^(E-52+133) */
    shift = 52 - 7 + (-126 - E);
    out_exp = 0;
    if (shift > 60) return sign;
  }
  uint64_t q = sig >> shift;
  uint64_t rem = sig & ((1ULL << shift) - 1);
  uint64_t half = 1ULL << (shift - 1);
  if (rem > half || (rem == half && (q & 1))) q += 1;
  uint32_t bits;
  if (out_exp == 0) {
    bits = (uint32_t)q; /* q <= 2^7; q == 2^7 carries into the smallest normal */
  } else {
    /* q in [2^7, 2^8]; a carry to 2^8 bumps the exponent */
    if (q == (1ULL << 8)) { q >>= 1; out_exp += 1; }
    if (out_exp >= 255) return (uint16_t)(sign | 0x7F80u);
    bits = (out_exp << 7) | (uint32_t)(q & 0x7F);
  }
  return (uint16_t)(sign | bits);
}

SYNTH_HD double sg_unit_open0(uint64_t bits) { return (double)((bits >> 11) + 1) * 0x1.0p-53; }
SYNTH_HD double sg_unit_closed0(uint64_t bits) { return (double)(bits >> 11) * 0x1.0p-53; }

/* Both normals of Box-Muller pair p of stream key: z[2p] (cos) and z[2p+1] (sin). */
SYNTH_HD void sg_normal_pair(uint64_t key, uint64_t p, double* z_even, double* z_odd) {
  double u1 = sg_unit_open0(sg_draw(key, 2 * p));
  double u2 = sg_unit_closed0(sg_draw(key, 2 * p + 1));
  double r = sqrt(-2.0 * log(u1));
  double a = 6.283185307179586476925286766559 * u2;
  *z_even = r * cos(a);
  *z_odd = r * sin(a);
}

#endif /* SYNTH_GEN_CORE_H */
