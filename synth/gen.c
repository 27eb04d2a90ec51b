/*
 * Seeded synthetic inputs: counter-based normal and uniform draws.
 *
 * This file holds input generation only. It computes nothing of the decode
 * step itself; both the CUDA path and the CPU oracle receive what it writes.
 *
 * The generator's definition (SplitMix64 streams, Box-Muller normals, fp64 -> bf16
 * rounding) is stated in gen_core.h, which the device library gen_dev.cu shares.
 *
 * Built as a plain shared library (gcc -O2 -fopenmp -shared -fPIC); the
 * Python wrapper in this folder calls it through ctypes.
 */
#include "gen_core.h"

uint64_t synth_stream_key(uint64_t seed, uint64_t tid) { return sg_stream_key(seed, tid); }

uint64_t synth_draw(uint64_t key, uint64_t i) { return sg_draw(key, i); }

uint16_t synth_f64_to_bf16(double v) { return sg_f64_to_bf16(v); }

/* Standard normal draw number idx of stream key. */
double synth_normal_at(uint64_t key, uint64_t idx) {
  double z0, z1;
  sg_normal_pair(key, idx >> 1, &z0, &z1);
  return (idx & 1) ? z1 : z0;
}

/* out[i] = bf16(mean + std * z[start + i]) for i in [0, n). Each Box-Muller pair is evaluated
   once and gives both of its draws. */
void synth_normal_bf16(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n, double mean,
                       double std, uint16_t* out) {
  if (n == 0) return;
  const uint64_t key = synth_stream_key(seed, tid);
  const uint64_t p0 = start >> 1, p1 = (start + n - 1) >> 1;
#pragma omp parallel for schedule(static)
  for (long long q = 0; q <= (long long)(p1 - p0); ++q) {
    const uint64_t p = p0 + (uint64_t)q;
    double z0, z1;
    sg_normal_pair(key, p, &z0, &z1);
    if (2 * p >= start) out[2 * p - start] = sg_f64_to_bf16(mean + std * z0);
    if (2 * p + 1 < start + n) out[2 * p + 1 - start] = sg_f64_to_bf16(mean + std * z1);
  }
}

/* out[i] = mean + std * z[start + i] in fp64 (for inputs the method keeps in full precision). */
void synth_normal_f64(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n, double mean,
                      double std, double* out) {
  if (n == 0) return;
  const uint64_t key = synth_stream_key(seed, tid);
  const uint64_t p0 = start >> 1, p1 = (start + n - 1) >> 1;
#pragma omp parallel for schedule(static)
  for (long long q = 0; q <= (long long)(p1 - p0); ++q) {
    const uint64_t p = p0 + (uint64_t)q;
    double z0, z1;
    sg_normal_pair(key, p, &z0, &z1);
    if (2 * p >= start) out[2 * p - start] = mean + std * z0;
    if (2 * p + 1 < start + n) out[2 * p + 1 - start] = mean + std * z1;
  }
}

/* out[i] = B(K(seed, tid), start + i): raw 64-bit draws. */
void synth_bits(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n, uint64_t* out) {
  uint64_t key = synth_stream_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i) out[i] = synth_draw(key, start + (uint64_t)i);
}
