/*
 * Seeded synthetic inputs on the device: the generator of gen_core.h written straight into
 * device memory, for workloads whose weights are too large to draw on the host (the MoE
 * stack's 127 G expert weights). Same streams, same draws, same bf16 rounding as gen.c; only
 * ln / sqrt / cos / sin are CUDA's. Input generation only: nothing of the decode step.
 *
 * Built with nvcc -fmad=false so that mean + std * z rounds twice, as on the host.
 */
#include <cuda_runtime.h>

#include "gen_core.h"

namespace {

constexpr int kThreads = 256;

// One thread per Box-Muller pair p in [p0, p1] (grid-stride); both of its draws are written
// where they fall inside [start, start + n).
__global__ void __launch_bounds__(kThreads) normal_bf16_kernel(uint64_t key, uint64_t start, uint64_t n, double mean,
                                                              double stdv, uint64_t p0, uint64_t n_pairs,
                                                              uint16_t* __restrict__ out) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t q = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n_pairs; q += stride) {
    const uint64_t p = p0 + q;
    double z0, z1;
    sg_normal_pair(key, p, &z0, &z1);
    if (2 * p >= start) out[2 * p - start] = sg_f64_to_bf16(mean + stdv * z0);
    if (2 * p + 1 < start + n) out[2 * p + 1 - start] = sg_f64_to_bf16(mean + stdv * z1);
  }
}

}  // namespace

/* out_dev[i] = bf16(mean + std * z[start + i]) for i in [0, n), queued on `stream`
   (cudaStream_t; NULL: legacy default). Returns the launch's cudaError_t. */
extern "C" int synth_normal_bf16_dev(uint64_t seed, uint64_t tid, uint64_t start, uint64_t n, double mean, double stdv,
                                     void* out_dev, void* stream) {
  if (n == 0) return (int)cudaSuccess;
  if (!out_dev) return (int)cudaErrorInvalidValue;
  const uint64_t p0 = start >> 1, p1 = (start + n - 1) >> 1;
  const uint64_t n_pairs = p1 - p0 + 1;
  uint64_t blocks = (n_pairs + kThreads - 1) / kThreads;
  if (blocks > 65536) blocks = 65536;
  normal_bf16_kernel<<<(unsigned)blocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      sg_stream_key(seed, tid), start, n, mean, stdv, p0, n_pairs, static_cast<uint16_t*>(out_dev));
  return (int)cudaGetLastError();
}
