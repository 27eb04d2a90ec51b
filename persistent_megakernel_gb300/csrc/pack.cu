// Device packer: the host packer's layouts written by a kernel, for weights too large to stage
// through host memory (the MoE stack's 67 GB of MXFP4 experts). The encoders are quant.h's,
// the ones the host packer runs, so both give the same bytes.
//
// One warp per output row (grid-stride). FP8 rows: the warp reduces the row's largest
// magnitude, then every lane encodes a strided share of the row. MXFP4 rows: every lane owns
// whole 32-weight blocks (64 B in, 16 B of codes + 1 scale byte out).
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/dec.h"
#include "quant.h"

namespace decimpl {
namespace {

constexpr int kPackThreads = 256;

__global__ void __launch_bounds__(kPackThreads) pack_rows_kernel(int dtype, const uint16_t* __restrict__ a,
                                                                 const uint16_t* __restrict__ b, int rows, int cols,
                                                                 uint8_t* __restrict__ vals,
                                                                 uint8_t* __restrict__ scales) {
  const int lane = (int)(threadIdx.x & 31u);
  const long long n_out = (long long)rows * (b ? 2 : 1);
  const long long n_warps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long orow = (((long long)blockIdx.x * blockDim.x) + threadIdx.x) >> 5; orow < n_out; orow += n_warps) {
    // pair mode: output row 2r is a's row r, 2r + 1 is b's row r
    const uint16_t* src = b ? (((orow & 1) ? b : a) + (size_t)(orow >> 1) * cols) : (a + (size_t)orow * cols);
    if (dtype == DEC_BF16) {
      uint16_t* dst = reinterpret_cast<uint16_t*>(vals) + (size_t)orow * cols;
      for (int j = 8 * lane; j < cols; j += 8 * 32)  // cols % 8 == 0: 16-byte chunks
        *reinterpret_cast<uint4*>(dst + j) = *reinterpret_cast<const uint4*>(src + j);
    } else if (dtype == DEC_FP8_E4M3_ROWSCALE) {
      uint32_t am = 0;
      for (int j = lane; j < cols; j += 32) {
        const uint32_t x = src[j] & 0x7FFFu;
        if (x > am && x <= 0x7F80u) am = x;  // NaNs skipped, as the host packer does
      }
      am = __reduce_max_sync(0xffffffffu, am);
      const float s = decq::fp8_row_scale(decq::bf16_to_f32((uint16_t)am));
      uint8_t* dst = vals + (size_t)orow * cols;
      for (int j = lane; j < cols; j += 32) dst[j] = decq::fp8_code(src[j], s);
      if (lane == 0) reinterpret_cast<float*>(scales)[orow] = s;
    } else {
      uint8_t* dv = vals + (size_t)orow * (cols / 2);
      uint8_t* ds = scales + (size_t)orow * (cols / 32);
      for (int blk = lane; blk < cols / 32; blk += 32) {
        uint16_t v[32];
        const uint4* x = reinterpret_cast<const uint4*>(src + 32 * blk);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 c = x[q];
          const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            v[8 * q + 2 * h] = (uint16_t)(w[h] & 0xFFFFu);
            v[8 * q + 2 * h + 1] = (uint16_t)(w[h] >> 16);
          }
        }
        const int e = decq::mxfp4_block_exponent(v);
        uint32_t out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t word = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int i = 8 * q + 2 * k;  // byte k of word q holds elements i (low nibble), i + 1
            const uint32_t byte = decq::mxfp4_code(v[i], e) | (decq::mxfp4_code(v[i + 1], e) << 4);
            word |= byte << (8 * k);
          }
          out[q] = word;
        }
        *reinterpret_cast<uint4*>(dv + 16 * blk) = make_uint4(out[0], out[1], out[2], out[3]);
        ds[blk] = (uint8_t)e;
      }
    }
  }
}

// FP8 KV-cache entries: out[i] = e4m3fn(v[i] / s), the host packer's encoder.
__global__ void __launch_bounds__(kPackThreads) pack_kv_fp8_kernel(const uint16_t* __restrict__ v, size_t n, float s,
                                                                   uint8_t* __restrict__ out) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) out[i] = decq::fp8_code(v[i], s);
}

}  // namespace
}  // namespace decimpl

extern "C" cudaError_t dec_launch_pack_kv_fp8(const uint16_t* v, size_t n, float s, uint8_t* out, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  size_t blocks = (n + decimpl::kPackThreads - 1) / decimpl::kPackThreads;
  if (blocks > 8192) blocks = 8192;
  decimpl::pack_kv_fp8_kernel<<<(unsigned)blocks, decimpl::kPackThreads, 0, stream>>>(v, n, s, out);
  return cudaGetLastError();
}

// Queue the packing kernel (arguments already validated by the caller).
extern "C" cudaError_t dec_launch_pack(int dtype, const uint16_t* a, const uint16_t* b, int rows, int cols,
                                       void* vals, void* scales, cudaStream_t stream) {
  const long long n_out = (long long)rows * (b ? 2 : 1);
  if (n_out == 0) return cudaSuccess;
  const long long warps_per_block = decimpl::kPackThreads / 32;
  long long blocks = (n_out + warps_per_block - 1) / warps_per_block;
  if (blocks > 8192) blocks = 8192;
  decimpl::pack_rows_kernel<<<(unsigned)blocks, decimpl::kPackThreads, 0, stream>>>(
      dtype, a, b, rows, cols, static_cast<uint8_t*>(vals), static_cast<uint8_t*>(scales));
  return cudaGetLastError();
}
