// Host weight packer: bf16 matrices -> the layouts the megakernel streams.
//
// FP8: dynamic per-row e4m3fn quantisation of a bf16 matrix (Ling-3.0-flash on DGX Spark,
// section "optimisation 2: online FP8 LM head": the bf16 head is quantised at load time,
// halving its read). MXFP4: OCP Microscaling v1.0 FP4 (e2m1) elements with one E8M0 scale per
// 32 weights of a row (the MXFP4 experts of the same article, "optimisation 1"). The encoders
// (quant.h) are the ones the device packer (pack.cu) runs, so both give the same bytes.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/dec.h"
#include "quant.h"

namespace {

void pack_fp8_row(const uint16_t* w, int cols, uint8_t* codes, float* scale) {
  const float s = decq::fp8_row_scale(decq::bf16_to_f32(decq::amax_bits(w, cols)));
  *scale = s;
  for (int j = 0; j < cols; ++j) codes[j] = decq::fp8_code(w[j], s);
}

void pack_mxfp4_row(const uint16_t* w, int cols, uint8_t* codes, uint8_t* scales) {
  for (int b = 0; b < cols / 32; ++b) {
    const uint16_t* blk = w + 32 * b;
    const int e = decq::mxfp4_block_exponent(blk);
    scales[b] = (uint8_t)e;
    for (int i = 0; i < 32; i += 2)
      codes[(32 * b + i) / 2] = (uint8_t)(decq::mxfp4_code(blk[i], e) | (decq::mxfp4_code(blk[i + 1], e) << 4));
  }
}

dec_status check(dec_dtype dt, int rows, int cols) {
  if (rows < 0 || cols <= 0) return DEC_ERR_SHAPE;
  if (dt == DEC_BF16) return cols % 8 ? DEC_ERR_SHAPE : DEC_OK;
  if (dt == DEC_FP8_E4M3_ROWSCALE) return cols % 16 ? DEC_ERR_SHAPE : DEC_OK;
  if (dt == DEC_MXFP4) return cols % 32 ? DEC_ERR_SHAPE : DEC_OK;
  return DEC_ERR_DTYPE;
}

void pack_row(dec_dtype dt, const uint16_t* w, int r, int cols, void* out_values, void* out_scales, int out_row) {
  if (dt == DEC_BF16) {
    std::memcpy(static_cast<uint16_t*>(out_values) + (size_t)out_row * cols, w + (size_t)r * cols, (size_t)cols * 2);
  } else if (dt == DEC_FP8_E4M3_ROWSCALE) {
    pack_fp8_row(w + (size_t)r * cols, cols, static_cast<uint8_t*>(out_values) + (size_t)out_row * cols,
                 static_cast<float*>(out_scales) + out_row);
  } else {
    pack_mxfp4_row(w + (size_t)r * cols, cols, static_cast<uint8_t*>(out_values) + (size_t)out_row * (cols / 2),
                   static_cast<uint8_t*>(out_scales) + (size_t)out_row * (cols / 32));
  }
}

}  // namespace

extern "C" {

dec_status dec_packed_bytes(dec_dtype dtype, int rows, int cols, size_t* values_bytes, size_t* scales_bytes) {
  const dec_status st = check(dtype, rows, cols);
  if (st != DEC_OK) return st;
  size_t v = 0, s = 0;
  if (dtype == DEC_BF16) v = (size_t)rows * cols * 2;
  if (dtype == DEC_FP8_E4M3_ROWSCALE) { v = (size_t)rows * cols; s = (size_t)rows * 4; }
  if (dtype == DEC_MXFP4) { v = (size_t)rows * cols / 2; s = (size_t)rows * cols / 32; }
  if (values_bytes) *values_bytes = v;
  if (scales_bytes) *scales_bytes = s;
  return DEC_OK;
}

dec_status dec_pack(dec_dtype dtype, const uint16_t* w, int rows, int cols, void* out_values, void* out_scales) {
  const dec_status st = check(dtype, rows, cols);
  if (st != DEC_OK) return st;
  if (!w || !out_values || (dtype != DEC_BF16 && !out_scales)) return DEC_ERR_INVALID_ARG;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) pack_row(dtype, w, r, cols, out_values, out_scales, r);
  return DEC_OK;
}

dec_status dec_pack_pair(dec_dtype dtype, const uint16_t* a, const uint16_t* b, int rows, int cols, void* out_values,
                         void* out_scales) {
  const dec_status st = check(dtype, rows, cols);
  if (st != DEC_OK) return st;
  if (!a || !b || !out_values || (dtype != DEC_BF16 && !out_scales)) return DEC_ERR_INVALID_ARG;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    pack_row(dtype, a, r, cols, out_values, out_scales, 2 * r);
    pack_row(dtype, b, r, cols, out_values, out_scales, 2 * r + 1);
  }
  return DEC_OK;
}

dec_status dec_pack_kv_fp8(const uint16_t* v, size_t n, float scale, uint8_t* out) {
  if (n && (!v || !out)) return DEC_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return DEC_ERR_INVALID_ARG;
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i) out[i] = decq::fp8_code(v[i], scale);
  return DEC_OK;
}

}  // extern "C"
