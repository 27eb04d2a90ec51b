// Host weight packer: bf16 matrices -> the layouts the megakernel streams.
//
// FP8: dynamic per-row e4m3fn quantisation of a bf16 matrix (Ling-3.0-flash on DGX Spark,
// section "optimisation 2: online FP8 LM head": the bf16 head is quantised at load time,
// halving its read). MXFP4: OCP Microscaling v1.0 FP4 (e2m1) elements with one E8M0 scale per
// 32 weights of a row (the MXFP4 experts of the same article, "optimisation 1"). Both
// encoders round to nearest, ties to the even code, and saturate to the largest finite value;
// every decision is taken in exact arithmetic or in correctly rounded IEEE fp32.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/dec.h"

namespace {

float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// e4m3fn code of |y| (y finite, >= 0), round half to even, saturated to 448.
uint8_t e4m3_magnitude(float y) {
  if (!(y > 0.f)) return 0;
  if (y >= 448.f) return 0x7E;
  int e;
  std::frexp(y, &e);  // y = f * 2^e, f in [0.5, 1): floor(log2 y) = e - 1
  int E = e - 1;
  if (E < -6) {       // subnormal range: units of 2^-9
    const float q = std::nearbyint(std::ldexp(y, 9));  // exact scaling, ties to even
    return (uint8_t)q;  // q == 8 is the smallest normal 2^-6, code 0x08
  }
  // normal: y = 2^E * (1 + m/8)
  float q = std::nearbyint((std::ldexp(y, -E) - 1.0f) * 8.0f);  // exact: y / 2^E in [1, 2)
  if (q == 8.f) {
    q = 0.f;
    ++E;
  }
  const int code = ((E + 7) << 3) | (int)q;
  return code > 0x7E ? 0x7E : (uint8_t)code;
}

// e2m1 code of |a| (a finite, >= 0): nearest of {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the
// even code, saturated to 6.
uint8_t e2m1_magnitude(double a) {
  if (a <= 0.25) return 0;
  if (a < 0.75) return 1;
  if (a <= 1.25) return 2;
  if (a < 1.75) return 3;
  if (a <= 2.5) return 4;
  if (a < 3.5) return 5;
  if (a <= 5.0) return 6;
  return 7;
}

// floor(log2 |v|) of a non-zero bf16 value, exactly, from its bits.
int bf16_floor_log2(uint16_t b) {
  const int ex = (b >> 7) & 0xFF;
  const int m = b & 0x7F;
  if (ex) return ex - 127;
  int hb = 6;  // subnormal: value = m * 2^-133
  while (!(m >> hb)) --hb;
  return hb - 133;
}

void pack_fp8_row(const uint16_t* w, int cols, uint8_t* codes, float* scale) {
  float amax = 0.f;
  for (int j = 0; j < cols; ++j) amax = std::fmax(amax, std::fabs(bf16_to_f32(w[j])));
  const float s = amax > 0.f ? amax / 448.0f : 1.0f;
  *scale = s;
  for (int j = 0; j < cols; ++j) {
    const float v = bf16_to_f32(w[j]);
    const float y = v / s;  // correctly rounded fp32 division
    codes[j] = (uint8_t)(e4m3_magnitude(std::fabs(y)) | (std::signbit(v) ? 0x80 : 0));
  }
}

void pack_mxfp4_row(const uint16_t* w, int cols, uint8_t* codes, uint8_t* scales) {
  for (int b = 0; b < cols / 32; ++b) {
    const uint16_t* blk = w + 32 * b;
    uint16_t amax_bits = 0;
    float amax = 0.f;
    for (int i = 0; i < 32; ++i) {
      const float a = std::fabs(bf16_to_f32(blk[i]));
      if (a > amax) {
        amax = a;
        amax_bits = blk[i] & 0x7FFF;
      }
    }
    int e = amax > 0.f ? bf16_floor_log2(amax_bits) - 2 + 127 : 0;
    if (e < 0) e = 0;
    if (e > 254) e = 254;
    scales[b] = (uint8_t)e;
    for (int i = 0; i < 32; i += 2) {
      uint8_t c[2];
      for (int h = 0; h < 2; ++h) {
        const float v = bf16_to_f32(blk[i + h]);
        const double y = std::ldexp((double)std::fabs(v), 127 - e);  // exact division by 2^(e-127)
        c[h] = (uint8_t)(e2m1_magnitude(y) | (std::signbit(v) ? 0x8 : 0));
      }
      codes[(32 * b + i) / 2] = (uint8_t)(c[0] | (c[1] << 4));
    }
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

}  // extern "C"
