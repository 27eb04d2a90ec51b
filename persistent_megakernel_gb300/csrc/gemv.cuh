// Warp-level matrix-vector tile products for the megakernel (sm_103a).
//
// A tile is nr <= NR rows x kn columns of a weight matrix in shared memory (rows of kn
// values, bf16 / e4m3 / e2m1 codes, MXFP4 scales after the values). Lane l owns the 16-byte
// column chunks l, l + 32, ... of every row. Loads of U chunks are issued before any of their
// math, and every (row, token) keeps two independent fp32x2 accumulator chains, so a warp has
// many independent shared-memory loads and FMAs in flight.
//
// Activations are fp32 in shared memory in a "quarter-plane" layout: with CW weights per
// 16-byte chunk and NVt = K / CW chunks per row, element k of token m sits at
//   act[m * K + (((k % CW) / 4) * NVt + k / CW) * 4 + k % 4]
// so the four activations of quarter q of chunk v are one 16-byte vector, and the 32 lanes
// of a warp read 32 consecutive vectors (no bank conflicts).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "dec_internal.h"
#include "ptx.cuh"

#ifndef DEC_MX_H2
#define DEC_MX_H2 1  // MXFP4: products and block partial sums in f16x2, one f32 conversion per block
#endif

namespace decimpl {
#if DEC_MX_H2
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte) {
  uint32_t h;
  asm("{ .reg .b8 t; .reg .b16 s; cvt.u16.u32 s, %1; cvt.u8.u16 t, s; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h) : "r"(byte));
  return h;
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// (lo, hi) -> f16x2 with lo in the low half
__device__ __forceinline__ uint32_t f32x2_to_h2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float2 h2_to_float2(uint32_t h) {
  float2 r;
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }" : "=f"(r.x), "=f"(r.y) : "r"(h));
  return r;
}
// A chunk's activations are scaled by 2^-k, k >= 0 the smallest shift that brings their largest
// magnitude below 2^8: products with e2m1 weights (|w| <= 6) stay below 1536 and a partial sum
// of 8 products below 2^14, far inside f16's range. 2^k multiplies the block's fp32 result.
__device__ __forceinline__ int h2_shift(float amax) {
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
  return e > 7 ? min(e - 7, 120) : 0;
}
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float((uint32_t)(127 + k) << 23); }
#endif
}  // namespace decimpl

namespace decimpl {

template <int WT>
struct WCfg {
  static constexpr int CW = WT == W_BF16 ? 8 : (WT == W_FP8 ? 16 : 32);  // weights per 16-byte chunk
  static constexpr int Q = CW / 4;                                       // activation quarters
};

__host__ __device__ __forceinline__ int chunk_width(int wtype) { return wtype == W_BF16 ? 8 : (wtype == W_FP8 ? 16 : 32); }

// Position of activation element k in the quarter-plane layout (see above).
__device__ __forceinline__ int act_pos(int k, int cw, int nvt) { return (((k % cw) >> 2) * nvt + k / cw) * 4 + (k & 3); }

template <int NR, int MT>
struct Acc {
  float2 c[NR][MT][2];
};

template <int NR, int MT>
__device__ __forceinline__ void acc_zero(Acc<NR, MT>& A) {
#pragma unroll
  for (int j = 0; j < NR; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m) A.c[j][m][0] = A.c[j][m][1] = make_float2(0.f, 0.f);
}

// A += W[tile] * act for this tile's columns [kc, kc + kn) of a K-column op.
// Only the first Mv (<= MT) tokens' activations are read; the others count as zero.
template <int WT, int MT, int NR>
__device__ __forceinline__ void warp_gemv(const uint8_t* slot, int nr, int kn, int kc, const float* act, int K,
                                          int Mv, Acc<NR, MT>& A, int lane) {
  constexpr int CW = WCfg<WT>::CW, Q = WCfg<WT>::Q;
  constexpr int U = WT == W_BF16 ? (MT == 1 ? 4 : 2) : (WT == W_FP8 ? 2 : 1);  // chunks per batch
  const int rb = WT == W_BF16 ? 2 * kn : (WT == W_FP8 ? kn : kn / 2);
  const int NV = kn / CW, NVt = K / CW, vb = kc / CW;
  const uint8_t* scales = slot + ((nr * rb + 15) & ~15);
  for (int v0 = lane; v0 < NV; v0 += 32 * U) {
    if constexpr (WT != W_MXFP4) {
      float4 a[U][MT][Q];
      uint4 w[U][NR];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        const bool ok = v < NV;
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int q = 0; q < Q; ++q)
            a[u][m][q] = (ok && (MT == 1 || m < Mv))
                             ? *reinterpret_cast<const float4*>(act + m * K + ((q * NVt + vb + v) << 2))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NR; ++j)
          w[u][j] = (ok && j < nr) ? *reinterpret_cast<const uint4*>(slot + (size_t)j * rb + v * 16)
                                   : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          const uint32_t ww[4] = {w[u][j].x, w[u][j].y, w[u][j].z, w[u][j].w};
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            // one token: two chains per row; several tokens: their chains are already independent
            float2 c0 = A.c[j][m][0], c1 = MT == 1 ? A.c[j][m][1] : make_float2(0.f, 0.f);
            float2& cb = *(MT == 1 ? &c1 : &c0);
            if constexpr (WT == W_BF16) {
              // word e holds weights 2e, 2e+1; quarter q = e / 2 holds activations 4q .. 4q+3
              c0 = ffma2(make_float2(bf16_lo(ww[0]), bf16_hi(ww[0])), make_float2(a[u][m][0].x, a[u][m][0].y), c0);
              cb = ffma2(make_float2(bf16_lo(ww[1]), bf16_hi(ww[1])), make_float2(a[u][m][0].z, a[u][m][0].w), cb);
              c0 = ffma2(make_float2(bf16_lo(ww[2]), bf16_hi(ww[2])), make_float2(a[u][m][1].x, a[u][m][1].y), c0);
              cb = ffma2(make_float2(bf16_lo(ww[3]), bf16_hi(ww[3])), make_float2(a[u][m][1].z, a[u][m][1].w), cb);
            } else {
              // word q holds e4m3 weights 4q .. 4q+3
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                c0 = ffma2(e4m3x2_to_float2(ww[q] & 0xFFFFu), make_float2(a[u][m][q].x, a[u][m][q].y), c0);
                cb = ffma2(e4m3x2_to_float2(ww[q] >> 16), make_float2(a[u][m][q].z, a[u][m][q].w), cb);
              }
            }
            A.c[j][m][0] = c0;
            if constexpr (MT == 1) A.c[j][m][1] = c1;
          }
        }
    } else {
      // MXFP4: a chunk is one 32-weight block with one E8M0 scale; byte b holds weights
      // 2b (low nibble) and 2b+1. Two halves of 16 weights keep the activations in registers.
      const int v = v0;
      uint4 w[NR];
      float X[NR];
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        w[j] = (j < nr) ? *reinterpret_cast<const uint4*>(slot + (size_t)j * rb + v * 16) : make_uint4(0u, 0u, 0u, 0u);
        X[j] = (j < nr) ? e8m0_to_float(scales[(size_t)j * (kn / 32) + v]) : 0.f;
      }
#if DEC_MX_H2
      // one token only: a window's per-token scales and f16x2 sums hold more registers than the
      // fp32 path below (measured on the MoE stack's 4-token windows: 7 % slower)
      if constexpr (MT == 1) {
        // per token: the chunk's activation scale first, then both halves in f16x2
        int up[MT];
        uint32_t hs[NR][MT][2];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          float amax = 0.f;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 x = (MT == 1 || m < Mv) ? *reinterpret_cast<const float4*>(act + m * K + ((q * NVt + vb + v) << 2))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
          }
          up[m] = h2_shift(amax);
#pragma unroll
          for (int j = 0; j < NR; ++j) hs[j][m][0] = hs[j][m][1] = 0u;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t ah[MT][8];
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const float down = pow2f(-up[m]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 x = (MT == 1 || m < Mv)
                                   ? *reinterpret_cast<const float4*>(act + m * K + (((4 * h + q) * NVt + vb + v) << 2))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
              ah[m][2 * q] = f32x2_to_h2(x.x * down, x.y * down);
              ah[m][2 * q + 1] = f32x2_to_h2(x.z * down, x.w * down);
            }
          }
#pragma unroll
          for (int j = 0; j < NR; ++j) {
            const uint32_t w0 = h ? w[j].z : w[j].x, w1 = h ? w[j].w : w[j].y;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              uint32_t a0 = hs[j][m][0], a1 = hs[j][m][1];
              a0 = hfma2_u32(e2m1x2_to_h2(w0 & 0xFFu), ah[m][0], a0);
              a1 = hfma2_u32(e2m1x2_to_h2((w0 >> 8) & 0xFFu), ah[m][1], a1);
              a0 = hfma2_u32(e2m1x2_to_h2((w0 >> 16) & 0xFFu), ah[m][2], a0);
              a1 = hfma2_u32(e2m1x2_to_h2(w0 >> 24), ah[m][3], a1);
              a0 = hfma2_u32(e2m1x2_to_h2(w1 & 0xFFu), ah[m][4], a0);
              a1 = hfma2_u32(e2m1x2_to_h2((w1 >> 8) & 0xFFu), ah[m][5], a1);
              a0 = hfma2_u32(e2m1x2_to_h2((w1 >> 16) & 0xFFu), ah[m][6], a0);
              a1 = hfma2_u32(e2m1x2_to_h2(w1 >> 24), ah[m][7], a1);
              hs[j][m][0] = a0;
              hs[j][m][1] = a1;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < NR; ++j)
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const float2 f0 = h2_to_float2(hs[j][m][0]), f1 = h2_to_float2(hs[j][m][1]);
            const float Xe = X[j] * pow2f(up[m]);
            A.c[j][m][0] = ffma2(make_float2(Xe, Xe), make_float2(f0.x + f1.x, f0.y + f1.y), A.c[j][m][0]);
          }
        continue;
      }
#endif
      float2 blk[NR][MT];
#pragma unroll
      for (int j = 0; j < NR; ++j)
#pragma unroll
        for (int m = 0; m < MT; ++m) blk[j][m] = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float4 a[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            a[m][q] = (MT == 1 || m < Mv)
                          ? *reinterpret_cast<const float4*>(act + m * K + (((4 * h + q) * NVt + vb + v) << 2))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          const uint32_t w0 = h ? w[j].z : w[j].x, w1 = h ? w[j].w : w[j].y;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            float2 b = blk[j][m];
            b = ffma2(e2m1x2_to_float2(w0 & 0xFFu), make_float2(a[m][0].x, a[m][0].y), b);
            b = ffma2(e2m1x2_to_float2((w0 >> 8) & 0xFFu), make_float2(a[m][0].z, a[m][0].w), b);
            b = ffma2(e2m1x2_to_float2((w0 >> 16) & 0xFFu), make_float2(a[m][1].x, a[m][1].y), b);
            b = ffma2(e2m1x2_to_float2(w0 >> 24), make_float2(a[m][1].z, a[m][1].w), b);
            b = ffma2(e2m1x2_to_float2(w1 & 0xFFu), make_float2(a[m][2].x, a[m][2].y), b);
            b = ffma2(e2m1x2_to_float2((w1 >> 8) & 0xFFu), make_float2(a[m][2].z, a[m][2].w), b);
            b = ffma2(e2m1x2_to_float2((w1 >> 16) & 0xFFu), make_float2(a[m][3].x, a[m][3].y), b);
            b = ffma2(e2m1x2_to_float2(w1 >> 24), make_float2(a[m][3].z, a[m][3].w), b);
            blk[j][m] = b;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NR; ++j)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float2 xx = make_float2(X[j], X[j]);
          A.c[j][m][0] = ffma2(xx, blk[j][m], A.c[j][m][0]);
        }
    }
  }
}

// Sum the accumulators over the 32 lanes; lane j*MT + m ends up holding row j, token m
// (nr * MT <= 32), which it returns.
template <int NR, int MT>
__device__ __forceinline__ float warp_rowsums(Acc<NR, MT>& A, int nr, int lane) {
  float mine = 0.f;
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    if (j < nr) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float t = (A.c[j][m][0].x + A.c[j][m][0].y) + (A.c[j][m][1].x + A.c[j][m][1].y);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == j * MT + m) mine = t;
      }
    }
  }
  return mine;
}

}  // namespace decimpl

namespace decimpl {

// ------------------------------------------------------------------ activations in registers
template <int WT>
struct RegCfg {  // chunks per lane an op's activations may occupy in registers (K <= 32 * NI * CW)
  static constexpr int NI = WT == W_BF16 ? 10 : (WT == W_FP8 ? 5 : 3);
};

// For a one-token op whose columns this warp covers fit in NI chunks per lane, the warp loads
// its activations once per op and keeps them in registers, so a tile costs one shared-memory
// read per weight byte instead of two (the bulk copy writing the slot is the third access).
template <int WT, int NI>
struct ActRegs {
  float4 a[NI][WCfg<WT>::Q];
};

#if DEC_MX_H2
// MXFP4: f16 pairs (elements 2k, 2k+1 of chunk i in h[i][k]) scaled by 2^-k_i; e[i] = 2^k_i.
template <int NI>
struct ActRegs<W_MXFP4, NI> {
  uint32_t h[NI][16];
  float e[NI];
};
#endif

// Load chunks v = lane + 32 i (i < NI) of columns [c0, c0 + cn) of the op's activation plane.
template <int WT, int NI>
__device__ __forceinline__ void act_regs_load(ActRegs<WT, NI>& R, const float* act, int K, int c0, int cn, int lane) {
  constexpr int CW = WCfg<WT>::CW, Q = WCfg<WT>::Q;
  const int NVt = K / CW, vb = c0 / CW, NV = cn / CW;
#if DEC_MX_H2
  if constexpr (WT == W_MXFP4) {
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int v = lane + 32 * i;
      float4 x[8];
      float amax = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        x[q] = v < NV ? *reinterpret_cast<const float4*>(act + ((q * NVt + vb + v) << 2)) : make_float4(0.f, 0.f, 0.f, 0.f);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x[q].x), fabsf(x[q].y)), fmaxf(fabsf(x[q].z), fabsf(x[q].w))));
      }
      const int k = h2_shift(amax);
      const float down = pow2f(-k);
      R.e[i] = pow2f(k);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        R.h[i][2 * q] = f32x2_to_h2(x[q].x * down, x[q].y * down);
        R.h[i][2 * q + 1] = f32x2_to_h2(x[q].z * down, x[q].w * down);
      }
    }
  } else
#endif
  {
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int v = lane + 32 * i;
#pragma unroll
      for (int q = 0; q < Q; ++q)
        R.a[i][q] = v < NV ? *reinterpret_cast<const float4*>(act + ((q * NVt + vb + v) << 2)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// Pin the accumulators: every FMA feeding them is issued before this point and no memory
// access moves across it. Bounds how far the compiler may run weight loads ahead of the math.
template <int NR, int MT>
__device__ __forceinline__ void acc_pin(Acc<NR, MT>& A) {
#pragma unroll
  for (int j = 0; j < NR; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m)
      asm volatile("" : "+f"(A.c[j][m][0].x), "+f"(A.c[j][m][0].y), "+f"(A.c[j][m][1].x), "+f"(A.c[j][m][1].y)::"memory");
}

// A += W[tile] * act for a tile whose columns are exactly the ones loaded in R (kn = cn).
// Software-pipelined over groups of F chunks: the loads of group g + 1 are issued before the
// math of group g, and the accumulators are pinned after it, so at most 2 F NR 16-byte weight
// vectors are live next to the activations.
template <int WT, int NR, int NI>
__device__ __forceinline__ void warp_gemv_reg(const uint8_t* slot, int nr, int kn, const ActRegs<WT, NI>& R,
                                              Acc<NR, 1>& A, int lane) {
  constexpr int CW = WCfg<WT>::CW;
  constexpr int F = NR >= 8 ? 1 : (NR >= 4 ? 2 : 4);  // chunks per group
  constexpr int NG = (NI + F - 1) / F;
  const int rb = WT == W_BF16 ? 2 * kn : (WT == W_FP8 ? kn : kn / 2);
  const int NV = kn / CW;
  const uint8_t* scales = slot + ((nr * rb + 15) & ~15);
  uint4 w[2][F][NR];
  auto load = [&](int g) {
#pragma unroll
    for (int f = 0; f < F; ++f) {
      const int i = g * F + f;
      const int v = lane + 32 * i;
      // chunks past the tile's columns contribute zero (their activations are zero)
      const bool ok = i < NI && v < NV;
#pragma unroll
      for (int j = 0; j < NR; ++j)
        w[g & 1][f][j] = (ok && j < nr) ? *reinterpret_cast<const uint4*>(slot + (size_t)j * rb + v * 16)
                                        : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load(0);
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    if (g + 1 < NG) load(g + 1);
#pragma unroll
    for (int f = 0; f < F; ++f) {
      const int i = g * F + f;
      if (i >= NI) break;
      const uint4* wg = w[g & 1][f];
      if constexpr (WT == W_BF16) {
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          float2 c0 = A.c[j][0][0], c1 = A.c[j][0][1];
          c0 = ffma2(make_float2(bf16_lo(wg[j].x), bf16_hi(wg[j].x)), make_float2(R.a[i][0].x, R.a[i][0].y), c0);
          c1 = ffma2(make_float2(bf16_lo(wg[j].y), bf16_hi(wg[j].y)), make_float2(R.a[i][0].z, R.a[i][0].w), c1);
          c0 = ffma2(make_float2(bf16_lo(wg[j].z), bf16_hi(wg[j].z)), make_float2(R.a[i][1].x, R.a[i][1].y), c0);
          c1 = ffma2(make_float2(bf16_lo(wg[j].w), bf16_hi(wg[j].w)), make_float2(R.a[i][1].z, R.a[i][1].w), c1);
          A.c[j][0][0] = c0;
          A.c[j][0][1] = c1;
        }
      } else if constexpr (WT == W_FP8) {
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          const uint32_t ww[4] = {wg[j].x, wg[j].y, wg[j].z, wg[j].w};
          float2 c0 = A.c[j][0][0], c1 = A.c[j][0][1];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            c0 = ffma2(e4m3x2_to_float2(ww[q] & 0xFFFFu), make_float2(R.a[i][q].x, R.a[i][q].y), c0);
            c1 = ffma2(e4m3x2_to_float2(ww[q] >> 16), make_float2(R.a[i][q].z, R.a[i][q].w), c1);
          }
          A.c[j][0][0] = c0;
          A.c[j][0][1] = c1;
        }
      } else {
        const int v = lane + 32 * i;
        const bool ok = v < NV;
#if DEC_MX_H2
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          const uint32_t ww[4] = {wg[j].x, wg[j].y, wg[j].z, wg[j].w};
          uint32_t h0 = 0u, h1 = 0u;  // two f16x2 partial sums of 8 products each
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            h0 = hfma2_u32(e2m1x2_to_h2(ww[q] & 0xFFu), R.h[i][4 * q], h0);
            h1 = hfma2_u32(e2m1x2_to_h2((ww[q] >> 8) & 0xFFu), R.h[i][4 * q + 1], h1);
            h0 = hfma2_u32(e2m1x2_to_h2((ww[q] >> 16) & 0xFFu), R.h[i][4 * q + 2], h0);
            h1 = hfma2_u32(e2m1x2_to_h2(ww[q] >> 24), R.h[i][4 * q + 3], h1);
          }
          const float2 f0 = h2_to_float2(h0), f1 = h2_to_float2(h1);
          const float X = (ok && j < nr) ? e8m0_to_float(scales[(size_t)j * (kn / 32) + v]) * R.e[i] : 0.f;
          A.c[j][0][0] = ffma2(make_float2(X, X), make_float2(f0.x + f1.x, f0.y + f1.y), A.c[j][0][0]);
        }
#else
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          const uint32_t ww[4] = {wg[j].x, wg[j].y, wg[j].z, wg[j].w};
          float2 b0 = make_float2(0.f, 0.f), b1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            // word q: bytes -> weights 8q .. 8q+7, activations quarters 2q, 2q+1
            b0 = ffma2(e2m1x2_to_float2(ww[q] & 0xFFu), make_float2(R.a[i][2 * q].x, R.a[i][2 * q].y), b0);
            b1 = ffma2(e2m1x2_to_float2((ww[q] >> 8) & 0xFFu), make_float2(R.a[i][2 * q].z, R.a[i][2 * q].w), b1);
            b0 = ffma2(e2m1x2_to_float2((ww[q] >> 16) & 0xFFu), make_float2(R.a[i][2 * q + 1].x, R.a[i][2 * q + 1].y),
                       b0);
            b1 = ffma2(e2m1x2_to_float2(ww[q] >> 24), make_float2(R.a[i][2 * q + 1].z, R.a[i][2 * q + 1].w), b1);
          }
          const float X = (ok && j < nr) ? e8m0_to_float(scales[(size_t)j * (kn / 32) + v]) : 0.f;
          const float2 xx = make_float2(X, X);
          A.c[j][0][0] = ffma2(xx, b0, A.c[j][0][0]);
          A.c[j][0][1] = ffma2(xx, b1, A.c[j][0][1]);
        }
#endif
      }
    }
    acc_pin(A);
  }
}

}  // namespace decimpl
