// The persistent decode megakernel for sm_103a.
//
// One CTA per SM (288 threads: 8 consumer warps + 1 producer warp, up to 227 KB of shared
// memory). Every CTA walks the step's op list. For each op the producer thread streams the
// CTA's share of the op's weights (or cached keys/values) into a ring of 32 KB shared-memory
// slots with bulk asynchronous copies tracked by mbarriers. It never waits for activations,
// so it runs ahead across op boundaries: the next op's bytes are in flight while the
// previous op is still finishing on other SMs (Muse Spark Open megakernel article, sections
// "the baseline nobody benchmarked" -- one resident kernel, warps start the next op before
// the previous one retires -- and "three bills" -- a per-SM ring of weight slots). The
// consumers wait on a GPU-scope counter for the op's input, compute on the landed tiles, and
// release-add the op's own counter. Every wait is bounded by %globaltimer; on expiry the CTA
// records the failure in the status word, raises the global abort flag, lets its copies in
// flight land and returns.
//
// Matrix-vector products: a tile is `nr` rows of a [rows][K] matrix. Consumer thread t owns
// the 16-byte column chunks t % tpr, t % tpr + tpr, ... of rows t / tpr + j * (256 / tpr);
// partial sums are reduced with warp shuffles and, across warps, through shared memory in a
// fixed order, so results are bitwise reproducible run to run and between launch modes.
// Activations sit in shared memory in fp32 and accumulation is fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/dec.h"
#include "dec_internal.h"
#include "ptx.cuh"

namespace decimpl {

// ------------------------------------------------------------------ shared memory map
constexpr int kCommonBytes = 8192;
constexpr int kOffFull = 0, kOffEmpty = 64, kOffOp = 128, kOffRed = 512, kOffRes = 2560, kOffRope = 3584,
              kOffFlags = 5632, kOffRoute = 5696, kOffPRoute = 6720;
static_assert(sizeof(OpDesc) <= kOffRed - kOffOp, "OpDesc copy");
static_assert(sizeof(RouteBlock) <= kOffPRoute - kOffRoute, "RouteBlock copy");
static_assert(kOffPRoute + 4 * (1 + kMaxRouteSlots) <= kCommonBytes, "common area");

struct Smem {
  uint8_t* ring;
  float* act;         // op scratch: activations [M][K], attention state, argmax scratch ...
  uint64_t* full;     // [kMaxSlots]
  uint64_t* empty;    // [kMaxSlots]
  OpDesc* op;         // consumer copy of the current op
  float* red;         // [8 warps][64] cross-warp partial sums
  float* res;         // [256] results of the current tile
  float2* rope;       // [kMmax][64] (cos, sin) at pos + m
  int* flags;         // [16]
  RouteBlock* route;  // consumer copy of the layer's routing
  int* proute;        // producer copy: [0] n_slots, [1 + slot] expert id
};

__device__ __forceinline__ Smem carve(uint8_t* base, const KParams& p) {
  Smem s;
  s.ring = base;
  s.act = reinterpret_cast<float*>(base + (size_t)p.nslot * kSlotBytes);
  uint8_t* c = base + (size_t)p.nslot * kSlotBytes + p.act_bytes;
  s.full = reinterpret_cast<uint64_t*>(c + kOffFull);
  s.empty = reinterpret_cast<uint64_t*>(c + kOffEmpty);
  s.op = reinterpret_cast<OpDesc*>(c + kOffOp);
  s.red = reinterpret_cast<float*>(c + kOffRed);
  s.res = reinterpret_cast<float*>(c + kOffRes);
  s.rope = reinterpret_cast<float2*>(c + kOffRope);
  s.flags = reinterpret_cast<int*>(c + kOffFlags);
  s.route = reinterpret_cast<RouteBlock*>(c + kOffRoute);
  s.proute = reinterpret_cast<int*>(c + kOffPRoute);
  return s;
}

// ------------------------------------------------------------------ failure handling
__device__ __forceinline__ bool aborted(const KParams& p) {
  return *reinterpret_cast<volatile uint32_t*>(&p.status->abort) != 0u;
}

__device__ void raise_error(const KParams& p, uint32_t code, int op, uint32_t ctr, uint32_t obs, uint32_t tgt,
                            uint32_t where) {
  if (atomicCAS(&p.status->code, 0u, code) == 0u) {
    p.status->op = op;
    p.status->cta = blockIdx.x;
    p.status->counter = ctr;
    p.status->observed = obs;
    p.status->target = tgt;
    p.status->where = where;
  }
  __threadfence();
  atomicExch(&p.status->abort, 1u);
}

// Wait until counter >= target (wrap-safe). False on abort or timeout (timeout recorded).
__device__ bool wait_counter(const KParams& p, int ctr, uint32_t target, int op, uint32_t where) {
  uint32_t v = ld_acquire(&p.ctr[ctr]);
  if ((int32_t)(v - target) >= 0) return true;
  const uint64_t t0 = gtimer();
  for (;;) {
    v = ld_acquire(&p.ctr[ctr]);
    if ((int32_t)(v - target) >= 0) return true;
    if (aborted(p)) return false;
    if (gtimer() - t0 > p.timeout_ns) {
      raise_error(p, DEC_ERR_TIMEOUT, op, (uint32_t)ctr, v, target, where);
      return false;
    }
  }
}

__device__ bool wait_mbar(const KParams& p, uint32_t bar, uint32_t parity, int op, uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (int it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15) == 0) {
      if (aborted(p)) return false;
      if (gtimer() - t0 > p.timeout_ns) {
        raise_error(p, DEC_ERR_TIMEOUT, op, 0xFFFFFFFFu, 0u, parity, where);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ work partition
// Rows [a, b) of an R-row op owned by `cta`, in units of `unit` rows.
__device__ __forceinline__ void cta_rows(int R, int unit, int C, int cta, int& a, int& b) {
  const long long U = R / unit;
  a = (int)(U * cta / C) * unit;
  b = (int)(U * (cta + 1) / C) * unit;
}

// Attention: kv head g has ns_max splits of the positions [0, S), S = pos + M.
__device__ __forceinline__ void split_range(int S, int ns, int j, int& head, int& s, int& p0, int& p1) {
  head = j / ns;
  s = j % ns;
  p0 = (int)((long long)S * s / ns);
  p1 = (int)((long long)S * (s + 1) / ns);
}

__device__ __forceinline__ int row_bytes(int wtype, int K) {
  return wtype == W_BF16 ? 2 * K : (wtype == W_FP8 ? K : K / 2);
}

// ------------------------------------------------------------------ producer
struct Producer {
  const KParams& p;
  Smem& s;
  uint32_t T;  // tiles issued so far (ring position)
  bool ok;

  __device__ bool issue(int op_idx, const void* src, uint32_t bytes, const void* src2, uint32_t bytes2,
                        uint32_t off2) {
    const uint32_t slot = T % (uint32_t)p.nslot;
    const uint32_t parity = ((T / (uint32_t)p.nslot) & 1u) ^ 1u;
    if (!wait_mbar(p, smem_addr(&s.empty[slot]), parity, op_idx, 1)) return false;
    const uint32_t fb = smem_addr(&s.full[slot]);
    const uint32_t dst = smem_addr(s.ring + (size_t)slot * kSlotBytes);
    mbar_expect_tx(fb, bytes + bytes2);
    bulk_g2s(dst, src, bytes, fb);
    if (bytes2) bulk_g2s(dst + off2, src2, bytes2, fb);
    ++T;
    return true;
  }

  __device__ bool gemv_tile(int op_idx, const OpDesc& op, int mat, int r0, int nr) {
    const int rb = row_bytes(op.wtype, op.K);
    const char* src = static_cast<const char*>(op.w) + (size_t)mat * op.w_mstride + (size_t)r0 * rb;
    const uint32_t bytes = (uint32_t)(nr * rb);
    if (op.wtype == W_MXFP4) {
      const int sb = op.K / 32;
      const char* s2 = static_cast<const char*>(op.ws) + (size_t)mat * op.ws_mstride + (size_t)r0 * sb;
      return issue(op_idx, src, bytes, s2, (uint32_t)(nr * sb), (bytes + 15u) & ~15u);
    }
    return issue(op_idx, src, bytes, nullptr, 0u, 0u);
  }

  __device__ void run(uint32_t epoch, int pos, int M) {
    const int C = p.n_ctas, cta = blockIdx.x;
    int n_slots = 0;
    for (int oi = p.op_begin; oi < p.op_end && ok; ++oi) {
      const OpDesc op = p.ops[oi];
      if (op.pwait_ctr >= 0) {
        if (!wait_counter(p, op.pwait_ctr, (epoch + 1u) * (uint32_t)op.pwait_n, oi, 2)) {
          ok = false;
          break;
        }
        const RouteBlock* rb = reinterpret_cast<const RouteBlock*>(op.route);
        n_slots = __ldcg(&rb->n_slots);
        for (int i = 0; i < n_slots; ++i) s.proute[1 + i] = __ldcg(&rb->expert[i]);
      }
      switch (op.type) {
        case OP_ATTN: {
          const int S = pos + M, ns = p.ns_max;
          for (int j = cta; j < p.n_kv * ns && ok; j += C) {
            int head, sidx, p0, p1;
            split_range(S, ns, j, head, sidx, p0, p1);
            const int ce = min(p1, pos);
            for (int q = p0; q < ce && ok; q += kAttnTilePos) {
              const int n = min(kAttnTilePos, ce - q);
              const size_t off = ((size_t)head * p.cap + q) * kHeadDim;
              ok = issue(oi, op.kc + off, (uint32_t)n * 256u, op.vc + off, (uint32_t)n * 256u, (uint32_t)n * 256u);
            }
          }
          break;
        }
        case OP_SHARED_GATEUP:
        case OP_ROUTED_GATEUP: {
          const int s0 = op.slot0, s1 = op.type == OP_SHARED_GATEUP ? op.slot1 : n_slots;
          int a, b;
          cta_rows((s1 - s0) * op.N, op.unit, C, cta, a, b);
          for (int r = a; r < b && ok;) {
            const int sl = s0 + r / op.N, lr = r % op.N;
            const int nr = min(op.rpt, min(b - r, op.N - lr));
            const int expert = op.type == OP_SHARED_GATEUP ? p.E + sl : s.proute[1 + sl];
            ok = gemv_tile(oi, op, expert, lr, nr);
            r += nr;
          }
          break;
        }
        case OP_EXP_DOWN: {
          int a, b;
          cta_rows(op.N, op.unit, C, cta, a, b);
          for (int sl = 0; sl < n_slots && ok; ++sl)
            for (int r = a; r < b && ok; r += op.rpt)
              ok = gemv_tile(oi, op, s.proute[1 + sl], r, min(op.rpt, b - r));
          break;
        }
        default: {
          int a, b;
          cta_rows(op.N, op.unit, C, cta, a, b);
          for (int r = a; r < b && ok; r += op.rpt) ok = gemv_tile(oi, op, 0, r, min(op.rpt, b - r));
          break;
        }
      }
    }
    // Every copy in flight must land before the CTA may exit: wait for the last nslot tiles.
    const uint32_t n = T < (uint32_t)p.nslot ? T : (uint32_t)p.nslot;
    for (uint32_t k = 0; k < n; ++k) {
      const uint32_t t = T - 1u - k;
      const uint32_t slot = t % (uint32_t)p.nslot;
      const uint32_t parity = (t / (uint32_t)p.nslot) & 1u;
      const uint32_t fb = smem_addr(&s.full[slot]);
      const uint64_t t0 = gtimer();
      while (!mbar_try_wait(fb, parity)) {
        if (gtimer() - t0 > p.timeout_ns) break;
      }
    }
  }
};

// ------------------------------------------------------------------ consumer helpers
// x[m][k] of the op's residual / norm input.
__device__ __forceinline__ float load_x(const KParams& p, const OpDesc& op, const StepState& st, int m, int k) {
  switch (op.xsrc) {
    case X_F32:
      return __ldcg(p.hs + ((size_t)op.x_idx * p.Mmax + m) * p.H + k);
    case X_EMBED: {
      const uint16_t* e = static_cast<const uint16_t*>(op.x_src) + (size_t)st.tokens[m] * p.H + k;
      return __uint_as_float((uint32_t)__ldg(e) << 16);
    }
    case X_HIDDEN_IN: {
      const uint16_t* e = static_cast<const uint16_t*>(st.hidden_in) + (size_t)m * p.H + k;
      return __uint_as_float((uint32_t)__ldg(e) << 16);
    }
    default:
      return 0.f;
  }
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------------ GEMV tile
// res[i * MT + m] = sum_k W[i][k] * act[m][k] for the nr rows in `slot` (before row scales).
template <int WT, int MT>
__device__ __forceinline__ void gemv_tile(const uint8_t* slot, int nr, int K, int tpr, const float* act, float* red,
                                          float* res, uint32_t empty_bar, int tid) {
  constexpr int CW = WT == W_BF16 ? 8 : (WT == W_FP8 ? 16 : 32);  // weights per 16-byte chunk
  const int rb = WT == W_BF16 ? 2 * K : (WT == W_FP8 ? K : K / 2);
  const int NV = K / CW;
  const int rgn = kConsumerThreads / tpr;
  const int rg = tid / tpr, tl = tid % tpr;
  const uint8_t* scales = slot + ((nr * rb + 15) & ~15);

  float acc[kRmax][MT];
#pragma unroll
  for (int j = 0; j < kRmax; ++j)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[j][m] = 0.f;

  for (int v = tl; v < NV; v += tpr) {
    if constexpr (WT == W_BF16) {
      float a[MT][8];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const float4 x0 = *reinterpret_cast<const float4*>(act + m * K + v * 8);
        const float4 x1 = *reinterpret_cast<const float4*>(act + m * K + v * 8 + 4);
        a[m][0] = x0.x; a[m][1] = x0.y; a[m][2] = x0.z; a[m][3] = x0.w;
        a[m][4] = x1.x; a[m][5] = x1.y; a[m][6] = x1.z; a[m][7] = x1.w;
      }
#pragma unroll
      for (int j = 0; j < kRmax; ++j) {
        const int i = rg + j * rgn;
        if (i < nr) {
          const uint4 w = *reinterpret_cast<const uint4*>(slot + (size_t)i * rb + v * 16);
          const float wf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                               bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            float t = acc[j][m];
#pragma unroll
            for (int e = 0; e < 8; ++e) t = fmaf(wf[e], a[m][e], t);
            acc[j][m] = t;
          }
        }
      }
    } else if constexpr (WT == W_FP8) {
      float a[MT][16];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 x = *reinterpret_cast<const float4*>(act + m * K + v * 16 + 4 * q);
          a[m][4 * q] = x.x; a[m][4 * q + 1] = x.y; a[m][4 * q + 2] = x.z; a[m][4 * q + 3] = x.w;
        }
#pragma unroll
      for (int j = 0; j < kRmax; ++j) {
        const int i = rg + j * rgn;
        if (i < nr) {
          const uint4 w = *reinterpret_cast<const uint4*>(slot + (size_t)i * rb + v * 16);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
          float wf[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 lo = e4m3x2_to_float2(ww[q] & 0xFFFFu);
            const float2 hi = e4m3x2_to_float2(ww[q] >> 16);
            wf[4 * q] = lo.x; wf[4 * q + 1] = lo.y; wf[4 * q + 2] = hi.x; wf[4 * q + 3] = hi.y;
          }
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            float t = acc[j][m];
#pragma unroll
            for (int e = 0; e < 16; ++e) t = fmaf(wf[e], a[m][e], t);
            acc[j][m] = t;
          }
        }
      }
    } else {  // MXFP4: one 16-byte chunk = one 32-weight block with one E8M0 scale
      float bs[kRmax][MT];
#pragma unroll
      for (int j = 0; j < kRmax; ++j)
#pragma unroll
        for (int m = 0; m < MT; ++m) bs[j][m] = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float a[MT][16];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 x = *reinterpret_cast<const float4*>(act + m * K + v * 32 + 16 * h + 4 * q);
            a[m][4 * q] = x.x; a[m][4 * q + 1] = x.y; a[m][4 * q + 2] = x.z; a[m][4 * q + 3] = x.w;
          }
#pragma unroll
        for (int j = 0; j < kRmax; ++j) {
          const int i = rg + j * rgn;
          if (i < nr) {
            const uint2 w = *reinterpret_cast<const uint2*>(slot + (size_t)i * rb + v * 16 + 8 * h);
            const uint32_t ww[2] = {w.x, w.y};
            float wf[16];
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const float2 f = e2m1x2_to_float2((ww[q] >> (8 * b)) & 0xFFu);
                wf[8 * q + 2 * b] = f.x;
                wf[8 * q + 2 * b + 1] = f.y;
              }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              float t = bs[j][m];
#pragma unroll
              for (int e = 0; e < 16; ++e) t = fmaf(wf[e], a[m][e], t);
              bs[j][m] = t;
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kRmax; ++j) {
        const int i = rg + j * rgn;
        if (i < nr) {
          const float X = e8m0_to_float(scales[(size_t)i * (K / 32) + v]);
#pragma unroll
          for (int m = 0; m < MT; ++m) acc[j][m] = fmaf(X, bs[j][m], acc[j][m]);
        }
      }
    }
  }
  // This warp no longer reads the slot.
  __syncwarp();
  if ((tid & 31) == 0) mbar_arrive(empty_bar);

  // Reduce within the warp (a warp never spans two row groups: tpr >= 32) ...
  const int warp = tid >> 5, lane = tid & 31;
  const int wpr = tpr >> 5;  // warps per row group
#pragma unroll
  for (int j = 0; j < kRmax; ++j) {
    const int i = rg + j * rgn;
    if (i < nr) {
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float t = acc[j][m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) {
          if (wpr == 1)
            res[i * MT + m] = t;
          else
            red[warp * 64 + j * MT + m] = t;
        }
      }
    }
  }
  if (wpr > 1) {
    consumer_sync();
    // ... then across the warps of a row group, in warp order.
    if (tid < nr * MT) {
      const int i = tid / MT, m = tid % MT;
      const int g = i % rgn, j = i / rgn;
      float t = 0.f;
      for (int w = 0; w < wpr; ++w) t += red[(g * wpr + w) * 64 + j * MT + m];
      res[tid] = t;
    }
  }
  consumer_sync();
}

template <int MT>
__device__ __forceinline__ void gemv_w(int wtype, const uint8_t* slot, int nr, int K, int tpr, const float* act,
                                       float* red, float* res, uint32_t eb, int tid) {
  if (wtype == W_BF16)
    gemv_tile<W_BF16, MT>(slot, nr, K, tpr, act, red, res, eb, tid);
  else if (wtype == W_FP8)
    gemv_tile<W_FP8, MT>(slot, nr, K, tpr, act, red, res, eb, tid);
  else
    gemv_tile<W_MXFP4, MT>(slot, nr, K, tpr, act, red, res, eb, tid);
}

__device__ __noinline__ void gemv_any(int M, int wtype, const uint8_t* slot, int nr, int K, int tpr, const float* act,
                                      float* red, float* res, uint32_t eb, int tid) {
  switch (M) {
    case 1: gemv_w<1>(wtype, slot, nr, K, tpr, act, red, res, eb, tid); break;
    case 2: gemv_w<2>(wtype, slot, nr, K, tpr, act, red, res, eb, tid); break;
    case 3: gemv_w<3>(wtype, slot, nr, K, tpr, act, red, res, eb, tid); break;
    default: gemv_w<4>(wtype, slot, nr, K, tpr, act, red, res, eb, tid); break;
  }
}

// ------------------------------------------------------------------ attention
// Scratch in s.act (floats):
//   q    [MG][128]   query rows of the kv group, rotated, times log2(e)/sqrt(128)
//   sc   [MG][64]    scores of the current tile, then probabilities
//   mrun, lrun, scale [32] each
//   kv   bf16 [2][kMmax][128]  this call's own rows (keys then values), laid out like a slot
//   ored [16][128]   sum over position classes (M = 1 path)
//   cw   [MG][ns]    combine weights
struct AttnScratch {
  float* q;
  float* sc;
  float* mrun;
  float* lrun;
  float* scale;
  uint8_t* kvnew;
  float* ored;
  float* cw;
};

__device__ __forceinline__ AttnScratch attn_scratch(const KParams& p, const Smem& s, int M) {
  const int MG = M * p.G;
  AttnScratch a;
  float* f = s.act;
  a.q = f; f += MG * 128;
  a.sc = f; f += MG * 64;
  a.mrun = f; f += 32;
  a.lrun = f; f += 32;
  a.scale = f; f += 32;
  a.kvnew = reinterpret_cast<uint8_t*>(f); f += (2 * kMmax * 256) / 4;
  a.ored = f; f += 16 * 128;
  a.cw = f;
  return a;
}

// sc[mh][j] = q[mh] . K[j] for the tile's n rows (256 B each). Eight lanes share one position
// (16 dims, 32 contiguous bytes each), so a warp reads four whole rows per step without bank
// conflicts; NQ query rows are held in registers.
template <int NQ>
__device__ __forceinline__ void attn_scores(const uint8_t* krows, int n, const AttnScratch& a, int mh0, int MG,
                                            int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 3, sub = lane & 7;
  float q[NQ][16];
#pragma unroll
  for (int h = 0; h < NQ; ++h)
#pragma unroll
    for (int e = 0; e < 16; ++e) q[h][e] = (mh0 + h < MG) ? a.q[(mh0 + h) * 128 + sub * 16 + e] : 0.f;
  for (int j0 = warp * 4; j0 < n; j0 += 32) {
    const int j = j0 + grp;
    float kf[16];
    if (j < n) {
      const uint4 k0 = *reinterpret_cast<const uint4*>(krows + (size_t)j * 256 + sub * 32);
      const uint4 k1 = *reinterpret_cast<const uint4*>(krows + (size_t)j * 256 + sub * 32 + 16);
      const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        kf[2 * e] = bf16_lo(kw[e]);
        kf[2 * e + 1] = bf16_hi(kw[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) kf[e] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < NQ; ++h) {
      float t = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) t = fmaf(q[h][e], kf[e], t);
      t += __shfl_xor_sync(0xffffffffu, t, 4);
      t += __shfl_xor_sync(0xffffffffu, t, 2);
      t += __shfl_xor_sync(0xffffffffu, t, 1);
      if (sub == 0 && j < n && mh0 + h < MG) a.sc[(mh0 + h) * 64 + j] = t;
    }
  }
}

// Online softmax over one tile for every (m, h): running max, rescale, p = 2^(s - max).
// vis_base < 0: every row is visible (cached rows); else tile row j is this call's row
// vis_base + j, visible to token m iff vis_base + j <= m (causal within the window).
__device__ __forceinline__ void attn_softmax(const AttnScratch& a, int n, int M, int G, int vis_base, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const int MG = M * G;
  for (int mh = warp; mh < MG; mh += kConsumerWarps) {
    const int m = mh / G;
    float mx = -INFINITY;
    for (int j = lane; j < n; j += 32) {
      const bool vis = vis_base < 0 || (vis_base + j <= m);
      const float sv = vis ? a.sc[mh * 64 + j] : -INFINITY;
      a.sc[mh * 64 + j] = sv;
      mx = fmaxf(mx, sv);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mold = a.mrun[mh];
    const float mnew = fmaxf(mold, mx);
    float sum = 0.f;
    for (int j = lane; j < n; j += 32) {
      const float sv = a.sc[mh * 64 + j];
      const float pj = (mnew == -INFINITY) ? 0.f : exp2f(sv - mnew);
      a.sc[mh * 64 + j] = pj;
      sum += pj;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      const float sc = (mnew == -INFINITY) ? 1.f : ((mold == -INFINITY) ? 0.f : exp2f(mold - mnew));
      a.scale[mh] = sc;
      a.lrun[mh] = a.lrun[mh] * sc + sum;
      a.mrun[mh] = mnew;
    }
  }
}

// Value pass, any M: thread t owns dims (2 (t % 64), +1) of pairs mh = t / 64 + 4k.
struct OGen {
  float o[8][2];
};

__device__ __forceinline__ void attn_values_generic(OGen& acc, const uint8_t* vrows, int n, const AttnScratch& a,
                                                    int MG, int tid) {
  const int dp = tid & 63, hs = tid >> 6;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int mh = hs + 4 * k;
    if (mh < MG) {
      const float sc = a.scale[mh];
      acc.o[k][0] *= sc;
      acc.o[k][1] *= sc;
    }
  }
  for (int j = 0; j < n; ++j) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(vrows + (size_t)j * 256 + dp * 4);
    const float v0 = bf16_lo(v), v1 = bf16_hi(v);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int mh = hs + 4 * k;
      if (mh < MG) {
        const float pj = a.sc[mh * 64 + j];
        acc.o[k][0] = fmaf(pj, v0, acc.o[k][0]);
        acc.o[k][1] = fmaf(pj, v1, acc.o[k][1]);
      }
    }
  }
}

// Value pass, M = 1: thread t owns dims 8 (t % 16) .. +8 of rows j = t / 16 (mod 16), for all G
// heads of the group; the 16 row classes are summed once, at the end of the split.
template <int G_>
struct O1 {
  float o[G_][8];
};

template <int G_>
__device__ __forceinline__ void attn_values_m1(O1<G_>& acc, const uint8_t* vrows, int n, const AttnScratch& a,
                                               int tid) {
  const int c = tid & 15, pc = tid >> 4;
#pragma unroll
  for (int h = 0; h < G_; ++h) {
    const float sc = a.scale[h];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc.o[h][e] *= sc;
  }
  for (int j = pc; j < n; j += 16) {
    const uint4 v = *reinterpret_cast<const uint4*>(vrows + (size_t)j * 256 + c * 16);
    const float vf[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                         bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
    for (int h = 0; h < G_; ++h) {
      const float pj = a.sc[h * 64 + j];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc.o[h][e] = fmaf(pj, vf[e], acc.o[h][e]);
    }
  }
}

// ------------------------------------------------------------------ consumer
struct Consumer {
  const KParams& p;
  Smem& s;
  uint32_t T;  // ring tiles consumed
  uint32_t epoch;
  const StepState& st;
  int tid;

  __device__ bool wait_dep(int ctr, int n, int op_idx, uint32_t where) {
    if (ctr < 0) return true;
    if (tid == 0) s.flags[0] = wait_counter(p, ctr, (epoch + 1u) * (uint32_t)n, op_idx, where) ? 1 : 0;
    consumer_sync();
    const bool ok = s.flags[0] != 0;
    consumer_sync();
    return ok;
  }

  __device__ void signal(int ctr) {
    consumer_sync();
    if (tid == 0 && ctr >= 0) {
      __threadfence();
      red_release(&p.ctr[ctr], 1u);
    }
  }

  // Arrive at ticket t (n arrivals per step); true in the last arrival (all consumers agree).
  __device__ bool ticket(int t, int n) {
    consumer_sync();
    if (tid == 0) {
      __threadfence();
      const uint32_t old = atom_add_acq_rel(&p.tickets[t], 1u);
      s.flags[1] = (old == (epoch + 1u) * (uint32_t)n - 1u) ? 1 : 0;
    }
    consumer_sync();
    const bool last = s.flags[1] != 0;
    if (last) __threadfence();
    return last;
  }

  __device__ bool next_tile(int op_idx, uint32_t& slot) {
    slot = T % (uint32_t)p.nslot;
    const uint32_t parity = (T / (uint32_t)p.nslot) & 1u;
    ++T;
    return consumer_all(wait_mbar(p, smem_addr(&s.full[slot]), parity, op_idx, 3));
  }

  // ---------------------------------------------------------------- prologues
  __device__ void norm_prologue(const OpDesc& op, int M) {
    const int H = p.H;
    for (int m = 0; m < M; ++m) {
      float ss = 0.f;
      for (int k = tid; k < H; k += kConsumerThreads) {
        const float v = load_x(p, op, st, m, k);
        s.act[m * H + k] = v;
        ss = fmaf(v, v, ss);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if ((tid & 31) == 0) s.red[tid >> 5] = ss;
      consumer_sync();
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) tot += s.red[w];
      const float rstd = 1.0f / sqrtf(tot / (float)H + p.eps);
      for (int k = tid; k < H; k += kConsumerThreads) {
        const float g = op.norm ? __uint_as_float((uint32_t)__ldg(op.gain + k) << 16) : 1.f;
        s.act[m * H + k] = op.norm ? s.act[m * H + k] * rstd * g : s.act[m * H + k];
      }
      consumer_sync();
    }
  }

  __device__ void copy_prologue(const float* src, int K, int M) {
    for (int i = tid; i < M * K; i += kConsumerThreads) s.act[i] = __ldcg(src + i);
    consumer_sync();
  }

  // ---------------------------------------------------------------- GEMV ops
  __device__ bool gemv_op(int oi, const OpDesc& op, int M) {
    const int C = p.n_ctas, cta = blockIdx.x;
    const int H = p.H;
    // prologue: the activation every tile of this op multiplies
    switch (op.type) {
      case OP_OPROJ:
      case OP_DOWN:
        copy_prologue(op.act, op.K, M);
        break;
      case OP_EXP_DOWN:
        break;  // per slot, below
      default:
        norm_prologue(op, M);  // QKV, gate/up, router, experts, LM head (op.norm = 0: plain copy)
        break;
    }
    if (op.type == OP_ROUTED_GATEUP || op.type == OP_EXP_DOWN) {
      const int* src = op.route;
      int* dst = reinterpret_cast<int*>(s.route);
      for (int i = tid; i < (int)(sizeof(RouteBlock) / 4); i += kConsumerThreads) dst[i] = __ldcg(src + i);
      consumer_sync();
    }
    float best_v = -INFINITY;
    int best_i = 0x7FFFFFFF;
    bool ok = true;

    if (op.type == OP_EXP_DOWN) {
      // x'' = x' + sum over slots of w[m][slot] * (W_down,expert h[slot][m]); each slot's
      // h rows are loaded into act before its tiles, partial sums accumulate in acc[].
      int a, b;
      cta_rows(op.N, op.unit, C, cta, a, b);
      const int I = op.K;
      float* hsl = s.act;                 // [M][I]
      float* accd = s.act + kMmax * I;    // [(b - a)][M]
      for (int t = tid; t < (b - a) * M; t += kConsumerThreads) accd[t] = 0.f;
      const int n_slots = s.route->n_slots;
      for (int sl = 0; sl < n_slots && ok; ++sl) {
        consumer_sync();
        for (int i = tid; i < M * I; i += kConsumerThreads)
          hsl[i] = __ldcg(op.eh + ((size_t)sl * p.Mmax + i / I) * I + i % I);
        consumer_sync();
        for (int r = a; r < b && ok; r += op.rpt) {
          const int nr = min(op.rpt, b - r);
          uint32_t slot;
          if (!next_tile(oi, slot)) { ok = false; break; }
          gemv_any(M, op.wtype, s.ring + (size_t)slot * kSlotBytes, nr, I, op.tpr, hsl, s.red, s.res,
                   smem_addr(&s.empty[slot]), tid);
          for (int t = tid; t < nr * M; t += kConsumerThreads) {
            const int i = t / M, m = t % M;
            accd[(r - a + i) * M + m] += s.route->w[m][sl] * s.res[t];
          }
        }
      }
      consumer_sync();
      if (ok)
        for (int t = tid; t < (b - a) * M; t += kConsumerThreads) {
          const int i = t / M, m = t % M;
          op.x_out[(size_t)m * H + a + i] = load_x(p, op, st, m, a + i) + accd[t];
        }
      if (ok) signal(op.sig_ctr);
      return ok;
    }

    // Row tiles of this CTA: [a, b) within the op's row space.
    const bool experts = op.type == OP_SHARED_GATEUP || op.type == OP_ROUTED_GATEUP;
    int s0 = 0, s1 = 1;
    if (experts) {
      s0 = op.slot0;
      s1 = op.type == OP_SHARED_GATEUP ? op.slot1 : s.route->n_slots;
    }
    int a, b;
    cta_rows((s1 - s0) * op.N, op.unit, C, cta, a, b);
    for (int r = a; r < b && ok;) {
      const int sl = s0 + r / op.N, lr = r % op.N;
      const int nr = min(op.rpt, min(b - r, op.N - lr));
      uint32_t slot;
      if (!next_tile(oi, slot)) { ok = false; break; }
      gemv_any(M, op.wtype, s.ring + (size_t)slot * kSlotBytes, nr, op.K, op.tpr, s.act, s.red, s.res,
               smem_addr(&s.empty[slot]), tid);
      // epilogue on res[i * M + m] for rows lr + i
      switch (op.type) {
        case OP_QKV:
        case OP_ROUTER:
          for (int t = tid; t < nr * M; t += kConsumerThreads)
            op.out[(size_t)(t % M) * op.N + lr + t / M] = s.res[t];
          break;
        case OP_OPROJ:
        case OP_DOWN:
          for (int t = tid; t < nr * M; t += kConsumerThreads) {
            const int i = t / M, m = t % M;
            op.x_out[(size_t)m * H + lr + i] = load_x(p, op, st, m, lr + i) + s.res[t];
          }
          break;
        case OP_GATEUP:
          for (int t = tid; t < (nr / 2) * M; t += kConsumerThreads) {
            const int jj = t / M, m = t % M;
            const float g = s.res[(2 * jj) * M + m], u = s.res[(2 * jj + 1) * M + m];
            op.out[(size_t)m * (op.N / 2) + lr / 2 + jj] = silu(g) * u;
          }
          break;
        case OP_SHARED_GATEUP:
        case OP_ROUTED_GATEUP: {
          const int I = op.N / 2;
          for (int t = tid; t < (nr / 2) * M; t += kConsumerThreads) {
            const int jj = t / M, m = t % M;
            const float g = s.res[(2 * jj) * M + m], u = s.res[(2 * jj + 1) * M + m];
            op.eh[((size_t)sl * p.Mmax + m) * I + lr / 2 + jj] = silu(g) * u;
          }
          break;
        }
        case OP_LMHEAD:
          if (tid < nr * M) {
            const int i = tid / M, m = tid % M;
            const int row = lr + i;
            float v = s.res[tid];
            if (op.wtype == W_FP8) v *= __ldg(static_cast<const float*>(op.ws) + row);
            op.out[(size_t)m * op.N + row] = v;
            if (v > best_v || (v == best_v && row < best_i)) {
              best_v = v;
              best_i = row;
            }
          }
          break;
        default:
          break;
      }
      r += nr;
    }
    if (!ok) return false;

    if (op.type == OP_ROUTER) {
      if (ticket(op.ticket, C)) {
        router_finish(op, M);
        signal(op.sig_ctr);
      }
      return true;
    }
    if (op.type == OP_LMHEAD) {
      lmhead_finish(op, M, best_v, best_i);
      return true;
    }
    signal(op.sig_ctr);
    return true;
  }

  // Last router CTA: top-k per token (largest first, lower index on ties), softmax over the
  // selected logits, union of the experts of the window (shared experts first).
  __device__ void router_finish(const OpDesc& op, int M) {
    const int E = p.E, k = p.top_k;
    float* r = s.act;  // [M][E]
    for (int i = tid; i < M * E; i += kConsumerThreads) r[i] = __ldcg(op.out + (size_t)(i / E) * op.N + i % E);
    consumer_sync();
    RouteBlock* rb = s.route;
    const int warp = tid >> 5, lane = tid & 31;
    for (int m = 0; m < M; ++m) {
      for (int kk = 0; kk < k; ++kk) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
        for (int e = tid; e < E; e += kConsumerThreads) {
          const float v = r[m * E + e];
          if (v > bv || (v == bv && e < bi)) { bv = v; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) {
          s.red[warp] = bv;
          s.flags[4 + warp] = bi;
        }
        consumer_sync();
        if (tid == 0) {
          float v = s.red[0];
          int i = s.flags[4];
          for (int w = 1; w < kConsumerWarps; ++w)
            if (s.red[w] > v || (s.red[w] == v && s.flags[4 + w] < i)) { v = s.red[w]; i = s.flags[4 + w]; }
          rb->topk[m][kk] = i;
          rb->topk_w[m][kk] = v;  // logit for now
          r[m * E + i] = -INFINITY;
        }
        consumer_sync();
      }
    }
    if (tid == 0) {
      for (int m = 0; m < M; ++m) {
        const float mx = rb->topk_w[m][0];
        float sum = 0.f;
        for (int kk = 0; kk < k; ++kk) {
          const float e = expf(rb->topk_w[m][kk] - mx);
          rb->topk_w[m][kk] = e;
          sum += e;
        }
        for (int kk = 0; kk < k; ++kk) rb->topk_w[m][kk] = rb->topk_w[m][kk] / sum;
      }
      int n = 0;
      for (int sh = 0; sh < p.n_shared; ++sh) {
        rb->expert[n] = E + sh;
        for (int m = 0; m < kMmax; ++m) rb->w[m][n] = m < M ? 1.f : 0.f;
        ++n;
      }
      for (int m = 0; m < M; ++m)
        for (int kk = 0; kk < k; ++kk) {
          const int e = rb->topk[m][kk];
          int sl = p.n_shared;
          while (sl < n && rb->expert[sl] != e) ++sl;
          if (sl == n) {
            rb->expert[n] = e;
            for (int mm = 0; mm < kMmax; ++mm) rb->w[mm][n] = 0.f;
            ++n;
          }
          rb->w[m][sl] = rb->topk_w[m][kk];
        }
      rb->n_slots = n;
    }
    consumer_sync();
    int* dst = op.route;
    const int* src = reinterpret_cast<const int*>(rb);
    for (int i = tid; i < (int)(sizeof(RouteBlock) / 4); i += kConsumerThreads) dst[i] = src[i];
  }

  // Block argmax -> per-CTA partial -> last CTA reduces all partials (lowest index on ties).
  __device__ void lmhead_finish(const OpDesc& op, int M, float best_v, int best_i) {
    float* bv = s.act;
    int* bi = reinterpret_cast<int*>(s.act + kConsumerThreads);
    consumer_sync();
    bv[tid] = best_v;
    bi[tid] = best_i;
    consumer_sync();
    if (tid < M) {
      float v = -INFINITY;
      int i = 0x7FFFFFFF;
      for (int t = tid; t < kConsumerThreads; t += M)
        if (bv[t] > v || (bv[t] == v && bi[t] < i)) { v = bv[t]; i = bi[t]; }
      p.am_val[blockIdx.x * kMmax + tid] = v;
      p.am_idx[blockIdx.x * kMmax + tid] = i;
    }
    if (ticket(op.ticket, p.n_ctas)) {
      if (tid < M) {
        float v = -INFINITY;
        int i = 0x7FFFFFFF;
        for (int c = 0; c < p.n_ctas; ++c) {
          const float cv = __ldcg(p.am_val + c * kMmax + tid);
          const int ci = __ldcg(p.am_idx + c * kMmax + tid);
          if (cv > v || (cv == v && ci < i)) { v = cv; i = ci; }
        }
        p.am_out[tid] = i;
      }
    }
  }

  // ---------------------------------------------------------------- attention op
  template <int G_>
  __device__ bool attn_op(int oi, const OpDesc& op, int pos, int M) {
    const int C = p.n_ctas, cta = blockIdx.x;
    const int G = p.G, MG = M * G, ns = p.ns_max, S = pos + M;
    const bool fast = (G_ > 0) && (M == 1);
    const AttnScratch a = attn_scratch(p, s, M);
    const float qscale = 1.4426950408889634f / sqrtf(128.f);  // log2(e) / sqrt(d)
    for (int j = cta; j < p.n_kv * ns; j += C) {
      int head, sidx, p0, p1;
      split_range(S, ns, j, head, sidx, p0, p1);
      // rotated, scaled queries of the group
      for (int idx = tid; idx < MG * 64; idx += kConsumerThreads) {
        const int mh = idx >> 6, i = idx & 63;
        const int m = mh / G, h = head * G + mh % G;
        const float* qr = op.act + (size_t)m * p.qkv_rows + h * 128;
        const float x1 = __ldcg(qr + i), x2 = __ldcg(qr + i + 64);
        const float2 cs = s.rope[m * 64 + i];
        a.q[mh * 128 + i] = (x1 * cs.x - x2 * cs.y) * qscale;
        a.q[mh * 128 + i + 64] = (x1 * cs.y + x2 * cs.x) * qscale;
      }
      if (tid < MG) {
        a.mrun[tid] = -INFINITY;
        a.lrun[tid] = 0.f;
      }
      O1<(G_ > 0 ? G_ : 1)> o1;
      OGen og;
#pragma unroll
      for (int h = 0; h < (G_ > 0 ? G_ : 1); ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) o1.o[h][e] = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) og.o[k][0] = og.o[k][1] = 0.f;
      consumer_sync();

      auto tile = [&](const uint8_t* kr, const uint8_t* vr, int n, int vis_base, uint32_t eb) {
        if (fast)
          attn_scores<(G_ > 0 ? G_ : 1)>(kr, n, a, 0, MG, tid);
        else if (MG % 5 == 0)
          for (int mh0 = 0; mh0 < MG; mh0 += 5) attn_scores<5>(kr, n, a, mh0, MG, tid);
        else
          for (int mh0 = 0; mh0 < MG; mh0 += 4) attn_scores<4>(kr, n, a, mh0, MG, tid);
        consumer_sync();
        attn_softmax(a, n, M, G, vis_base, tid);
        consumer_sync();
        if (fast)
          attn_values_m1<(G_ > 0 ? G_ : 1)>(o1, vr, n, a, tid);
        else
          attn_values_generic(og, vr, n, a, MG, tid);
        if (eb) {
          __syncwarp();
          if ((tid & 31) == 0) mbar_arrive(eb);
        }
        consumer_sync();
      };

      // cached rows [p0, min(p1, pos)) arrive through the ring
      const int ce = min(p1, pos);
      for (int q = p0; q < ce; q += kAttnTilePos) {
        const int n = min(kAttnTilePos, ce - q);
        uint32_t slot;
        if (!next_tile(oi, slot)) return false;
        const uint8_t* base = s.ring + (size_t)slot * kSlotBytes;
        tile(base, base + n * 256, n, -1, smem_addr(&s.empty[slot]));
      }
      // this call's own rows [max(p0, pos), p1): rotate k, round k and v to bf16, append them
      // to the cache (the new rows of the KV history), then attend to them causally
      const int nb = max(p0, pos);
      if (nb < p1) {
        const int nn = p1 - nb;
        uint16_t* kn = reinterpret_cast<uint16_t*>(a.kvnew);
        uint16_t* vn = kn + nn * 128;
        for (int idx = tid; idx < nn * 64; idx += kConsumerThreads) {
          const int r = idx >> 6, i = idx & 63;
          const int m = nb - pos + r;
          const float* kr = op.act + (size_t)m * p.qkv_rows + (p.n_q + head) * 128;
          const float* vr = op.act + (size_t)m * p.qkv_rows + (p.n_q + p.n_kv + head) * 128;
          const float k1 = __ldcg(kr + i), k2 = __ldcg(kr + i + 64);
          const float2 cs = s.rope[m * 64 + i];
          const __nv_bfloat16 r1 = __float2bfloat16_rn(k1 * cs.x - k2 * cs.y);
          const __nv_bfloat16 r2 = __float2bfloat16_rn(k1 * cs.y + k2 * cs.x);
          const __nv_bfloat16 v1 = __float2bfloat16_rn(__ldcg(vr + i));
          const __nv_bfloat16 v2 = __float2bfloat16_rn(__ldcg(vr + i + 64));
          const uint16_t b1 = __bfloat16_as_ushort(r1), b2 = __bfloat16_as_ushort(r2);
          const uint16_t c1 = __bfloat16_as_ushort(v1), c2 = __bfloat16_as_ushort(v2);
          kn[r * 128 + i] = b1;
          kn[r * 128 + i + 64] = b2;
          vn[r * 128 + i] = c1;
          vn[r * 128 + i + 64] = c2;
          const size_t off = ((size_t)head * p.cap + pos + m) * kHeadDim;
          op.kc[off + i] = b1;
          op.kc[off + i + 64] = b2;
          op.vc[off + i] = c1;
          op.vc[off + i + 64] = c2;
        }
        consumer_sync();
        tile(a.kvnew, a.kvnew + nn * 256, nn, nb - pos, 0u);
      }
      // split partial: (running max, running sum, unnormalised output) per (m, h)
      float* part = p.part + (size_t)(head * ns + sidx) * p.Mmax * G * 130;
      if (tid < MG) {
        part[tid * 130] = a.mrun[tid];
        part[tid * 130 + 1] = a.lrun[tid];
      }
      if (fast) {
        const int c = tid & 15, pc = tid >> 4;
        for (int h = 0; h < G; ++h) {
#pragma unroll
          for (int hh = 0; hh < (G_ > 0 ? G_ : 1); ++hh)
            if (hh == h)
#pragma unroll
              for (int e = 0; e < 8; ++e) a.ored[pc * 128 + c * 8 + e] = o1.o[hh][e];
          consumer_sync();
          if (tid < 128) {
            float t = 0.f;
            for (int q = 0; q < 16; ++q) t += a.ored[q * 128 + tid];
            part[h * 130 + 2 + tid] = t;
          }
          consumer_sync();
        }
      } else {
        const int dp = tid & 63, hs = tid >> 6;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int mh = hs + 4 * k;
          if (mh < MG) {
            part[mh * 130 + 2 + 2 * dp] = og.o[k][0];
            part[mh * 130 + 2 + 2 * dp + 1] = og.o[k][1];
          }
        }
      }
      // the last split of this kv head merges all of them (log-sum-exp in base 2)
      if (ticket(op.ticket + head, ns)) {
        const float* hp = p.part + (size_t)(head * ns) * p.Mmax * G * 130;
        const size_t sstride = (size_t)p.Mmax * G * 130;
        const int warp = tid >> 5, lane = tid & 31;
        for (int mh = warp; mh < MG; mh += kConsumerWarps) {
          float mx = -INFINITY;
          for (int q = lane; q < ns; q += 32) mx = fmaxf(mx, __ldcg(hp + q * sstride + mh * 130));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          float l = 0.f;
          for (int q = lane; q < ns; q += 32) {
            const float mq = __ldcg(hp + q * sstride + mh * 130);
            const float w = mq == -INFINITY ? 0.f : exp2f(mq - mx);
            a.cw[mh * ns + q] = w;
            l += w * __ldcg(hp + q * sstride + mh * 130 + 1);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
          const float inv = 1.0f / l;
          for (int q = lane; q < ns; q += 32) a.cw[mh * ns + q] *= inv;
        }
        consumer_sync();
        for (int idx = tid; idx < MG * 128; idx += kConsumerThreads) {
          const int mh = idx >> 7, d = idx & 127;
          float o = 0.f;
          for (int q = 0; q < ns; ++q) o = fmaf(a.cw[mh * ns + q], __ldcg(hp + q * sstride + mh * 130 + 2 + d), o);
          const int m = mh / G, h = head * G + mh % G;
          op.out[(size_t)m * p.n_q * 128 + h * 128 + d] = o;
        }
        signal(op.sig_ctr);
      }
    }
    return true;
  }

  // ---------------------------------------------------------------- main loop
  __device__ bool run(int pos, int M) {
    for (int oi = p.op_begin; oi < p.op_end; ++oi) {
      {
        const int* src = reinterpret_cast<const int*>(p.ops + oi);
        int* dst = reinterpret_cast<int*>(s.op);
        for (int i = tid; i < (int)(sizeof(OpDesc) / 4); i += kConsumerThreads) dst[i] = __ldg(src + i);
      }
      consumer_sync();
      const OpDesc& op = *s.op;
      if (!wait_dep(op.wait_ctr, op.wait_n, oi, 4)) return false;
      if (!wait_dep(op.wait2_ctr, op.wait2_n, oi, 5)) return false;
      bool ok;
      if (op.type == OP_ATTN) {
        if (p.G == 5)
          ok = attn_op<5>(oi, op, pos, M);
        else if (p.G == 4)
          ok = attn_op<4>(oi, op, pos, M);
        else
          ok = attn_op<0>(oi, op, pos, M);
      } else {
        ok = gemv_op(oi, op, M);
      }
      if (!ok) return false;
      consumer_sync();
    }
    if (p.op_end == p.n_ops) {
      // step end: the last CTA advances the step state (and feeds the argmax back if chained)
      if (ticket(p.step_ticket, p.n_ctas) && tid == 0) {
        StepState* g = p.state;
        if (st.chain) {
          const int tok = __ldcg(p.am_out);
          if (st.gen_out) st.gen_out[st.gen_idx] = tok;
          g->gen_idx = st.gen_idx + 1;
          g->tokens[0] = tok;
          g->pos = st.pos + 1;
        }
        __threadfence();
        g->epoch = epoch + 1u;
      }
    }
    return true;
  }
};

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kThreads, 1) dec_megakernel(const KParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem s = carve(smem_raw, p);
  const int tid = threadIdx.x;
  __shared__ StepState st;
  if (tid == 0) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.state);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&st);
    for (int i = 0; i < (int)(sizeof(StepState) / 4); ++i) dst[i] = __ldcg(src + i);
    for (int i = 0; i < p.nslot; ++i) {
      mbar_init(smem_addr(&s.full[i]), 1);
      mbar_init(smem_addr(&s.empty[i]), kConsumerWarps);
    }
    mbar_init_fence();
  }
  __syncthreads();
  const uint32_t epoch = st.epoch;
  const int pos = st.pos, M = st.m;

  if (tid >= kConsumerThreads) {
    if (tid == kConsumerThreads) {
      Producer pr{p, s, 0u, true};
      pr.run(epoch, pos, M);
    }
    return;
  }
  // RoPE table of this call's positions (fp64 angle, then fp32 cos/sin).
  if (tid < M * 64) {
    const int m = tid >> 6, i = tid & 63;
    const double inv = pow((double)p.rope_base, -2.0 * (double)i / 128.0);
    double sn, cs;
    sincos((double)(pos + m) * inv, &sn, &cs);
    s.rope[tid] = make_float2((float)cs, (float)sn);
  }
  consumer_sync();
  Consumer c{p, s, 0u, epoch, st, tid};
  c.run(pos, M);
}

}  // namespace decimpl

// ------------------------------------------------------------------ host launch
extern "C" cudaError_t dec_launch_megakernel(const decimpl::KParams* kp, int cooperative, cudaStream_t stream) {
  using namespace decimpl;
  const size_t smem = (size_t)kp->nslot * kSlotBytes + kp->act_bytes + kCommonBytes;
  static size_t attr_bytes = 0;  // largest dynamic size the kernel has been allowed so far
  if (smem > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(dec_megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_bytes = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)kp->n_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = cooperative ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dec_megakernel, *kp);
}

extern "C" size_t dec_megakernel_smem_bytes(int nslot, int act_bytes) {
  return (size_t)nslot * decimpl::kSlotBytes + (size_t)act_bytes + decimpl::kCommonBytes;
}

// Common area plus the kernel's static shared memory, which the dynamic part must leave room for.
extern "C" int dec_megakernel_common_bytes(void) { return decimpl::kCommonBytes + 2048; }
