// The persistent decode megakernel for sm_103a.
//
// One CTA per SM: 7 consumer warps and 1 producer warp. Every CTA walks the step's op list
// (Muse Spark Open megakernel article, section "the baseline nobody benchmarked": one
// resident kernel whose warps start the next op before the previous one retires). For each op
// a CTA owns a contiguous share of the op's rows (or of the attention positions) and splits it
// again among its consumer warps. Each consumer warp has its own ring of kStages slots. Lane w
// of the producer warp streams consumer warp w's tiles of weights / cached keys and values
// into that warp's slots with bulk asynchronous copies (the TMA engine's non-tensor mode); it
// never waits for activations -- weights and KV history do not depend on the running step --
// so it runs ahead across op boundaries and the next op's bytes are in flight while the
// previous op is still finishing on other SMs (same article, section "three bills": a per-SM
// ring of weight slots that already holds the next op's first tiles).
//
// Activations move between SMs as tagged 64-bit words (value + step tag, see ptx.cuh): an op's
// prologue polls exactly the data it needs, so a hand-off costs one L2 round trip and no
// fence (a fence with bulk copies in flight costs microseconds). Within an op a warp computes
// its tiles with no CTA-wide barrier. Every wait is bounded by %globaltimer: on expiry the
// waiting thread records the failure in the status word and raises the global abort flag;
// every other wait sees the flag, copies in flight land, and the kernel returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "../../include/dec.h"
#include "dec_internal.h"
#include "gemv.cuh"
#include "ptx.cuh"
#include "smem_attr.h"

namespace decimpl {

#ifdef DEC_TRACE
#define TRACE(p, oi, field, value)                                                                       \
  do {                                                                                                   \
    if ((p).trace) (p).trace[((size_t)blockIdx.x * (p).n_ops + (oi)) * kTraceFields + (field)] = (value); \
  } while (0)
#else
#define TRACE(p, oi, field, value) \
  do {                             \
  } while (0)
#endif

// ------------------------------------------------------------------ shared memory map
constexpr int kCommonBytes = 9728;
constexpr int kOffFull = 0, kOffEmpty = 256, kOffOp = 512, kOffRed = 1024, kOffResW = 3072, kOffRope = 5120,
              kOffFlags = 7168, kOffRoute = 7232, kOffNTiles = 8192;
constexpr int kFlagTicket = 1;  // flags[kFlagTicket]: verdict of the last ticket
constexpr int kFlagLate = 2;    // flags[kFlagLate]: input words re-polled in this op (DEC_TRACE)
constexpr int kFlagRoute = 8;   // flags[kFlagRoute]: route_tag of the routing that sits in `route`
static_assert(kConsumerWarps * kStages * 8 <= kOffEmpty - kOffFull, "full barriers");
static_assert(sizeof(OpDesc) <= kOffRed - kOffOp, "OpDesc copy");
static_assert(kOffRoute + sizeof(RouteBlock) <= kOffNTiles, "routing block");
static_assert(kOffNTiles + 4 * kConsumerWarps <= kCommonBytes, "common area");

struct Smem {
  uint8_t* ring;        // [warp][stage][slot_bytes]
  float* act;           // op scratch: activations [M][K], residual rows, attention state ...
  uint64_t* full;       // [warp][stage]
  uint64_t* empty;      // [warp][stage]
  OpDesc* op;           // consumer copy of the current op
  float* red;           // [8][64] cross-warp scratch
  float* resw;          // [8][64] per-warp scratch
  float2* rope;         // [kMmax][64] (cos, sin) at pos + m
  volatile int* flags;  // [16]
  RouteBlock* route;    // this CTA's routing of the current MoE layer
  uint32_t* ntiles;     // [warp] tiles each consumer warp has taken from its ring
  int slot_bytes;
  __device__ __forceinline__ uint8_t* slot(int w, int st) const {
    return ring + ((size_t)w * kStages + st) * slot_bytes;
  }
};

__device__ __forceinline__ Smem carve(uint8_t* base, const KParams& p) {
  Smem s;
  const size_t ring = (size_t)kConsumerWarps * kStages * p.slot_bytes;
  s.ring = base;
  s.act = reinterpret_cast<float*>(base + ring);
  uint8_t* c = base + ring + p.act_bytes;
  s.full = reinterpret_cast<uint64_t*>(c + kOffFull);
  s.empty = reinterpret_cast<uint64_t*>(c + kOffEmpty);
  s.op = reinterpret_cast<OpDesc*>(c + kOffOp);
  s.red = reinterpret_cast<float*>(c + kOffRed);
  s.resw = reinterpret_cast<float*>(c + kOffResW);
  s.rope = reinterpret_cast<float2*>(c + kOffRope);
  s.flags = reinterpret_cast<volatile int*>(c + kOffFlags);
  s.route = reinterpret_cast<RouteBlock*>(c + kOffRoute);
  s.ntiles = reinterpret_cast<uint32_t*>(c + kOffNTiles);
  s.slot_bytes = p.slot_bytes;
  return s;
}

// The dynamic shared memory and the step state every device function of the kernel can reach:
// out-of-line functions rebuild their context from these, the grid-constant parameters and the
// thread index, so no per-thread state ever travels through local memory.
extern __shared__ __align__(1024) uint8_t smem_raw[];
__shared__ StepState g_st;  // copied in by the kernel's first thread

// ------------------------------------------------------------------ failure handling
__device__ __forceinline__ bool aborted(const KParams& p) {
  return *reinterpret_cast<volatile uint32_t*>(&p.status->abort) != 0u;
}

__device__ __noinline__ void raise_error(const KParams& p, uint32_t code, int op, uint32_t ctr, uint32_t obs,
                                         uint32_t tgt, uint32_t where) {
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

__device__ __noinline__ bool wait_mbar_slow(const KParams& p, uint32_t bar, uint32_t parity, int op, uint32_t where) {
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

__device__ __forceinline__ bool wait_mbar(const KParams& p, uint32_t bar, uint32_t parity, int op, uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_mbar_slow(p, bar, parity, op, where);
}

// Spin until the arrival counter reaches target (wrap-safe), bounded like every wait.
__device__ __noinline__ bool wait_counter_slow(const KParams& p, const uint32_t* c, uint32_t target, int op,
                                               uint32_t where) {
  const uint64_t t0 = gtimer();
  for (int it = 1;; ++it) {
    const uint32_t v = ld_relaxed(c);
    if ((int32_t)(v - target) >= 0) return true;
    if ((it & 15) == 0) {
      if (aborted(p)) return false;
      if (gtimer() - t0 > p.timeout_ns) {
        raise_error(p, DEC_ERR_TIMEOUT, op, (uint32_t)(c - p.ctr), v, target, where);
        return false;
      }
    }
  }
}

#ifndef DEC_STREAM_EVICT_FIRST
#define DEC_STREAM_EVICT_FIRST 1  // weights / KV history stream through L2 as evict-first
#endif
#ifndef DEC_L2_AHEAD
#define DEC_L2_AHEAD 4  // tiles per warp the producer asks L2 for beyond its ring while the ring waits
#endif
#ifndef DEC_POLL_DATA
#define DEC_POLL_DATA 1  // 1: no arrival counts: consumers poll the tagged inputs directly
#endif
#ifndef DEC_ORDERED_ARRIVALS
#define DEC_ORDERED_ARRIVALS 0  // 1: release/acquire arrivals (data visible when the count is)
#endif
#ifndef DEC_POLL_BACKOFF_NS
#define DEC_POLL_BACKOFF_NS 0  // pause before re-reading words whose tag is not current yet
#endif
#ifndef DEC_GATHER_U
#define DEC_GATHER_U 1  // 4-word items each thread keeps in flight when loading an op's input
#endif
constexpr int kGatherU = DEC_GATHER_U;
#ifndef DEC_COPY_U
#define DEC_COPY_U 1  // the same for the o-proj / down-projection inputs (up to 6912 words a token)
#endif
constexpr int kCopyU = DEC_COPY_U;

// One item of W tagged words (W = 2 or 4: 16-byte aligned).
template <int W>
__device__ __forceinline__ void ld_item(const uint64_t* s, uint64_t (&w)[W]) {
  if constexpr (W == 1) {
    w[0] = ld_tagged(s);
  } else {
    ld_tagged2(s, w[0], w[1]);
    if constexpr (W == 4) ld_tagged2(s + 2, w[2], w[3]);
  }
}

// Re-poll one item of W tagged words until every word carries `tag` (values into out), bounded
// like every wait. Out of line: it runs only for the rare word still in flight after its
// producers' arrival count was seen.
template <int W>
__device__ __noinline__ bool poll_item_slow(const KParams& p, const uint64_t* src, float* out, uint32_t tag, int op,
                                            uint32_t where) {
  const uint64_t t0 = gtimer();
  for (int it = 1;; ++it) {
    uint64_t w[W];
    ld_item<W>(src, w);
    bool good = true;
    for (int k = 0; k < W; ++k) good &= tag_of(w[k]) == tag;
    if (good) {
      for (int k = 0; k < W; ++k) out[k] = value_of(w[k]);
      return true;
    }
#if DEC_POLL_BACKOFF_NS > 0
    __nanosleep(DEC_POLL_BACKOFF_NS);
#endif
    if ((it & 7) == 0) {
      if (aborted(p)) return false;
      if (gtimer() - t0 > p.timeout_ns) {
        raise_error(p, DEC_ERR_TIMEOUT, op, 0x40000000u, tag_of(w[0]), tag, where);
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

// Rows [aw, bw) of the CTA's [a, b) owned by consumer warp w.
__device__ __forceinline__ void warp_rows(int a, int b, int unit, int w, int& aw, int& bw) {
  const int U = (b - a) / unit;
  aw = a + (U * w / kConsumerWarps) * unit;
  bw = a + (U * (w + 1) / kConsumerWarps) * unit;
}

// Attention: every kv head has ns splits of the positions [0, S), S = pos + M.
__device__ __forceinline__ void split_range(int lo, int S, int ns, int j, int& head, int& s, int& p0, int& p1) {
  head = j / ns;
  s = j % ns;
  p0 = lo + (int)((long long)(S - lo) * s / ns);
  p1 = lo + (int)((long long)(S - lo) * (s + 1) / ns);
}

// First cached position a call's attention reads: with a sliding window of W positions the
// call's first token (at pos) sees pos - W + 1 .. pos; 0 for global attention.
__device__ __forceinline__ int attn_lo(const KParams& p, int pos) {
  return p.attn_window > 0 ? max(0, pos - p.attn_window + 1) : 0;
}

// Warps serving token m of an M-token window: m, m + M, ...; this warp is number gi of ng.
__device__ __forceinline__ void token_group(int w, int M, int& m, int& gi, int& ng) {
  m = w % M;
  gi = w / M;
  ng = (kConsumerWarps - m + M - 1) / M;
}

__device__ __forceinline__ int bytes_per_col(int wtype) { return wtype == W_BF16 ? 2 : 1; }  // MXFP4: K/2 below

// KV rows of one attention tile: fixed for tensor-core tiles, else what a ring slot holds.
__device__ __forceinline__ int attn_rows(const KParams& p, int slot_bytes) {
  return p.attn_tc ? kAttnTcRows : attn_rows_per_slot(slot_bytes, p.kv_fp8);
}

__device__ __forceinline__ int row_bytes(int wtype, int K) {
  return wtype == W_BF16 ? 2 * K : (wtype == W_FP8 ? K : K / 2);
}

// Token m's activations k .. k+3 (k a multiple of 4) as the B operand of the tensor-core GEMV
// (m16n8k16, eight columns): 16-column step k / 16, lane 4 g + t holds columns g = m (bf16 high
// parts) and g = m + 4 (the residues), rows 2t, 2t+1 in its first register, 2t+8, 2t+9 in its
// second. 256 bytes per step: the same bytes as kMmax tokens of fp32.
__device__ __forceinline__ void put_bfrag(float* act, int m, int k, float4 x) {
  uint32_t* bf = reinterpret_cast<uint32_t*>(act);
  const int kk = k >> 4, c = k & 15, reg = c >> 3, t0 = (c & 7) >> 1;
  const float v[4] = {x.x, x.y, x.z, x.w};
  float hi[4], lo[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    hi[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
    lo[e] = v[e] - hi[e];
  }
  bf[((kk * 32 + 4 * m + t0) << 1) + reg] = pack_bf16x2(hi[0], hi[1]);
  bf[((kk * 32 + 4 * m + t0 + 1) << 1) + reg] = pack_bf16x2(hi[2], hi[3]);
  bf[((kk * 32 + 4 * (m + 4) + t0) << 1) + reg] = pack_bf16x2(lo[0], lo[1]);
  bf[((kk * 32 + 4 * (m + 4) + t0 + 1) << 1) + reg] = pack_bf16x2(lo[2], lo[3]);
}

struct Tile {
  int mat;       // expert id (expert ops), kv head (attention), else 0
  int sl;        // expert slot (expert ops), split index (attention)
  int r0, nr;    // rows (matrix ops) or positions (attention)
  int kc, kn;    // column chunk
  bool last_k;   // last column chunk of the row group
};

// Per-warp tile sequence of a matrix op; the producer and the consumer walk it identically.
struct GemvIter {
  int mode;      // 0: one matrix; 1: expert gate/up (rows run across slots); 2: expert down (slots
                 // outer); 3: column split (every warp covers all of the CTA's rows, warp w columns
                 // [kw0, kw1)); 4: expert down, slot split (the CTA's rows of every slot cut into
                 // nch chunks of R rows; warp w takes items w, w + 7, ... of slot-major order)
  int N, K, R, Kc;
  int aw, bw, s0, s1;
  int r, kc, sl;
  int kw0, kw1;
  int nch, item;
  const int* experts;  // expert id per slot (routed ops); null: expert id = mat_base + slot
  int mat_base;

  __device__ __forceinline__ void init(const OpDesc& op, int C, int cta, int w, int n_slots, const int* expert_ids, int base) {
    mat_base = base;
    N = op.N;
    K = op.K;
    R = op.R;
    Kc = op.Kc;
    experts = expert_ids;
    if (op.type == OP_ROUTED_GATEUP)
      mode = 1;
    else if (op.type == OP_EXP_DOWN)
      mode = op.csplit ? 4 : 2;
    else
      mode = op.csplit ? 3 : 0;
    s0 = 0;
    s1 = 1;
    if (mode == 1) {
      s0 = op.slot0;
      s1 = n_slots;
    } else if (mode == 2 || mode == 4) {
      s1 = n_slots;
    }
    int a, b;
    cta_rows(mode == 1 ? (s1 - s0) * N : N, op.unit, C, cta, a, b);
    nch = 0;
    item = w;
    if (mode == 4) {
      aw = a;
      bw = b;
      nch = b > a ? (b - a + R - 1) / R : 0;
      kw0 = kw1 = 0;
    } else if (mode == 3) {
      aw = a;
      bw = b;
      const int kwid = op.kw ? op.kw : Kc;  // this warp's columns, walked in tiles of Kc
      kw0 = min(K, w * kwid);
      kw1 = w == kConsumerWarps - 1 ? K : min(K, kw0 + kwid);
    } else {
      warp_rows(a, b, op.unit, w, aw, bw);
      kw0 = kw1 = 0;
    }
    r = aw;
    kc = 0;
    sl = 0;
  }

  __device__ __forceinline__ bool next(Tile& t) {
    if (mode == 4) {
      if (item >= (s1 - s0) * nch) return false;
      const int slot = s0 + item / nch, c = item % nch;
      t.mat = experts ? experts[slot] : mat_base + slot;
      t.sl = slot;
      t.r0 = aw + c * R;
      t.nr = min(R, bw - t.r0);
      t.kc = 0;
      t.kn = K;
      t.last_k = true;
      item += kConsumerWarps;
      return true;
    }
    if (mode == 3) {
      if (r >= bw || kw0 >= kw1) return false;
      t.mat = 0;
      t.sl = 0;
      t.r0 = r;
      t.nr = min(R, bw - r);
      t.kc = kw0 + kc;
      t.kn = min(Kc, kw1 - t.kc);
      t.last_k = t.kc + t.kn >= kw1;
      kc += t.kn;
      if (t.last_k) {
        kc = 0;
        r += t.nr;
      }
      return true;
    }
    if (mode == 2) {
      while (sl < s1 && r >= bw) {
        ++sl;
        r = aw;
      }
      if (sl >= s1 || aw >= bw) return false;
      t.mat = experts ? experts[sl] : mat_base + sl;
      t.sl = sl;
      t.r0 = r;
      t.nr = min(R, bw - r);
    } else {
      if (r >= bw) return false;
      if (mode == 1) {
        const int slot = s0 + r / N, lr = r % N;
        t.mat = experts ? experts[slot] : mat_base + slot;
        t.sl = slot;
        t.r0 = lr;
        t.nr = min(R, min(bw - r, N - lr));
      } else {
        t.mat = 0;
        t.sl = 0;
        t.r0 = r;
        t.nr = min(R, bw - r);
      }
    }
    t.kc = kc;
    t.kn = min(Kc, K - kc);
    t.last_k = kc + t.kn >= K;
    kc += t.kn;
    if (t.last_k) {
      kc = 0;
      r += t.nr;
    }
    return true;
  }
};

// Per-warp tile sequence of the attention op: the CTA's splits j = cta, cta + C, ...; within a
// split the warps of token m share the cached positions [p0, min(p1, pos)).
struct AttnIter {
  int C, S, ns, nsplit, pos, P;
  int lo;  // first position any token of the call attends to (a sliding window's start)
  int gi, ng;
  int j, q, qe, head;
  bool fresh;

  __device__ __forceinline__ void init(const KParams& p, int cta, int w, int pos_, int M, int P_) {
    C = p.n_ctas;
    pos = pos_;
    S = pos + M;
    lo = attn_lo(p, pos);
    ns = p.ns_max;
    nsplit = p.n_kv * ns;
    P = P_;
    int m;
    token_group(w, M, m, gi, ng);
    j = cta;
    fresh = true;
  }

  __device__ __forceinline__ void enter_split() {
    int s, p0, p1;
    split_range(lo, S, ns, j, head, s, p0, p1);
    const int ce = max(p0, min(p1, pos));
    q = p0 + (int)((long long)(ce - p0) * gi / ng);
    qe = p0 + (int)((long long)(ce - p0) * (gi + 1) / ng);
    fresh = false;
  }

  // Next tile of the current split only (the consumer steps splits itself).
  __device__ __forceinline__ bool next_in_split(Tile& t) {
    if (fresh) enter_split();
    if (q >= qe) return false;
    t.mat = head;
    t.sl = j;
    t.r0 = q;
    t.nr = min(P, qe - q);
    q += t.nr;
    return true;
  }

  __device__ __forceinline__ bool next_split() {
    j += C;
    fresh = true;
    return j < nsplit;
  }

  // Producer: next tile across splits.
  __device__ __forceinline__ bool next(Tile& t) {
    while (j < nsplit) {
      if (next_in_split(t)) return true;
      next_split();
    }
    return false;
  }
};

// ------------------------------------------------------------------ producer warp
// Lane w of the producer warp streams consumer warp w's tiles into that warp's ring slots:
// its cursor (op, tile iterator, tiles issued) lives in the lane's registers and runs ahead
// across op boundaries, so the next op's first tiles are in flight while the consumers poll
// for that op's input. The lanes advance together (SIMT), each issuing when its warp has a
// free slot; a lane stalls only at a routed-expert op until this CTA's consumers have computed
// the layer's routing.
// Greedy steps one launch runs (at least one).
__device__ __forceinline__ int steps_of(const KParams& p) { return p.n_steps > 1 ? p.n_steps : 1; }

// Tag of one MoE layer's routing within one step (epoch: the step's count of completed steps):
// steps that run in one launch route the same layers again.
__device__ __forceinline__ int route_tag(uint32_t epoch, int layer, int L) {
  return (int)((epoch * (uint32_t)(L + 1) + (uint32_t)layer + 1u) & 0x7FFFFFFFu);
}

struct LaneCursor {
  int oi, started;
  int step;    // step of the launch the cursor is in (pos + step, epoch0 + step)
  uint32_t n;  // tiles issued to this lane's warp
  GemvIter g;
  AttnIter a;
};

struct Producer {
  const KParams& p;
  Smem& s;
  int pos, M;       // of the launch's first step; step k decodes at pos + k
  uint64_t policy;  // L2 policy of the streamed bytes
  uint32_t epoch0;  // completed steps when the launch began

  __device__ __forceinline__ void stream(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
#if DEC_STREAM_EVICT_FIRST
    bulk_g2s_hint(dst, src, bytes, bar, policy);
#else
    bulk_g2s(dst, src, bytes, bar);
#endif
  }

  // Expert ids of the current MoE layer's routing, once the consumers have published it.
  __device__ __forceinline__ const int* routing(const OpDesc* op, int step) {
    if (s.flags[kFlagRoute] != route_tag(epoch0 + (uint32_t)step, __ldg(&op->layer), p.L)) return nullptr;
    __threadfence_block();
    return s.route->expert;
  }

  __device__ __forceinline__ void copy_gemv(const OpDesc* op, const Tile& t, uint8_t* dst, uint32_t fb) {
    if (__ldg(&op->tc)) {
      // tensor-core tile: boxes of kGemvTcRows rows x 64 columns, 128-byte swizzle, always whole
      // (rows past the tile are the next rows of the matrix, or zeros past its end; unused)
      const int nb = t.kn / 64;
      const CUtensorMap* tm = op->tmap;
      mbar_expect_tx(fb, (uint32_t)(nb * kGemvTcRows * 128));
      const uint32_t d = smem_addr(dst);
      for (int b = 0; b < nb; ++b) tma_load_2d(d + b * kGemvTcRows * 128, tm, t.kc + 64 * b, t.r0, fb, policy);
      return;
    }
    const int wtype = __ldg(&op->wtype), K = __ldg(&op->K);
    const int rb = row_bytes(wtype, K);
    const char* base = static_cast<const char*>(op->w) + (size_t)t.mat * __ldg(&op->w_mstride);
    const int cb = wtype == W_MXFP4 ? t.kn / 2 : t.kn * bytes_per_col(wtype);  // bytes of one row chunk
    const int koff = wtype == W_MXFP4 ? t.kc / 2 : t.kc * bytes_per_col(wtype);
    const uint32_t total = (uint32_t)(cb * t.nr);
    const uint32_t sbytes = wtype == W_MXFP4 ? (uint32_t)(t.nr * (t.kn / 32)) : 0u;
    mbar_expect_tx(fb, total + sbytes);
    const uint32_t d = smem_addr(dst);
    if (t.kn == K) {
      stream(d, base + (size_t)t.r0 * rb, total, fb);
    } else {
      for (int i = 0; i < t.nr; ++i) stream(d + i * cb, base + (size_t)(t.r0 + i) * rb + koff, (uint32_t)cb, fb);
    }
    if (sbytes) {
      const int K32 = K / 32;
      const char* sb = static_cast<const char*>(op->ws) + (size_t)t.mat * __ldg(&op->ws_mstride);
      const uint32_t d2 = d + ((total + 15u) & ~15u);
      if (t.kn == K) {
        stream(d2, sb + (size_t)t.r0 * K32, sbytes, fb);
      } else {
        for (int i = 0; i < t.nr; ++i)
          stream(d2 + i * (t.kn / 32), sb + (size_t)(t.r0 + i) * K32 + t.kc / 32, (uint32_t)(t.kn / 32), fb);
      }
    }
  }

  __device__ __forceinline__ void copy_attn(const OpDesc* op, const Tile& t, uint8_t* dst, uint32_t fb) {
    if (p.attn_tc) {
      // four boxes of kAttnTcRows rows x 64 columns, 128-byte swizzle: keys 0-63, keys 64-127,
      // values 0-63, values 64-127. Always whole boxes: rows past the tile belong to later
      // positions (or, past the cache, are filled with zeros) and are masked by the consumer.
      const int y = (__ldg(&op->layer) * p.n_kv + t.mat) * p.cap + t.r0;
      mbar_expect_tx(fb, 4u * kAttnTcBoxBytes);
      const uint32_t d = smem_addr(dst);
      tma_load_2d(d, &p.tmap_k, 0, y, fb, policy);
      tma_load_2d(d + kAttnTcBoxBytes, &p.tmap_k, 64, y, fb, policy);
      tma_load_2d(d + 2 * kAttnTcBoxBytes, &p.tmap_v, 0, y, fb, policy);
      tma_load_2d(d + 3 * kAttnTcBoxBytes, &p.tmap_v, 64, y, fb, policy);
      return;
    }
    const int rb = kv_row_bytes(p.kv_fp8);
    const uint32_t bytes = (uint32_t)(t.nr * rb);
    const size_t off = ((size_t)t.mat * p.cap + t.r0) * rb;  // bytes
    mbar_expect_tx(fb, 2u * bytes);
    const uint32_t d = smem_addr(dst);
    // a chained launch reads rows that its own earlier steps appended with plain stores; the
    // step-end rendezvous orders them before this lane's slot hand-back, this fence before the copy
    if (p.n_steps > 1) fence_proxy_async_global();
    stream(d, op->kc + off, bytes, fb);
    stream(d + bytes, op->vc + off, bytes, fb);
  }

  // Ask L2 for the bytes a tile will bring (cp.async.bulk.prefetch: no completion to wait for).
  // Sizes are multiples of 16 bytes and starts 16-byte aligned, like the copies themselves; the
  // MXFP4 scale run is rounded down (its last bytes come with the copy).
  __device__ __forceinline__ void prefetch_tile(const OpDesc* op, int type, const Tile& t) {
    if (type == OP_ATTN) {
      const int rb = kv_row_bytes(p.kv_fp8);
      const uint32_t bytes = (uint32_t)(t.nr * rb);
      const size_t off = ((size_t)t.mat * p.cap + t.r0) * rb;  // bytes
      prefetch_l2(op->kc + off, bytes);
      prefetch_l2(op->vc + off, bytes);
      return;
    }
    const int wtype = __ldg(&op->wtype), K = __ldg(&op->K);
    const int rb = row_bytes(wtype, K);
    const char* base = static_cast<const char*>(op->w) + (size_t)t.mat * __ldg(&op->w_mstride);
    const int cb = wtype == W_MXFP4 ? t.kn / 2 : t.kn * bytes_per_col(wtype);
    const int koff = wtype == W_MXFP4 ? t.kc / 2 : t.kc * bytes_per_col(wtype);
    if (t.kn == K) {
      prefetch_l2(base + (size_t)t.r0 * rb, (uint32_t)(cb * t.nr));
    } else {
      for (int i = 0; i < t.nr; ++i) prefetch_l2(base + (size_t)(t.r0 + i) * rb + koff, (uint32_t)cb);
    }
    if (wtype == W_MXFP4 && t.kn == K) {
      const uint32_t sbytes = (uint32_t)(t.nr * (K / 32)) & ~15u;
      const char* sb = static_cast<const char*>(op->ws) + (size_t)t.mat * __ldg(&op->ws_mstride);
      if (sbytes) prefetch_l2(sb + (size_t)t.r0 * (K / 32), sbytes);
    }
  }

  // Ask L2 for lane gl's share (of nl) of a byte range, in 16-byte granules (an unaligned range
  // is left to the copies).
  __device__ __forceinline__ void prefetch_share(const char* base, size_t bytes, int gl, int nl) {
    if (reinterpret_cast<uintptr_t>(base) & 15u) return;
    const size_t granules = bytes / 16, per = (granules + (size_t)nl - 1) / (size_t)nl;
    const size_t g0 = (size_t)gl * per;
    if (g0 >= granules) return;
    const size_t g1 = granules < g0 + per ? granules : g0 + per;
    prefetch_l2(base + g0 * 16, (uint32_t)((g1 - g0) * 16));
  }

  // Lane gl's share of expert e's matrix (values and scales) of an expert op.
  __device__ __forceinline__ void prefetch_expert(const OpDesc* op, int e, int gl, int nl) {
    const int K = __ldg(&op->K), N = __ldg(&op->N), wt = __ldg(&op->wtype);
    prefetch_share(static_cast<const char*>(op->w) + (size_t)e * __ldg(&op->w_mstride), (size_t)N * row_bytes(wt, K), gl, nl);
    if (wt == W_MXFP4)
      prefetch_share(static_cast<const char*>(op->ws) + (size_t)e * __ldg(&op->ws_mstride), (size_t)N * (K / 32), gl, nl);
  }

  // Expert prefetch (the Muse Spark Open megakernel article prefetches the experts the previous
  // step routed to): while cursor c waits at a routed gate/up op for the layer's routing, the
  // lanes of all CTAs ask L2 for the gate/up and down matrices of the shared experts, always
  // needed, and of the experts the layer's last routing chose, when at least half of those had
  // also been chosen by the routing before it (xpf_mode 1; 2: always). Once per op and step.
  __device__ __forceinline__ bool expert_prefetch(const LaneCursor& c, int w, int& key) {
    if (c.oi >= p.op_end) return false;
    const OpDesc* op = p.ops + c.oi;
    if (__ldg(&op->type) != OP_ROUTED_GATEUP) return false;
    const int32_t* rec = op->xpf;
    if (!rec) return false;
    const int k = c.step * p.n_ops + c.oi;
    if (k == key) return false;
    key = k;
    const OpDesc* dn = (c.oi + 1 < p.op_end && __ldg(&p.ops[c.oi + 1].type) == OP_EXP_DOWN) ? op + 1 : nullptr;
    const int gl = blockIdx.x * kConsumerWarps + w, nl = p.n_ctas * kConsumerWarps;
    for (int sh = 0; sh < p.n_shared; ++sh) {
      prefetch_expert(op, p.E + sh, gl, nl);
      if (dn) prefetch_expert(dn, p.E + sh, gl, nl);
    }
    const int hits = ld_relaxed_s32(rec), n = min(ld_relaxed_s32(rec + 1), kMaxRouteSlots);
    const int routed = n - p.n_shared;
    if (routed > 0 && (p.xpf_mode == 2 || 2 * hits >= routed))
      for (int j = p.n_shared; j < n; ++j) {
        const int e = ld_relaxed_s32(rec + 2 + j);
        if (e < 0 || e >= p.E) continue;  // a torn or stale record: a hint only
        prefetch_expert(op, e, gl, nl);
        if (dn) prefetch_expert(dn, e, gl, nl);
      }
    return true;
  }

  // Bytes a tile brings into its slot.
  __device__ __forceinline__ uint32_t tile_bytes(const OpDesc* op, int type, const Tile& t) const {
    if (type == OP_ATTN) return (uint32_t)(t.nr * 2 * kv_row_bytes(p.kv_fp8));
    const int wtype = __ldg(&op->wtype);
    if (wtype == W_MXFP4) return (uint32_t)(t.nr * (t.kn / 2) + t.nr * (t.kn / 32));
    return (uint32_t)(t.nr * t.kn * bytes_per_col(wtype));
  }

  // Point the lane's cursor at its next tile: ops without tiles for this lane are passed over.
  // Returns false if the lane has no tile to offer right now (all ops done, or a routed op whose
  // routing is not computed yet).
  __device__ __forceinline__ bool peek(LaneCursor& c, int w, Tile& t, AttnIter& pa, GemvIter& pg) {
    for (;;) {
      if (c.oi >= p.op_end) {
        if (c.step + 1 >= steps_of(p)) return false;
        ++c.step;  // the launch's next step: the same ops at the next position
        c.oi = p.op_begin;
        c.started = 0;
      }
      const OpDesc* op = p.ops + c.oi;
      const int type = __ldg(&op->type);
      if (!c.started) {
        if (type == OP_ATTN) {
          // a later step's attention reads cache rows the earlier steps appended: wait until
          // this CTA has taken the state of that step (its consumers passed the step end)
          if (c.step > 0) {
            const uint32_t e = *reinterpret_cast<volatile const uint32_t*>(&g_st.epoch);
            if ((int32_t)(e - (epoch0 + (uint32_t)c.step)) < 0) return false;
            __threadfence_block();
          }
          c.a.init(p, blockIdx.x, w, pos + c.step, M, attn_rows(p, s.slot_bytes));
        } else {
          const int* experts = nullptr;
          int n_slots = 0;
          if (type == OP_ROUTED_GATEUP || type == OP_EXP_DOWN) {
            experts = routing(op, c.step);
            if (!experts) return false;  // routing not computed yet
            n_slots = s.route->n_slots;
          }
          c.g.init(*op, p.n_ctas, blockIdx.x, w, n_slots, experts, 0);
        }
        c.started = 1;
      }
      pa = c.a;
      pg = c.g;
      if (type == OP_ATTN ? pa.next(t) : pg.next(t)) return true;
      ++c.oi;
      c.started = 0;
    }
  }

  __device__ __forceinline__ void issue(LaneCursor& c, int w, const Tile& t, const AttnIter& pa, const GemvIter& pg) {
    const OpDesc* op = p.ops + c.oi;
    const uint32_t st = c.n % (uint32_t)kStages;
    const uint32_t fb = smem_addr(&s.full[w * kStages + st]);
    if (__ldg(&op->type) == OP_ATTN) {
      c.a = pa;
      copy_attn(op, t, s.slot(w, st), fb);
    } else {
      c.g = pg;
      copy_gemv(op, t, s.slot(w, st), fb);
    }
#ifdef DEC_TRACE
    if (p.trace && blockIdx.x == 0 && c.n < (uint32_t)kTileLog)
      p.trace[(size_t)p.n_ctas * p.n_ops * kTraceFields + ((size_t)w * kTileLog + c.n) * kTileStamps] =
          (uint64_t)clock64();
    if (w == 0 && p.trace) {
      uint64_t* r = p.trace + ((size_t)blockIdx.x * p.n_ops + c.oi) * kTraceFields;
      const uint64_t now = gtimer();
      if (r[7] == 0) r[5] = now;
      r[6] = now;
      r[7] += 1;
    }
#endif
    ++c.n;
  }

  // Lane w streams consumer warp w's tiles: each round, every lane whose warp has a free slot
  // issues its next tile (the ring itself bounds the bytes in flight). When no lane can issue
  // (the consumers are waiting for an op's input, so their rings stay full), the lanes walk on
  // past their rings and ask L2 for up to DEC_L2_AHEAD more tiles each: HBM keeps streaming
  // through the hand-off instead of idling, and the ring's later copies of those tiles hit L2
  // (the Muse Spark Open megakernel article, section "three bills", prefetches the next task's
  // weights into L2 the same way; measured here, prefetching only while the ring waits beats
  // prefetching whole ops ahead, which competed with the current op's copies).
  __device__ __forceinline__ void run(int lane) {
    if (lane >= kConsumerWarps) return;
    constexpr unsigned kMask = (1u << kConsumerWarps) - 1u;
    const int w = lane;
    LaneCursor c;
    c.oi = p.op_begin;
    c.started = 0;
    c.step = 0;
    c.n = 0;
    LaneCursor pf = c;  // L2-prefetch cursor: at or ahead of the ring's
    uint32_t pf_n = 0;
    int xpf_key = -1;   // (step, op) of the last expert prefetch
    uint64_t t_idle = 0;
    for (;;) {
      Tile t;
      AttnIter pa;
      GemvIter pg;
      const bool have = peek(c, w, t, pa, pg);
      const bool done = c.oi >= p.op_end && c.step + 1 >= steps_of(p);
      const uint32_t st = c.n % (uint32_t)kStages;
      const bool ready =
          have && mbar_test_wait(smem_addr(&s.empty[w * kStages + st]), ((c.n / (uint32_t)kStages) & 1u) ^ 1u);
      // every lane whose warp has a free slot issues its next tile (the ring bounds the bytes in flight)
      const bool grant = ready;
      const unsigned granted = __ballot_sync(kMask, grant);
      if (grant) issue(c, w, t, pa, pg);
      const bool issued = granted != 0u;
      if (__all_sync(kMask, done)) break;
      if (issued) {
        t_idle = 0;
        continue;
      }
      // nothing issued: slots full or routing pending. While the ring waits, each
      // lane asks L2 for the tiles after its ring, up to DEC_L2_AHEAD of them, so HBM keeps
      // streaming through a hand-off; the ring's copies of those tiles then hit L2.
      {
        if (pf_n < c.n) {
          pf = c;
          pf_n = c.n;
        }
        Tile tp;
        AttnIter pa2;
        GemvIter pg2;
        bool did = false;
        if (pf_n < c.n + (uint32_t)DEC_L2_AHEAD) {
          if (peek(pf, w, tp, pa2, pg2)) {
            const int ptype = __ldg(&p.ops[pf.oi].type);
            prefetch_tile(p.ops + pf.oi, ptype, tp);
            if (ptype == OP_ATTN) pf.a = pa2;
            else pf.g = pg2;
            ++pf_n;
            did = true;
          } else if (p.xpf_mode) {
            did = expert_prefetch(pf, w, xpf_key);  // the cursor waits for a routing
          }
        }
        if (__any_sync(kMask, did)) continue;
      }
      // back off so the spinning lanes leave the scheduler's issue slots to the consumers
      __nanosleep(64);
      int stop = 0;
      if (w == 0) {
        const uint64_t now = gtimer();
        if (aborted(p)) {
          stop = 1;
        } else if (t_idle == 0) {
          t_idle = now;
        } else if (now - t_idle > p.timeout_ns) {
          raise_error(p, DEC_ERR_TIMEOUT, c.oi, 0xFFFFFFFEu, 0u, 0u, 1);
          stop = 1;
        }
      }
      if (__shfl_sync(kMask, stop, 0)) break;
    }
    // Every copy in flight must land before the CTA may exit (abort paths).
    const uint32_t n = c.n;
    for (uint32_t k = (n > (uint32_t)kStages ? n - kStages : 0u); k < n; ++k) {
      const uint32_t fb = smem_addr(&s.full[w * kStages + (k % (uint32_t)kStages)]);
      const uint64_t t0 = gtimer();
      while (!mbar_try_wait(fb, (k / (uint32_t)kStages) & 1u))
        if (gtimer() - t0 > p.timeout_ns) break;
    }
  }
};

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------------ attention (per warp)
// Scratch in s.act (floats):
//   q     [M*G][128]         rotated queries of the kv group, times log2(e)/sqrt(128)
//   sc    [warps][G][P]      scores, then probabilities, of each warp's current tile; reused for
//                            the splits' output slices in the merge
//   mg    [warps][G][132]    per-warp (max, sum, -, -, output[128]) at the end of a split
//   kvn   bf16 [2][M][128]   this call's own keys / values (rotated, rounded)
//   cw    [rows][ns]         merge weights
//   ml    [ns][rows] float2  the splits' (max, sum) in the merge
//   raw   [M][G+2][128]      this call's q, k, v rows of the kv group, as polled
struct AttnScratch {
  float* q;
  float* sc;
  float* mg;
  uint16_t* kvn;
  float* cw;
  float2* ml;
  float* raw;
};

__device__ __forceinline__ AttnScratch attn_scratch(const KParams& p, const Smem& s, int M, int P) {
  const AttnLayout l = attn_layout(M, p.G, P, p.ns_max);
  AttnScratch a;
  a.q = s.act + l.q;
  a.sc = s.act + l.sc;
  a.mg = s.act + l.mg;
  a.kvn = reinterpret_cast<uint16_t*>(s.act + l.kvn);
  a.cw = s.act + l.cw;
  a.ml = reinterpret_cast<float2*>(s.act + l.ml);
  a.raw = s.act + l.raw;
  return a;
}

template <int G_>
struct AttnState {
  float mrun[G_], lrun[G_];
  float o[G_][4];  // this lane's dims 4*lane .. +3
};

// e4m3fn code (bits 0-7 of x) -> float, exactly: the code's 7 low bits go to fp32 bits 20-26
// and its sign to bit 31, which is the value times 2^-120 (subnormal codes become fp32
// subnormals); the multiply by 2^120 restores it.
__device__ __forceinline__ float e4m3_to_float_bits(uint32_t x) {
  return __uint_as_float(((x & 0x7Fu) << 20) | ((x & 0x80u) << 24)) * 0x1p120f;
}

// One tile of n rows (keys at kr, values at vr; 256 B per bf16 row, 128 B per e4m3 row) for the
// G_ heads of token m. e4m3 rows hold the codes: the caller folds the keys' scale into q and
// applies the values' scale to the outputs.
// vis_base < 0: cached rows, row j at position row0 + j, visible iff >= lo_m (a sliding window's
// start for token m); else row j is this call's row vis_base + j, visible iff <= m.
template <int G_, bool KV8>
__device__ __forceinline__ void attn_warp_tile(AttnState<G_>& A, const float (&q)[G_][16], const uint8_t* kr,
                                               const uint8_t* vr, int n, int vis_base, int m, float* sc, int P,
                                               int lane, int row0 = 0, int lo_m = 0) {
  constexpr int RB = KV8 ? 128 : 256;
  const int grp = lane >> 3, sub = lane & 7;
  // scores: eight lanes per row, 16 dims each, four rows per step
  for (int j0 = 0; j0 < n; j0 += 4) {
    const int j = j0 + grp;
    float kf[16];
    if (j < n) {
      if constexpr (KV8) {
        const uint4 k0 = *reinterpret_cast<const uint4*>(kr + (size_t)j * RB + sub * 16);
        const uint32_t kw[4] = {k0.x, k0.y, k0.z, k0.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) kf[e] = e4m3_to_float_bits(kw[e >> 2] >> (8 * (e & 3)));
      } else {
        const uint4 k0 = *reinterpret_cast<const uint4*>(kr + (size_t)j * RB + sub * 32);
        const uint4 k1 = *reinterpret_cast<const uint4*>(kr + (size_t)j * RB + sub * 32 + 16);
        const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          kf[2 * e] = bf16_lo(kw[e]);
          kf[2 * e + 1] = bf16_hi(kw[e]);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) kf[e] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < G_; ++h) {
      float2 t = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        t = ffma2(make_float2(q[h][2 * e], q[h][2 * e + 1]), make_float2(kf[2 * e], kf[2 * e + 1]), t);
      float sv = t.x + t.y;
      sv += __shfl_xor_sync(0xffffffffu, sv, 4);
      sv += __shfl_xor_sync(0xffffffffu, sv, 2);
      sv += __shfl_xor_sync(0xffffffffu, sv, 1);
      if (sub == 0 && j < n) {
        const bool vis = vis_base < 0 ? row0 + j >= lo_m : vis_base + j <= m;
        sc[h * P + j] = vis ? sv : -INFINITY;
      }
    }
  }
  __syncwarp();
  // online softmax over the tile: lane j holds row j (n <= 32)
  float scale[G_];
#pragma unroll
  for (int h = 0; h < G_; ++h) {
    const float sv = lane < n ? sc[h * P + lane] : -INFINITY;
    float mx = sv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float mnew = fmaxf(A.mrun[h], mx);
    const float pj = (mnew == -INFINITY || sv == -INFINITY) ? 0.f : exp2f(sv - mnew);
    float sum = pj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < n) sc[h * P + lane] = pj;
    scale[h] = (mnew == -INFINITY) ? 1.f : (A.mrun[h] == -INFINITY ? 0.f : exp2f(A.mrun[h] - mnew));
    A.lrun[h] = A.lrun[h] * scale[h] + sum;
    A.mrun[h] = mnew;
  }
  __syncwarp();
  // values: lane owns dims 4*lane .. +3
#pragma unroll
  for (int h = 0; h < G_; ++h)
#pragma unroll
    for (int e = 0; e < 4; ++e) A.o[h][e] *= scale[h];
  for (int j = 0; j < n; ++j) {
    float2 v01, v23;
    if constexpr (KV8) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(vr + (size_t)j * RB + lane * 4);
      v01 = make_float2(e4m3_to_float_bits(v), e4m3_to_float_bits(v >> 8));
      v23 = make_float2(e4m3_to_float_bits(v >> 16), e4m3_to_float_bits(v >> 24));
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(vr + (size_t)j * RB + lane * 8);
      v01 = make_float2(bf16_lo(v.x), bf16_hi(v.x));
      v23 = make_float2(bf16_lo(v.y), bf16_hi(v.y));
    }
#pragma unroll
    for (int h = 0; h < G_; ++h) {
      const float pj = sc[h * P + j];
      const float2 pp = make_float2(pj, pj);
      const float2 o01 = ffma2(pp, v01, make_float2(A.o[h][0], A.o[h][1]));
      const float2 o23 = ffma2(pp, v23, make_float2(A.o[h][2], A.o[h][3]));
      A.o[h][0] = o01.x;
      A.o[h][1] = o01.y;
      A.o[h][2] = o23.x;
      A.o[h][3] = o23.y;
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ consumer
struct Consumer;
template <int WT, int MT, int NR, int NI>
__device__ __noinline__ bool gemv_tiles_entry(const KParams& p, int oi, const OpDesc& op, int M, float* xres, int a,
                                              float* accd);
template <int WT, int MT, int NR, int NI>
__device__ __noinline__ bool gemv_csplit_entry(const KParams& p, int oi, const OpDesc& op, int M, int a, float* parts);
template <int MT, int NR, int NI>
__device__ __noinline__ bool gemv_xsplit_entry(const KParams& p, int oi, const OpDesc& op, int M, int a, float* parts);
__device__ __noinline__ bool gemv_tc_entry(const KParams& p, int oi, const OpDesc& op, int M, float* xres, int a,
                                          float* parts);
template <int MT>
__device__ __noinline__ bool gemv_slot_entry(const KParams& p, int oi, const OpDesc& op, int sl, int M, int a,
                                             float* accd);
__device__ __noinline__ bool gemv_prologue_entry(const KParams& p, int oi, int M);
__device__ __noinline__ bool gemv_tiles_dispatch_entry(const KParams& p, int oi, int M);
__device__ __noinline__ bool gemv_epilogue_entry(const KParams& p, int oi, int M);
__device__ __noinline__ bool routing_entry(const KParams& p, int oi, int M);
__device__ __noinline__ bool copy_act_entry(const KParams& p, int oi, float* dst, const uint64_t* src, int M, int K,
                                            int src_stride, int cw);
template <int G_>
__device__ __noinline__ bool attn_entry(const KParams& p, int oi, int pos, int M);
template <int G_>
__device__ __noinline__ bool attn_tc_entry(const KParams& p, int oi, int r0, int r1, int m_tok, int M, int lo_m);

// A consumer thread's view of the kernel. Built from scratch wherever it is needed (see
// smem_raw), so out-of-line functions keep it in registers; the ring position of the thread's
// warp lives in shared memory between them (save_tiles).
struct Consumer {
  const KParams& p;
  Smem s;
  uint32_t epoch, tag;  // tag: the data tag of this step (epoch + 1; zeroed memory never matches)
  const StepState& st;
  int tid, warp, lane;
  uint32_t n_tiles;  // tiles consumed by this warp (ring position)

  __device__ __forceinline__ explicit Consumer(const KParams& p_)
      : p(p_),
        s(carve(smem_raw, p_)),
        epoch(g_st.epoch),
        tag(g_st.epoch + 1u),
        st(g_st),
        tid((int)threadIdx.x),
        warp((int)threadIdx.x >> 5),
        lane((int)threadIdx.x & 31),
        n_tiles(s.ntiles[threadIdx.x >> 5]) {}

  __device__ __forceinline__ void save_tiles() {
    __syncwarp();
    if (lane == 0) s.ntiles[warp] = n_tiles;
    __syncwarp();
  }

#ifdef DEC_TRACE
  __device__ __forceinline__ void tile_log(int field) {
    if (p.trace && lane == 0 && blockIdx.x == 0 && n_tiles < kTileLog) {
      uint64_t* base = p.trace + (size_t)p.n_ctas * p.n_ops * kTraceFields;
      base[((size_t)warp * kTileLog + n_tiles) * kTileStamps + 1 + field] = (uint64_t)clock64();
    }
  }
#else
  __device__ __forceinline__ void tile_log(int) {}
#endif

  // Arrive at ticket t (n arrivals per use); true in the last arrival (all consumers agree).
  // The last arrival sets the ticket back to zero: its next use comes in a later launch, after
  // every arrival of this one, so a call that skips the op holding a ticket (a layer or the LM
  // head run on its own) leaves no count behind.
  __device__ bool ticket(int t, int n) {
    consumer_sync();
    if (tid == 0) {
      const uint32_t old = atom_add_acq_rel(&p.tickets[t], 1u);
      const bool last = old == (uint32_t)n - 1u;
      if (last) atomicExch(&p.tickets[t], 0u);
      s.flags[kFlagTicket] = last ? 1 : 0;
    }
    consumer_sync();
    return s.flags[kFlagTicket] != 0;
  }

  // Wait until counter c has n arrivals in this step (builds with DEC_POLL_DATA=0). One thread
  // spins; the others wait at the barrier; the data behind the count is then read with its tags
  // checked (gather). By default the inputs are polled directly and this returns at once: a
  // ready input then costs one round trip to L2 instead of two.
  __device__ bool wait_counter(int c, int n, int oi, uint32_t where) {
#if DEC_POLL_DATA
    return true;  // the data is polled directly (its tags decide)
#endif
    bool ok = true;
    if (tid == 0) {
      const uint32_t target = (epoch + 1u) * (uint32_t)n;
      const uint32_t* ctr = p.ctr + c;
      if ((int32_t)(ld_relaxed(ctr) - target) < 0) ok = wait_counter_slow(p, ctr, target, oi, where);
#if DEC_ORDERED_ARRIVALS
      (void)ld_acquire(ctr);
#endif
    }
    return consumer_all(ok);
  }

  // This CTA has written its share of what counter c announces (and its threads are done with
  // the op: the barrier also guards the shared op copy).
  __device__ void arrive(int c) {
    consumer_sync();  // every warp's stores are issued
#if !DEC_POLL_DATA
#if DEC_ORDERED_ARRIVALS
    if (tid == 0) red_release(p.ctr + c, 1u);
#else
    if (tid == 0) red_relaxed(p.ctr + c, 1u);
#endif
#endif
  }

  // Wait for this warp's next tile; the verdict is uniform across the warp.
  __device__ bool next_slot(int op_idx, uint8_t*& slot, uint32_t& eb) {
    const uint32_t stg = n_tiles % (uint32_t)kStages;
    const uint32_t parity = (n_tiles / (uint32_t)kStages) & 1u;
    slot = s.slot(warp, stg);
    eb = smem_addr(&s.empty[warp * kStages + stg]);
    tile_log(0);
    const bool ok = wait_mbar(p, smem_addr(&s.full[warp * kStages + stg]), parity, op_idx, 3);
    tile_log(1);
    return __all_sync(0xffffffffu, ok);
  }

  // The warp is done reading its current slot: hand it back to the producer.
  __device__ void release(uint32_t eb) {
    tile_log(2);
    __syncwarp();
    if (lane == 0) mbar_arrive(eb);
    tile_log(3);
    ++n_tiles;
  }

  // ---------------------------------------------------------------- activation loads
  // Poll n items of W tagged words (item i at addr(i)) and hand each to sink(i, values); every
  // thread keeps U items in flight, so a prologue whose inputs are ready costs one round trip.
  template <int U, int W, class Addr, class Sink>
  __device__ __forceinline__ bool gather(int n, Addr addr, Sink sink, int oi, uint32_t where) {
    bool ok = true;
    for (int i0 = tid; i0 < n; i0 += U * kConsumerThreads) {
      // all U items' loads first, then the checks
      uint64_t w[U][W];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kConsumerThreads;
        if (i < n) {
          ld_item<W>(addr(i), w[u]);
        } else {
#pragma unroll
          for (int k = 0; k < W; ++k) w[u][k] = tagged(0.f, tag);
        }
      }
      uint32_t late = 0;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kConsumerThreads;
        float v[W];
        bool good = true;
#pragma unroll
        for (int k = 0; k < W; ++k) {
          v[k] = value_of(w[u][k]);
          good &= tag_of(w[u][k]) == tag;
        }
        if (i < n) {
          if (good)
            sink(i, v);
          else
            late |= 1u << u;
        }
      }
      // words not yet visible: poll them one by one
#ifdef DEC_TRACE
      if (late) atomicAdd(const_cast<int*>(&s.flags[kFlagLate]), __popc(late));
#endif
      for (int u = 0; late != 0u; ++u, late >>= 1) {
        if (!(late & 1u)) continue;
        const int i = i0 + u * kConsumerThreads;
        float v[W];
        if (!poll_item_slow<W>(p, addr(i), v, tag, oi, where)) return false;
        sink(i, v);
      }
    }
    return ok;
  }

  // Residual output x_m[row] = v of a residual op (o-proj, down, expert down): the tagged word,
  // and its bf16 rounding where the caller takes the result (a layer run on its own).
  __device__ __forceinline__ void put_x(const OpDesc& op, int m, int row, float v) {
    st_tagged(op.x_out + (size_t)m * p.H + row, v, tag);
    if (op.y_bf16) op.y_bf16[(size_t)m * p.H + row] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }

  __device__ __forceinline__ const uint16_t* x_bf16(const OpDesc& op, int m) const {
    return op.xsrc == X_EMBED ? static_cast<const uint16_t*>(op.x_src) + (size_t)st.tokens[m] * p.H
                              : static_cast<const uint16_t*>(st.hidden_in) + (size_t)m * p.H;
  }

  __device__ __forceinline__ const uint64_t* x_tagged(const OpDesc& op, int m) const {
    return p.hs + ((size_t)op.x_idx * p.Mmax + m) * p.H;
  }

  // ---------------------------------------------------------------- prologues
  // The gain is a weight: its first kGainPre vectors per thread are loaded before the input.
  static constexpr int kGainPre = 4;
  __device__ void load_gain(const OpDesc& op, uint2 (&g)[kGainPre]) {
    const int H4 = p.H / 4;
#pragma unroll
    for (int u = 0; u < kGainPre; ++u) {
      const int i = tid + u * kConsumerThreads;
      g[u] = (op.norm && i < H4) ? __ldg(reinterpret_cast<const uint2*>(op.gain) + i) : make_uint2(0u, 0u);
    }
  }

  // act = x_m * gain (op.norm) or x_m for the M tokens, written in the quarter-plane layout of
  // the op's weight type. RMSNorm's 1/rms is a scalar per token, so it is applied to the row
  // sums in the epilogue instead (W (x g / rms) = (W (x g)) / rms): the prologue needs no
  // barrier for it. Each thread sums the squares of the groups it loaded (group i = m*H/4 + k4
  // belongs to thread i mod threads in every CTA), warps reduce by a fixed tree, and lane 0
  // leaves the warp's partial in s.red[m * 8 + warp]; rstd() adds them in warp order, so every
  // CTA computes the same value. Returns this thread's polling verdict.
  __device__ __forceinline__ bool norm_prologue(const OpDesc& op, int M, const uint2 (&gpre)[kGainPre], int oi) {
    const int H = p.H, H4 = H / 4, n4 = M * H4;
    const int cw = chunk_width(op.wtype), nvt = H / cw;
    float ss[kMmax];
#pragma unroll
    for (int m = 0; m < kMmax; ++m) ss[m] = 0.f;
    auto put = [&](int i, float4 x) {
      const int m = i / H4, k4 = i - m * H4;
      if (op.norm) {
        // gains: the first kGainPre vectors of this thread were loaded before the wait
        const int u = (k4 - tid) / kConsumerThreads;
        const uint2 g = (M == 1 && u < kGainPre)
                            ? (u == 0 ? gpre[0] : (u == 1 ? gpre[1] : (u == 2 ? gpre[2] : gpre[3])))
                            : __ldg(reinterpret_cast<const uint2*>(op.gain) + k4);
#pragma unroll
        for (int mm = 0; mm < kMmax; ++mm) {
          if (mm == m) {
            ss[mm] = fmaf(x.x, x.x, ss[mm]);
            ss[mm] = fmaf(x.y, x.y, ss[mm]);
            ss[mm] = fmaf(x.z, x.z, ss[mm]);
            ss[mm] = fmaf(x.w, x.w, ss[mm]);
          }
        }
        x.x *= bf16_lo(g.x);
        x.y *= bf16_hi(g.x);
        x.z *= bf16_lo(g.y);
        x.w *= bf16_hi(g.y);
      }
      if (op.tc)
        put_bfrag(s.act, m, 4 * k4, x);
      else
        *reinterpret_cast<float4*>(s.act + m * H + act_pos(4 * k4, cw, nvt)) = x;
    };
    bool ok = true;
    if (op.xsrc == X_F32) {
      ok = gather<kGatherU, 4>(
          n4, [&](int i) { return x_tagged(op, i / H4) + 4 * (i % H4); },
          [&](int i, const float (&v)[4]) { put(i, make_float4(v[0], v[1], v[2], v[3])); }, oi, 7);
      if (tid == 0) TRACE(p, oi, 8, gtimer());
    } else {
      for (int i = tid; i < n4; i += kConsumerThreads) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(x_bf16(op, i / H4)) + i % H4);
        put(i, make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y)));
      }
    }
    if (op.norm) {
#pragma unroll
      for (int m = 0; m < kMmax; ++m) {
        float acc = ss[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) s.red[m * 8 + warp] = acc;
      }
    }
    return ok;
  }

  // 1/rms of token m for ops whose prologue was norm_prologue (after the prologue's barrier).
  __device__ __forceinline__ float rstd(int m) const {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += s.red[m * 8 + w];
    return 1.0f / sqrtf(tot / (float)p.H + p.eps);
  }

  // dst = M rows of K tagged words polled from global (row stride src_stride words), in the
  // quarter-plane layout of chunk width cw.
  __device__ __forceinline__ bool copy_act(float* dst, const uint64_t* src, int M, int K, int src_stride, int cw, int oi) {
    const int K4 = K / 4, nvt = cw ? K / cw : 0;
    return gather<kCopyU, 4>(
        M * K4, [&](int i) { return src + (size_t)(i / K4) * src_stride + 4 * (i % K4); },
        [&](int i, const float (&v)[4]) {
          if (cw == 0)  // the tensor-core B operand layout
            put_bfrag(dst, i / K4, 4 * (i % K4), make_float4(v[0], v[1], v[2], v[3]));
          else
            *reinterpret_cast<float4*>(dst + (i / K4) * K + act_pos(4 * (i % K4), cw, nvt)) =
                make_float4(v[0], v[1], v[2], v[3]);
        },
        oi, 9);
  }

  // xres[i][m] = x_m[a + i] for the CTA's rows [a, b): the residual input of the op.
  __device__ __forceinline__ bool load_residual(const OpDesc& op, float* xres, int a, int b, int M, int oi) {
    const int n = (b - a) * M;
    if (op.xsrc == X_F32)
      return gather<2, 1>(
          n, [&](int t) { return x_tagged(op, t % M) + a + t / M; },
          [&](int t, const float (&v)[1]) { xres[t] = v[0]; }, oi, 8);
    for (int t = tid; t < n; t += kConsumerThreads)
      xres[t] = __uint_as_float((uint32_t)__ldg(x_bf16(op, t % M) + a + t / M) << 16);
    return true;
  }

  // ---------------------------------------------------------------- routing (MoE layers)
  // Every CTA computes the layer's routing itself from the router logits (op.act) it polls:
  // top-k per token (largest first, lower index on ties), softmax over the selected logits,
  // and the union of the window's experts (shared experts first). The producer lanes read it
  // from shared memory once flags[kFlagRoute] names the layer. Uses the start of s.act.
  __device__ __forceinline__ bool ensure_routing(const OpDesc& op, int M, int oi) {
    if (s.flags[kFlagRoute] == route_tag(epoch, op.layer, p.L)) return true;
    const int E = p.E, k = p.top_k;
    float* r = s.act;  // [M][E]
    if (!wait_counter(op.aux_ctr, p.n_ctas, oi, 10)) return false;
    const bool ok = gather<4, 1>(
        M * E, [&](int i) { return op.act + i; }, [&](int i, const float (&v)[1]) { r[i] = v[0]; }, oi, 10);
    if (!consumer_all(ok)) return false;
    RouteBlock* rb = s.route;
    // Top-k per token, one warp per token (warp m < M takes token m): lane l owns logits
    // l, l + 32, ... and keeps its best one not yet taken; each of the k rounds reduces the
    // lanes' bests over the warp (larger logit first, lower index on ties), and the lane that
    // owned the winner takes it out and rescans its own logits. No CTA barrier inside.
    if (warp < M) {
      float* rm = r + warp * E;
      auto lane_best = [&](float& bv, int& bi) {
        bv = -INFINITY;
        bi = 0x7FFFFFFF;
        for (int e = lane; e < E; e += 32) {
          const float v = rm[e];
          if (v > bv) {  // ascending e: an equal later logit never replaces the lower index
            bv = v;
            bi = e;
          }
        }
      };
      float bv;
      int bi;
      lane_best(bv, bi);
      for (int kk = 0; kk < k; ++kk) {
        float v = bv;
        int i = bi;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v, o);
          const int oi = __shfl_xor_sync(0xffffffffu, i, o);
          if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
          }
        }
        if (i >= E) i = kk;  // no ordered logit left (NaN inputs): an in-range id, never a wild one
        if (lane == 0) {
          rb->topk[warp][kk] = i;
          rb->topk_w[warp][kk] = v;  // the logit, replaced by its weight below
        }
        if ((i & 31) == lane) {  // the owner takes the winner out and finds its next best
          rm[i] = -INFINITY;
          lane_best(bv, bi);
        }
        __syncwarp();
      }
    }
    consumer_sync();
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
      __threadfence_block();
      s.flags[kFlagRoute] = route_tag(epoch, op.layer, p.L);  // the producer lanes may now read the ids
    }
    consumer_sync();
    if (op.xpf && blockIdx.x == p.n_ctas - 1 && warp == 0) {
      // the layer's expert prefetch record, a hint the producers of every CTA read with relaxed
      // loads: how many of this routing's routed experts the layer's last routing also chose, the
      // slot count, then this routing's expert ids
      const int n = rb->n_slots, ns = p.n_shared;
      const int pn = min(max(ld_relaxed_s32(op.xpf + 1), 0), kMaxRouteSlots);
      const int pa = lane < pn ? ld_relaxed_s32(op.xpf + 2 + lane) : -1;
      const int pb = pn > 32 ? ld_relaxed_s32(op.xpf + 2 + 32) : -1;
      const int c0 = (lane >= ns && lane < n) ? rb->expert[lane] : -2;
      const int c1 = (lane + 32 >= ns && lane + 32 < n) ? rb->expert[lane + 32] : -2;
      bool f0 = false, f1 = false;
      for (int q = ns; q < pn; ++q) {
        const int e = __shfl_sync(0xffffffffu, pa, q & 31);
        const int pe = q < 32 ? e : pb;
        f0 |= pe == c0;
        f1 |= pe == c1;
      }
      const int hits = __popc(__ballot_sync(0xffffffffu, f0)) + __popc(__ballot_sync(0xffffffffu, f1));
      __syncwarp();
      if (lane < n) st_relaxed_s32(op.xpf + 2 + lane, rb->expert[lane]);
      if (lane + 32 < n) st_relaxed_s32(op.xpf + 2 + 32 + lane, rb->expert[lane + 32]);
      if (lane == 0) {
        st_relaxed_s32(op.xpf, hits);
        st_relaxed_s32(op.xpf + 1, n);
      }
    }
    if (blockIdx.x == 0) {  // a copy in global memory for inspection
      const int* src = reinterpret_cast<const int*>(rb);
      for (int i = tid; i < (int)(sizeof(RouteBlock) / 4); i += kConsumerThreads) op.route[i] = src[i];
      // the caller's copies of the selection (a layer run on its own)
      for (int i = tid; i < M * k; i += kConsumerThreads) {
        if (op.topk_idx_out) op.topk_idx_out[i] = rb->topk[i / k][i % k];
        if (op.topk_w_out) op.topk_w_out[i] = rb->topk_w[i / k][i % k];
      }
    }
    return true;
  }

  // ---------------------------------------------------------------- matrix ops
  // This warp's tiles of a matrix op. Results of a row group land in lane j*MT + m (row j,
  // token m); tokens m >= M (MT = 4 serving a 2- or 3-token window) are computed on zero
  // activations and dropped. NI > 0 (one token, whole rows): the warp keeps the op's
  // activations in NI chunks of registers per lane for the whole op; a separate instantiation,
  // so the shared-memory path's registers never sit next to them.
  template <int WT, int MT, int NR, int NI>
  __device__ __forceinline__ bool gemv_op_t(int oi, const OpDesc& op, int M, float* xres, int a, float* accd) {
    GemvIter it;
    const bool routed = op.type == OP_ROUTED_GATEUP || op.type == OP_EXP_DOWN;
    const int n_slots = routed ? s.route->n_slots : 0;
    it.init(op, p.n_ctas, blockIdx.x, warp, n_slots, routed ? s.route->expert : nullptr, 0);
    Acc<NR, MT> A;
    acc_zero(A);
    float best_v = -INFINITY;
    int best_i = 0x7FFFFFFF;
    Tile t;
    bool ok = true;
    const int i = lane / MT, m = lane % MT;
    // the RMSNorm scale of lane's token (norm ops), applied to its row sums
    const float rs = op.norm ? rstd(m < M ? m : 0) : 1.f;
    static_assert(NI == 0 || MT == 1, "register activations serve one token");
    ActRegs<WT, (NI > 0 ? NI : 1)> AR;
    if constexpr (NI > 0) act_regs_load(AR, s.act, op.K, 0, op.K, lane);
    while (it.next(t)) {
      uint8_t* slot;
      uint32_t eb;
      if (!next_slot(oi, slot, eb)) {
        ok = false;
        break;
      }
      const float* actp = (op.type == OP_EXP_DOWN && op.stage_all) ? s.act + (size_t)t.sl * M * op.K : s.act;
      if constexpr (NI > 0)
        warp_gemv_reg<WT, NR, NI>(slot, t.nr, t.kn, AR, A, lane);
      else
        warp_gemv<WT, MT, NR>(slot, t.nr, t.kn, t.kc, actp, op.K, M, A, lane);
      release(eb);
      if (!t.last_k) continue;
      const float v = warp_rowsums<NR, MT>(A, t.nr, lane) * rs;
      acc_zero(A);
      const bool mine = lane < t.nr * MT && m < M;
      switch (op.type) {
        case OP_QKV:
        case OP_ROUTER:
          if (mine) st_tagged(op.out + (size_t)m * op.N + t.r0 + i, v, tag);
          break;
        case OP_OPROJ:
        case OP_DOWN:
          if (mine) put_x(op, m, t.r0 + i, xres[(t.r0 + i - a) * M + m] + v);
          break;
        case OP_GATEUP:
        case OP_ROUTED_GATEUP: {
          // rows come in (gate, up) pairs: lanes (2jj)*MT + m and (2jj+1)*MT + m hold them
          const int jj = lane / MT;
          const float g = __shfl_sync(0xffffffffu, v, ((2 * jj) * MT + m) & 31);
          const float u = __shfl_sync(0xffffffffu, v, ((2 * jj + 1) * MT + m) & 31);
          if (lane < (t.nr / 2) * MT && m < M) {
            if (op.type == OP_GATEUP)
              st_tagged(op.out + (size_t)m * (op.N / 2) + t.r0 / 2 + jj, silu(g) * u, tag);
            else
              st_tagged(op.eh + ((size_t)t.sl * p.Mmax + m) * (op.N / 2) + t.r0 / 2 + jj, silu(g) * u, tag);
          }
          break;
        }
        case OP_EXP_DOWN:
          if (mine) accd[(t.r0 + i - a) * M + m] += s.route->w[m][t.sl] * v;
          break;
        case OP_LMHEAD:
          if (mine) {
            const int row = t.r0 + i;
            float y = v;
            if (op.wtype == W_FP8) y *= __ldg(static_cast<const float*>(op.ws) + row);
            op.logits[(size_t)m * op.N + row] = y;
            if (y > best_v || (y == best_v && row < best_i)) {
              best_v = y;
              best_i = row;
            }
          }
          break;
        default:
          break;
      }
    }
    if (op.type == OP_LMHEAD) {
      // lane l tracked token l % MT; the CTA reduction reads all 32 lanes of every warp
      s.resw[warp * 64 + lane] = best_v;
      reinterpret_cast<int*>(s.resw)[warp * 64 + 32 + lane] = best_i;
    }
    return ok;
  }

  // Column split: every warp covers all of the CTA's rows over its own column range, keeps its
  // activations in registers (one token, NI chunks per lane) and leaves a partial sum per row;
  // the warps' partials are added in warp order afterwards (csplit_epilogue).
  template <int WT, int MT, int NR, int NI>
  __device__ __forceinline__ bool gemv_csplit_t(int oi, const OpDesc& op, int M, int a, float* parts) {
    GemvIter it;
    it.init(op, p.n_ctas, blockIdx.x, warp, 0, nullptr, 0);
    Acc<NR, MT> A;
    static_assert(NI == 0 || MT == 1, "register activations serve one token");
    ActRegs<WT, (NI > 0 ? NI : 1)> AR;
    if constexpr (NI > 0)
      act_regs_load(AR, s.act, op.K, it.kw0, max(0, it.kw1 - it.kw0), lane);  // unconditional: no spills
    const int rows = it.bw - it.aw;
    Tile t;
    while (it.next(t)) {
      uint8_t* slot;
      uint32_t eb;
      if (!next_slot(oi, slot, eb)) return false;
      acc_zero(A);
      if constexpr (NI > 0)
        warp_gemv_reg<WT, NR, NI>(slot, t.nr, t.kn, AR, A, lane);
      else
        warp_gemv<WT, MT, NR>(slot, t.nr, t.kn, t.kc, s.act, op.K, M, A, lane);
      release(eb);
      const float v = warp_rowsums<NR, MT>(A, t.nr, lane);
      const int j = lane / MT, m = lane % MT;
      if (lane < t.nr * MT && m < M) parts[(warp * rows + (t.r0 + j - a)) * M + m] = v;
    }
    // a warp without columns contributes zeros
    if (it.kw0 >= it.kw1)
      for (int k = lane; k < rows * M; k += 32) parts[warp * rows * M + k] = 0.f;
    return true;
  }

  // Column split: row sums = the warps' partials added in warp order, then the op's output.
  __device__ void csplit_epilogue(const OpDesc& op, int M, int a, int b, const float* xres, const float* parts) {
    const int rows = b - a;
    auto rowsum = [&](int r, int m) {
      float v = 0.f;
      for (int w = 0; w < kConsumerWarps; ++w) v += parts[(w * rows + r) * M + m];
      return op.norm ? v * rstd(m) : v;
    };
    if (op.type == OP_GATEUP) {
      for (int t = tid; t < (rows / 2) * M; t += kConsumerThreads) {
        const int jj = t / M, m = t % M;
        const float g = rowsum(2 * jj, m), u = rowsum(2 * jj + 1, m);
        st_tagged(op.out + (size_t)m * (op.N / 2) + a / 2 + jj, silu(g) * u, tag);
      }
      return;
    }
    for (int t = tid; t < rows * M; t += kConsumerThreads) {
      const int r = t / M, m = t % M;
      const float v = rowsum(r, m);
      if (op.type == OP_OPROJ || op.type == OP_DOWN || op.type == OP_EXP_DOWN)
        put_x(op, m, a + r, xres[t] + v);
      else
        st_tagged(op.out + (size_t)m * op.N + a + r, v, tag);
    }
  }

  // Expert down, slot split (all hidden vectors staged): warp w takes chunks of R rows of the
  // slots in the GemvIter order, and adds each chunk's row sums, weighted by the token's routing
  // weight of that slot, to its own partial sums parts[w][row][m]; csplit_epilogue adds the
  // warps' partials in warp order and the residual. NI > 0: one token, the slot's activations
  // reloaded into registers whenever the slot changes.
  template <int MT, int NR, int NI>
  __device__ __forceinline__ bool gemv_xsplit_t(int oi, const OpDesc& op, int M, int a, float* parts) {
    GemvIter it;
    it.init(op, p.n_ctas, blockIdx.x, warp, s.route->n_slots, s.route->expert, 0);
    const int rows = it.bw - it.aw;
    float* pw = parts + warp * rows * M;
    Acc<NR, MT> A;
    static_assert(NI == 0 || MT == 1, "register activations serve one token");
    ActRegs<W_MXFP4, (NI > 0 ? NI : 1)> AR;
    int cur = -1;
    const int i = lane / MT, m = lane % MT;
    Tile t;
    while (it.next(t)) {
      uint8_t* slot;
      uint32_t eb;
      if (!next_slot(oi, slot, eb)) return false;
      const float* act = s.act + (size_t)t.sl * M * op.K;
      if constexpr (NI > 0) {
        if (t.sl != cur) {
          act_regs_load(AR, act, op.K, 0, op.K, lane);
          cur = t.sl;
        }
      }
      acc_zero(A);
      if constexpr (NI > 0)
        warp_gemv_reg<W_MXFP4, NR, NI>(slot, t.nr, t.kn, AR, A, lane);
      else
        warp_gemv<W_MXFP4, MT, NR>(slot, t.nr, t.kn, 0, act, op.K, M, A, lane);
      release(eb);
      const float v = warp_rowsums<NR, MT>(A, t.nr, lane);
      if (lane < t.nr * MT && m < M) pw[(t.r0 + i - a) * M + m] += s.route->w[m][t.sl] * v;
    }
    return true;
  }

  // Tensor-core tiles of a multi-token call (bf16 matrices of the multi-token list): every tile is
  // kGemvTcRows weight rows x Kc columns in boxes of 64 columns (128-byte swizzle); per 16-column
  // step one ldmatrix gives the A fragments (weights) and the B fragments (the tokens' bf16 high
  // parts in columns 0-3 and residues in 4-7, staged by the prologue) come from shared memory;
  // one m16n8k16 MMA with fp32 accumulation. A row group's results are D[row][m] + D[row][m + 4],
  // handed to the same per-(row, token) outputs as the CUDA-core path, eight rows at a time.
  __device__ __forceinline__ bool gemv_tc_t(int oi, const OpDesc& op, int M, float* xres, int a, float* parts) {
    constexpr int MT = kMmax;
    GemvIter it;
    it.init(op, p.n_ctas, blockIdx.x, warp, 0, nullptr, 0);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    float best_v = -INFINITY;
    int best_i = 0x7FFFFFFF;
    const uint32_t* bf = reinterpret_cast<const uint32_t*>(s.act);
    const int mq = lane >> 3, rr = lane & 7;
    const uint32_t aoff = (uint32_t)(((mq & 1) * 8 + rr) * 128);  // A: matrices 1, 3 = rows 8-15
    const int i = lane >> 2, m = lane & 3;                          // result lane: row i of 8, token m
    // norm ops: the RMSNorm scale applies to row sums (a column split adds it in the epilogue)
    const float rs = (op.norm && !op.csplit) ? rstd(m < M ? m : 0) : 1.f;
    Tile t;
    bool ok = true;
    if (op.csplit && it.kw0 >= it.kw1)  // a warp without columns contributes zeros
      for (int k = lane; k < (it.bw - it.aw) * M; k += 32) parts[warp * (it.bw - it.aw) * M + k] = 0.f;
    while (it.next(t)) {
      uint8_t* slot;
      uint32_t eb;
      if (!next_slot(oi, slot, eb)) {
        ok = false;
        break;
      }
      const uint32_t sb = smem_addr(slot);
      const int ns = t.kn >> 4, kg0 = t.kc >> 4;
#pragma unroll 4
      for (int j = 0; j < ns; ++j) {
        const int c = ((j & 3) << 1) + (mq >> 1);  // 16-byte column chunk within the 64-column box
        uint32_t af[4];
        ldsm_x4(sb + (uint32_t)((j >> 2) * kGemvTcRows * 128) + aoff + (uint32_t)((c ^ rr) << 4), af);
        const uint2 b = *reinterpret_cast<const uint2*>(bf + ((kg0 + j) * 32 + lane) * 2);
        mma_bf16_16816(d, af, b.x, b.y);
      }
      release(eb);
      if (!t.last_k) continue;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int src = 4 * i + (m >> 1);
        const float x0 = __shfl_sync(0xffffffffu, half ? d[2] : d[0], src);
        const float x1 = __shfl_sync(0xffffffffu, half ? d[3] : d[1], src);
        const float y0 = __shfl_sync(0xffffffffu, half ? d[2] : d[0], src + 2);
        const float y1 = __shfl_sync(0xffffffffu, half ? d[3] : d[1], src + 2);
        const float v = ((m & 1) ? x1 + y1 : x0 + y0) * rs;
        const int r0 = t.r0 + 8 * half, nr = min(8, t.nr - 8 * half);
        if (nr <= 0) break;
        const bool mine = lane < nr * MT && m < M;
        if (op.csplit) {  // column split: this warp's partial sums, added across warps afterwards
          if (mine) parts[(warp * (it.bw - it.aw) + (r0 + i - a)) * M + m] = v;
          continue;
        }
        switch (op.type) {
          case OP_QKV:
          case OP_ROUTER:
            if (mine) st_tagged(op.out + (size_t)m * op.N + r0 + i, v, tag);
            break;
          case OP_OPROJ:
          case OP_DOWN:
            if (mine) put_x(op, m, r0 + i, xres[(r0 + i - a) * M + m] + v);
            break;
          case OP_GATEUP: {
            const float g = __shfl_sync(0xffffffffu, v, ((2 * i) * MT + m) & 31);
            const float u = __shfl_sync(0xffffffffu, v, ((2 * i + 1) * MT + m) & 31);
            if (lane < (nr / 2) * MT && m < M) st_tagged(op.out + (size_t)m * (op.N / 2) + r0 / 2 + i, silu(g) * u, tag);
            break;
          }
          case OP_LMHEAD:
            if (mine) {
              const int row = r0 + i;
              op.logits[(size_t)m * op.N + row] = v;
              if (v > best_v || (v == best_v && row < best_i)) {
                best_v = v;
                best_i = row;
              }
            }
            break;
          default:
            break;
        }
      }
      d[0] = d[1] = d[2] = d[3] = 0.f;
    }
    if (op.type == OP_LMHEAD) {
      // lane l tracked token l % 4, as on the CUDA-core path
      s.resw[warp * 64 + lane] = best_v;
      reinterpret_cast<int*>(s.resw)[warp * 64 + 32 + lane] = best_i;
    }
    return ok;
  }

  // Instantiations: tile rows NR (bf16 2/4/8, FP8 4/8, MXFP4 8; the host's R fits) and, for
  // one token, the register chunks NI the warp's columns need (0: activations stay in shared
  // memory). The host only makes column-split ops whose columns fit in registers.
  template <int MT>
  __device__ bool gemv_dispatch(int oi, const OpDesc& op, int M, float* xres, int a, float* accd) {
    if constexpr (MT == kMmax)
      if (op.tc) return gemv_tc_entry(p, oi, op, M, xres, a, accd);
    const int kw = op.csplit ? op.Kc : op.K;  // columns one warp multiplies
    const bool whole = op.csplit || (op.Kc == op.K && op.type != OP_EXP_DOWN);
    if (op.wtype == W_BF16) {
      const int ni = (MT == 1 && whole) ? (kw <= 32 * 4 * 8 ? 4 : (kw <= 32 * 10 * 8 ? 10 : 0)) : 0;
      if (op.csplit) {
        if constexpr (MT == 1) {
          if (ni == 4) return gemv_csplit_entry<W_BF16, 1, 8, 4>(p, oi, op, M, a, accd);
          return gemv_csplit_entry<W_BF16, 1, 8, 10>(p, oi, op, M, a, accd);
        } else {
          return gemv_csplit_entry<W_BF16, MT, 8, 0>(p, oi, op, M, a, accd);
        }
      }
      if constexpr (MT == 1) {
        if (ni == 4) {
          if (op.R <= 2) return gemv_tiles_entry<W_BF16, 1, 2, 4>(p, oi, op, M, xres, a, accd);
          if (op.R <= 4) return gemv_tiles_entry<W_BF16, 1, 4, 4>(p, oi, op, M, xres, a, accd);
          return gemv_tiles_entry<W_BF16, 1, 8, 4>(p, oi, op, M, xres, a, accd);
        }
        if (ni == 10) {
          if (op.R <= 2) return gemv_tiles_entry<W_BF16, 1, 2, 10>(p, oi, op, M, xres, a, accd);
          if (op.R <= 4) return gemv_tiles_entry<W_BF16, 1, 4, 10>(p, oi, op, M, xres, a, accd);
          return gemv_tiles_entry<W_BF16, 1, 8, 10>(p, oi, op, M, xres, a, accd);
        }
      }
      if (op.R <= 2) return gemv_tiles_entry<W_BF16, MT, 2, 0>(p, oi, op, M, xres, a, accd);
      if (op.R <= 4) return gemv_tiles_entry<W_BF16, MT, 4, 0>(p, oi, op, M, xres, a, accd);
      return gemv_tiles_entry<W_BF16, MT, 8, 0>(p, oi, op, M, xres, a, accd);
    }
    if (op.wtype == W_FP8) {
      const bool regs = MT == 1 && whole && kw <= 32 * 5 * 16;
      if (op.csplit) {
        if constexpr (MT == 1) return gemv_csplit_entry<W_FP8, 1, 8, 5>(p, oi, op, M, a, accd);
        else return gemv_csplit_entry<W_FP8, MT, 8, 0>(p, oi, op, M, a, accd);
      }
      if constexpr (MT == 1) {
        if (regs) {
          if (op.R <= 4) return gemv_tiles_entry<W_FP8, 1, 4, 5>(p, oi, op, M, xres, a, accd);
          return gemv_tiles_entry<W_FP8, 1, 8, 5>(p, oi, op, M, xres, a, accd);
        }
      }
      if (op.R <= 4) return gemv_tiles_entry<W_FP8, MT, 4, 0>(p, oi, op, M, xres, a, accd);
      return gemv_tiles_entry<W_FP8, MT, 8, 0>(p, oi, op, M, xres, a, accd);
    }
    // MXFP4 keeps its activations in shared memory: decoding is the bottleneck there, and a
    // register copy would spill (measured: 10 % faster on the MoE stack)
    return gemv_tiles_entry<W_MXFP4, MT, 8, 0>(p, oi, op, M, xres, a, accd);
  }

  // Expert down, one slot (its hidden vectors staged in act by the caller).
  template <int MT>
  __device__ __forceinline__ bool gemv_slot(int oi, const OpDesc& op, int sl, int M, int a, float* accd) {
    int ca, cb, aw, bw;
    cta_rows(op.N, op.unit, p.n_ctas, blockIdx.x, ca, cb);
    warp_rows(ca, cb, op.unit, warp, aw, bw);
    Acc<8, MT> A;
    const int i = lane / MT, m = lane % MT;
    for (int r = aw; r < bw; r += op.R) {
      const int nr = min(op.R, bw - r);
      acc_zero(A);
      for (int kc = 0; kc < op.K; kc += op.Kc) {
        uint8_t* slot;
        uint32_t eb;
        if (!next_slot(oi, slot, eb)) return false;
        warp_gemv<W_MXFP4, MT, 8>(slot, nr, min(op.Kc, op.K - kc), kc, s.act, op.K, M, A, lane);
        release(eb);
      }
      const float v = warp_rowsums<8, MT>(A, nr, lane);
      if (lane < nr * MT && m < M) accd[(r + i - a) * M + m] += s.route->w[m][sl] * v;
    }
    return true;
  }

  // Rows [a, b) of the CTA, and where its residual rows (xres) and partial sums (accd) sit in
  // s.act; the same in all three phases of a matrix op.
  struct GemvGeo {
    int a, b;
    float* xres;
    float* accd;
  };
  __device__ __forceinline__ GemvGeo gemv_geo(const OpDesc& op, int M) const {
    GemvGeo g{0, 0, nullptr, nullptr};
    switch (op.type) {
      case OP_OPROJ:
      case OP_DOWN:
        cta_rows(op.N, op.unit, p.n_ctas, blockIdx.x, g.a, g.b);
        g.xres = s.act + (op.tc ? kMmax : M) * op.K;  // tensor-core B operand: kMmax tokens' bytes
        if (op.csplit) g.accd = g.xres + (g.b - g.a) * M;  // per-warp partial sums
        break;
      case OP_EXP_DOWN: {
        cta_rows(op.N, op.unit, p.n_ctas, blockIdx.x, g.a, g.b);
        const int hfl = op.stage_all ? s.route->n_slots * M * op.K : M * op.K;
        g.xres = s.act + hfl;
        g.accd = g.xres + (g.b - g.a) * M;
        break;
      }
      default:
        if (op.csplit) {
          cta_rows(op.N, op.unit, p.n_ctas, blockIdx.x, g.a, g.b);
          g.accd = s.act + (op.tc ? kMmax : M) * op.K;  // per-warp partial sums
        }
        break;
    }
    return g;
  }

  // Phase 1 of a matrix op: wait for its input, then poll the activations every tile multiplies
  // and the residual rows of this CTA into shared memory.
  __device__ __forceinline__ bool gemv_prologue(int oi, const OpDesc& op, int M) {
    // the gain is a weight: load it before waiting for the input
    uint2 gpre[kGainPre];
    load_gain(op, gpre);
    if (op.wait_ctr >= 0 && !wait_counter(op.wait_ctr, op.wait_n, oi, 4)) return false;
    if (tid == 0) TRACE(p, oi, 1, gtimer());
    if ((op.type == OP_ROUTED_GATEUP || op.type == OP_EXP_DOWN) && !routing_entry(p, oi, M)) return false;
    const int cw = chunk_width(op.wtype);
    const GemvGeo g = gemv_geo(op, M);
    bool ok = true;
    switch (op.type) {
      case OP_OPROJ:
      case OP_DOWN:
        ok &= copy_act(s.act, op.act, M, op.K, op.K, op.tc ? 0 : cw, oi);
        if (tid == 0) TRACE(p, oi, 8, gtimer());
        ok &= load_residual(op, g.xres, g.a, g.b, M, oi);
        break;
      case OP_EXP_DOWN:
        ok &= load_residual(op, g.xres, g.a, g.b, M, oi);
        // partial sums: one set per warp in the slot split, one for the CTA otherwise
        for (int t = tid; t < (op.csplit ? kConsumerWarps : 1) * (g.b - g.a) * M; t += kConsumerThreads) g.accd[t] = 0.f;
        if (op.stage_all)
          for (int sl = 0; sl < s.route->n_slots; ++sl)
            ok &= copy_act(s.act + (size_t)sl * M * op.K, op.eh + (size_t)sl * p.Mmax * op.K, M, op.K, op.K, cw, oi);
        break;
      default:
        ok &= norm_prologue(op, M, gpre, oi);
        break;
    }
    if (!consumer_all(ok)) return false;
    if (tid == 0) {
      TRACE(p, oi, 2, gtimer());
      TRACE(p, oi, 9, (uint64_t)s.flags[kFlagLate]);
    }
    return true;
  }

  // Phase 2: every warp's tiles (out-of-line tile loops).
  __device__ __forceinline__ bool gemv_tiles(int oi, const OpDesc& op, int M) {
    const GemvGeo g = gemv_geo(op, M);
    if (op.type == OP_EXP_DOWN && !op.stage_all) {
      // one slot at a time: stage its hidden vectors, then every warp runs its rows of it
      const int n_slots = s.route->n_slots, cw = chunk_width(op.wtype);
      for (int sl = 0; sl < n_slots; ++sl) {
        const bool ok = copy_act_entry(p, oi, s.act, op.eh + (size_t)sl * p.Mmax * op.K, M, op.K, op.K, cw);
        if (!consumer_all(ok)) return false;
        const bool r = M == 1 ? gemv_slot_entry<1>(p, oi, op, sl, M, g.a, g.accd)
                              : gemv_slot_entry<4>(p, oi, op, sl, M, g.a, g.accd);
        if (!consumer_all(r)) return false;
      }
    } else if (op.type == OP_EXP_DOWN && op.csplit) {
      bool r;
      if (M == 1)  // activations from shared memory: a register copy of the slot's would spill
        r = gemv_xsplit_entry<1, 10, 0>(p, oi, op, M, g.a, g.accd);
      else
        r = gemv_xsplit_entry<4, 8, 0>(p, oi, op, M, g.a, g.accd);
      if (!consumer_all(r)) return false;
    } else {
      const bool r = M == 1 ? gemv_dispatch<1>(oi, op, M, g.xres, g.a, g.accd)
                            : gemv_dispatch<4>(oi, op, M, g.xres, g.a, g.accd);
      if (!consumer_all(r)) return false;
    }
    if (tid == 0) TRACE(p, oi, 3, gtimer());
    return true;
  }

  // Phase 3: outputs that need every warp's results (column-split sums, expert-down residual
  // stores, the LM head's argmax) and the router's routing.
  __device__ __forceinline__ bool gemv_epilogue(int oi, const OpDesc& op, int M) {
    const GemvGeo g = gemv_geo(op, M);
    if (op.csplit) csplit_epilogue(op, M, g.a, g.b, g.xres, g.accd);
    if (op.type == OP_EXP_DOWN && !op.csplit) {
      for (int t = tid; t < (g.b - g.a) * M; t += kConsumerThreads) {
        const int i = t / M, m = t % M;
        put_x(op, m, g.a + i, g.xres[t] + g.accd[t]);
      }
    }
    if (op.type == OP_ROUTER) {
      arrive(op.ctr);  // before the routing, which waits for every CTA's logits
      return routing_entry(p, oi, M);
    }
    if (op.type == OP_LMHEAD) lmhead_finish(op, M);
    return true;
  }

  // Per-warp bests -> per-CTA partial -> the last CTA reduces all partials (lowest index on ties).
  __device__ __forceinline__ void lmhead_finish(const OpDesc& op, int M) {
    consumer_sync();
    const int MT = M == 1 ? 1 : 4;  // lane l of a warp tracked token l % MT
    {
      // this CTA's best per token: the lanes of each warp that tracked the same token, by
      // shuffles; then the warps' bests (lowest index among equal logits throughout)
      float v = s.resw[warp * 64 + lane];
      int i = reinterpret_cast<const int*>(s.resw)[warp * 64 + 32 + lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (o >= MT && (ov > v || (ov == v && oi < i))) {
          v = ov;
          i = oi;
        }
      }
      if (lane < MT) {
        s.red[lane * 8 + warp] = v;
        reinterpret_cast<int*>(s.red)[32 + lane * 8 + warp] = i;
      }
    }
    consumer_sync();
    if (tid < M) {
      float v = -INFINITY;
      int i = 0x7FFFFFFF;
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float wv = s.red[tid * 8 + w];
        const int wi = reinterpret_cast<const int*>(s.red)[32 + tid * 8 + w];
        if (wv > v || (wv == v && wi < i)) {
          v = wv;
          i = wi;
        }
      }
      p.am_val[blockIdx.x * kMmax + tid] = v;
      p.am_idx[blockIdx.x * kMmax + tid] = i;
    }
    if (ticket(op.ticket, p.n_ctas)) {
      // the last CTA reduces every CTA's best in parallel: each thread loads the partials of its
      // CTAs (all tokens' loads in flight together), then warps, then the warps' bests
      float v[kMmax];
      int ix[kMmax];
#pragma unroll
      for (int m = 0; m < kMmax; ++m) {
        v[m] = -INFINITY;
        ix[m] = 0x7FFFFFFF;
      }
      for (int c = tid; c < p.n_ctas; c += kConsumerThreads) {
        float cv[kMmax];
        int ci[kMmax];
#pragma unroll
        for (int m = 0; m < kMmax; ++m) {
          cv[m] = m < M ? __ldcg(p.am_val + c * kMmax + m) : -INFINITY;
          ci[m] = m < M ? __ldcg(p.am_idx + c * kMmax + m) : 0x7FFFFFFF;
        }
#pragma unroll
        for (int m = 0; m < kMmax; ++m)
          if (cv[m] > v[m] || (cv[m] == v[m] && ci[m] < ix[m])) {
            v[m] = cv[m];
            ix[m] = ci[m];
          }
      }
#pragma unroll
      for (int m = 0; m < kMmax; ++m) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, v[m], o);
          const int oi = __shfl_xor_sync(0xffffffffu, ix[m], o);
          if (ov > v[m] || (ov == v[m] && oi < ix[m])) {
            v[m] = ov;
            ix[m] = oi;
          }
        }
        if (lane == 0) {
          s.red[m * 8 + warp] = v[m];
          s.resw[m * 8 + warp] = __int_as_float(ix[m]);
        }
      }
      consumer_sync();
      if (tid < M) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float wv = s.red[tid * 8 + w];
          const int wi = __float_as_int(s.resw[tid * 8 + w]);
          if (wv > bv || (wv == bv && wi < bi)) {
            bv = wv;
            bi = wi;
          }
        }
        p.am_out[tid] = bi < p.V ? bi : 0;  // no ordered logit (NaN inputs): a valid token, never a wild one
      }
    }
  }

  // ---------------------------------------------------------------- attention on tensor cores
  // One warp, token m_tok's G_ heads over the cached rows [r0, r1) of the current split, in
  // tiles of kAttnTcRows rows that the producer brought by TMA with a 128-byte swizzle (keys in
  // two 64-column boxes, then values in two). Scores S = Q K^T and outputs O = P V are warp-level
  // bf16 MMAs (m16n8k16) with fp32 accumulation; the 16 rows of the A operand hold the G_ heads
  // twice, as bf16 high parts (rows 0-7) and the bf16 rounding residues (rows 8-15), so q and p
  // keep about 16 bits of mantissa and the two rows' products add up in fp32. Online softmax in
  // base 2 on the score fragments; the state (max, sum, output) goes to the warp's merge slice.
  template <int G_>
  __device__ __forceinline__ bool attn_tc_t(int oi, int r0, int r1, int m_tok, int M, int lo_m) {
    static_assert(G_ <= 8, "at most 8 query heads per kv head on the tensor-core path");
    const int P = kAttnTcRows;
    const AttnScratch a = attn_scratch(p, s, M, P);
    const int g = lane >> 2, tq = lane & 3;
    // Q fragments per 16-column step: rows g (high parts) and g + 8 (residues) of head g
    uint32_t qf[8][4];
    {
      const float* qr = a.q + (m_tok * G_ + (g < G_ ? g : 0)) * 128;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int d0 = 16 * kk + 2 * tq;
        float x[4] = {qr[d0], qr[d0 + 1], qr[d0 + 8], qr[d0 + 9]};
        if (g >= G_) x[0] = x[1] = x[2] = x[3] = 0.f;
        float hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hi[e] = __bfloat162float(__float2bfloat16_rn(x[e]));
          lo[e] = x[e] - hi[e];
        }
        qf[kk][0] = pack_bf16x2(hi[0], hi[1]);
        qf[kk][1] = pack_bf16x2(lo[0], lo[1]);
        qf[kk][2] = pack_bf16x2(hi[2], hi[3]);
        qf[kk][3] = pack_bf16x2(lo[2], lo[3]);
      }
    }
    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float mrun = -INFINITY, lrun = 0.f;
    // this lane's row of the 8x8 matrices it addresses for ldmatrix, and its swizzle phase
    const int mq = lane >> 3, rr = lane & 7;
    const uint32_t koff = (uint32_t)(((mq >> 1) * 8 + rr) * 128);  // keys: matrices 2, 3 = rows 8-15
    const uint32_t voff = (uint32_t)(((mq & 1) * 8 + rr) * 128);   // values: matrices 1, 3 = rows 8-15
    bool ok = true;
    for (int r = r0; r < r1; r += P) {
      const int nr = min(P, r1 - r);
      uint8_t* slot;
      uint32_t eb;
      if (!next_slot(oi, slot, eb)) {
        ok = false;
        break;
      }
      const uint32_t kb = smem_addr(slot), vb = kb + 2 * kAttnTcBoxBytes;
      float sc4[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int c = 2 * kk + (mq & 1);  // 16-byte column chunk of the 128 dims
        uint32_t b[4];
        ldsm_x4(kb + (uint32_t)((c >> 3) * kAttnTcBoxBytes) + koff + (uint32_t)((((c & 7) ^ rr)) << 4), b);
        mma_bf16_16816(sc4[0], qf[kk], b[0], b[1]);
        mma_bf16_16816(sc4[1], qf[kk], b[2], b[3]);
      }
      // scores of head g at rows 8j + 2 tq + e (high + residue rows), masked past the tile
      float sv[2][2], mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = 8 * j + 2 * tq + e;
          sv[j][e] = (row < nr && r + row >= lo_m) ? sc4[j][e] + sc4[j][2 + e] : -INFINITY;
          mx = fmaxf(mx, sv[j][e]);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mnew = fmaxf(mrun, mx);
      const float scale = (mnew == -INFINITY) ? 1.f : (mrun == -INFINITY ? 0.f : exp2f(mrun - mnew));
      float pv[2][2], psum = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pv[j][e] = (sv[j][e] == -INFINITY) ? 0.f : exp2f(sv[j][e] - mnew);
          psum += pv[j][e];
        }
      lrun = lrun * scale + psum;
      mrun = mnew;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= scale;
        o[j][1] *= scale;
        o[j][2] *= scale;
        o[j][3] *= scale;
      }
      uint32_t pf[4];
      {
        float hi[2][2], lo[2][2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            hi[j][e] = __bfloat162float(__float2bfloat16_rn(pv[j][e]));
            lo[j][e] = pv[j][e] - hi[j][e];
          }
        pf[0] = pack_bf16x2(hi[0][0], hi[0][1]);
        pf[1] = pack_bf16x2(lo[0][0], lo[0][1]);
        pf[2] = pack_bf16x2(hi[1][0], hi[1][1]);
        pf[3] = pack_bf16x2(lo[1][0], lo[1][1]);
      }
      if (nr < P) {
        // value rows past the tile may hold anything the cache holds there: zero them, so a
        // zero probability never meets a non-finite value
        __syncwarp();
        for (int i = lane; i < (P - nr) * 16; i += 32) {
          const int row = nr + i / 16, ch = i % 16;
          *reinterpret_cast<uint4*>(slot + 2 * kAttnTcBoxBytes + (ch >> 3) * kAttnTcBoxBytes + row * 128 +
                                    ((ch & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the slot's next bulk fill comes after these writes
        __syncwarp();
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int c = 2 * jj + (mq >> 1);  // 16-byte column chunk: dims 8c .. 8c + 7
        uint32_t b[4];
        ldsm_x4_t(vb + (uint32_t)((c >> 3) * kAttnTcBoxBytes) + voff + (uint32_t)((((c & 7) ^ rr)) << 4), b);
        mma_bf16_16816(o[2 * jj], pf, b[0], b[1]);
        mma_bf16_16816(o[2 * jj + 1], pf, b[2], b[3]);
      }
      release(eb);
    }
    // the warp's state: head g's max, sum (its four lanes' parts) and output dims 8j + 2 tq + e
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 1);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 2);
    float* mgw = a.mg + warp * G_ * kPart;
    if (g < G_) {
      if (tq == 0) {
        mgw[g * kPart] = mrun;
        mgw[g * kPart + 1] = lrun;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int d = 8 * j + 2 * tq;
        mgw[g * kPart + 4 + d] = o[j][0] + o[j][2];
        mgw[g * kPart + 4 + d + 1] = o[j][1] + o[j][3];
      }
    }
    __syncwarp();
    return ok;
  }

  // ---------------------------------------------------------------- attention op
  template <int G_>
  __device__ __forceinline__ bool attn_op(int oi, const OpDesc& op, int pos, int M) {
    if (op.wait_ctr >= 0 && !wait_counter(op.wait_ctr, op.wait_n, oi, 4)) return false;
    if (tid == 0) TRACE(p, oi, 1, gtimer());
    const int P = attn_rows(p, s.slot_bytes);
    const int rb = kv_row_bytes(p.kv_fp8);
    const int G = G_, MG = M * G, ns = p.ns_max;
    const AttnScratch a = attn_scratch(p, s, M, P);
    const float qscale = 1.4426950408889634f / sqrtf(128.f);  // log2(e) / sqrt(d)
    int m_tok, gi, ng;
    token_group(warp, M, m_tok, gi, ng);
    // this warp's token (at pos + m_tok) sees cached positions from lo_m on
    const int lo_m = p.attn_window > 0 ? max(0, pos + m_tok - p.attn_window + 1) : 0;
    AttnIter it;
    it.init(p, blockIdx.x, warp, pos, M, P);
    float* sc = a.sc + warp * G * P;
    const uint64_t* qkv = op.act;
    const size_t sstride = (size_t)p.Mmax * G * kPart;  // words per split partial
    uint64_t* lpart = p.part + (size_t)op.layer * p.n_kv * ns * sstride;
    const int GR = (G + 2) * 32;  // float4 groups of one token's q, k, v rows of the kv group
    for (; it.j < it.nsplit; it.next_split()) {
      int head, sidx, p0, p1;
      split_range(it.lo, it.S, ns, it.j, head, sidx, p0, p1);
      const int nb = max(p0, pos), nn = max(0, p1 - nb);  // this call's own rows in the split
      // CTA prologue: poll the group's q (and, for the split holding this call's rows, k and v)
      // in one batch; rotate and scale the queries; round, keep and append the own rows
      const int per_m = nn > 0 ? GR : G * 32;
      bool ok = gather<4, 4>(
          M * per_m,
          [&](int i) {
            const int m = i / per_m, r = i - m * per_m;
            const uint64_t* row = qkv + (size_t)m * p.qkv_rows;
            if (r < G * 32) return row + head * G * 128 + 4 * r;
            if (r < (G + 1) * 32) return row + (p.n_q + head) * 128 + 4 * (r - G * 32);
            return row + (p.n_q + p.n_kv + head) * 128 + 4 * (r - (G + 1) * 32);
          },
          [&](int i, const float (&v)[4]) {
            const int m = i / per_m, r = i - m * per_m;
            *reinterpret_cast<float4*>(a.raw + (m * GR + r) * 4) = make_float4(v[0], v[1], v[2], v[3]);
          },
          oi, 11);
      if (!consumer_all(ok)) return false;
      for (int idx = tid; idx < MG * 64; idx += kConsumerThreads) {
        const int mh = idx >> 6, i = idx & 63;
        const int m = mh / G;
        const float* qr = a.raw + m * GR * 4 + (mh % G) * 128;
        const float x1 = qr[i], x2 = qr[i + 64];
        const float2 cs = s.rope[m * 64 + i];
        a.q[mh * 128 + i] = (x1 * cs.x - x2 * cs.y) * qscale;
        a.q[mh * 128 + i + 64] = (x1 * cs.y + x2 * cs.x) * qscale;
      }
      // FP8 cache: this layer's key / value scales of the group's kv head (1 without scales)
      const float sk = p.kv_fp8 && op.kv_scale ? op.kv_scale[head] : 1.f;
      const float sv = p.kv_fp8 && op.kv_scale ? op.kv_scale[p.n_kv + head] : 1.f;
      for (int idx = tid; idx < nn * 64; idx += kConsumerThreads) {
        const int r = idx >> 6, i = idx & 63;
        const int m = nb - pos + r;
        const float* kr = a.raw + m * GR * 4 + G * 128;
        const float* vr = kr + 128;
        const float2 cs = s.rope[m * 64 + i];
        const float k1 = kr[i] * cs.x - kr[i + 64] * cs.y, k2 = kr[i] * cs.y + kr[i + 64] * cs.x;
        const size_t row = (size_t)head * p.cap + pos + m;  // append to the KV history
        if (p.kv_fp8) {
          // e4m3fn of x / s: the fp32 quotient rounded to nearest even, saturated to +-448
          const uint8_t b1 = e4m3_rn_satfinite(__fdiv_rn(k1, sk)), b2 = e4m3_rn_satfinite(__fdiv_rn(k2, sk));
          const uint8_t c1 = e4m3_rn_satfinite(__fdiv_rn(vr[i], sv)), c2 = e4m3_rn_satfinite(__fdiv_rn(vr[i + 64], sv));
          uint8_t* kvn8 = reinterpret_cast<uint8_t*>(a.kvn);
          kvn8[r * 128 + i] = b1;
          kvn8[r * 128 + i + 64] = b2;
          kvn8[(nn + r) * 128 + i] = c1;
          kvn8[(nn + r) * 128 + i + 64] = c2;
          op.kc[row * 128 + i] = b1;
          op.kc[row * 128 + i + 64] = b2;
          op.vc[row * 128 + i] = c1;
          op.vc[row * 128 + i + 64] = c2;
        } else {
          const uint16_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(k1));
          const uint16_t b2 = __bfloat16_as_ushort(__float2bfloat16_rn(k2));
          const uint16_t c1 = __bfloat16_as_ushort(__float2bfloat16_rn(vr[i]));
          const uint16_t c2 = __bfloat16_as_ushort(__float2bfloat16_rn(vr[i + 64]));
          a.kvn[r * 128 + i] = b1;
          a.kvn[r * 128 + i + 64] = b2;
          a.kvn[(nn + r) * 128 + i] = c1;
          a.kvn[(nn + r) * 128 + i + 64] = c2;
          uint16_t* kc16 = reinterpret_cast<uint16_t*>(op.kc);
          uint16_t* vc16 = reinterpret_cast<uint16_t*>(op.vc);
          kc16[row * 128 + i] = b1;
          kc16[row * 128 + i + 64] = b2;
          vc16[row * 128 + i] = c1;
          vc16[row * 128 + i + 64] = c2;
        }
      }
      consumer_sync();
      if (tid == 0 && it.j == (int)blockIdx.x) {
        TRACE(p, oi, 2, gtimer());
      }
      // per warp: token m_tok's G heads over this warp's share of the cached rows
      AttnState<G_> A;
#pragma unroll
      for (int h = 0; h < G_; ++h) {
        A.mrun[h] = -INFINITY;
        A.lrun[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) A.o[h][e] = 0.f;
      }
      float q[G_][16];
      const int sub = lane & 7;
      auto load_q = [&]() {
#pragma unroll
        for (int h = 0; h < G_; ++h)
#pragma unroll
          for (int e = 0; e < 16; ++e) q[h][e] = a.q[(m_tok * G + h) * 128 + sub * 16 + e] * sk;
      };
      Tile t;
      if (p.attn_tc) {
        // the cached rows on the tensor cores (out of line); the warp's state comes back
        // through its slice of the merge scratch
        if (it.fresh) it.enter_split();
        save_tiles();
        if (!attn_tc_entry<G_>(p, oi, it.q, it.qe, m_tok, M, lo_m)) ok = false;
        n_tiles = s.ntiles[warp];
        it.q = it.qe;
        load_q();  // for this call's own rows, after the call (nothing to keep live across it)
        const float* mgw = a.mg + warp * G * kPart;
#pragma unroll
        for (int h = 0; h < G_; ++h) {
          A.mrun[h] = mgw[h * kPart];
          A.lrun[h] = mgw[h * kPart + 1];
#pragma unroll
          for (int e = 0; e < 4; ++e) A.o[h][e] = mgw[h * kPart + 4 + lane * 4 + e];
        }
        __syncwarp();
      } else {
        load_q();
        while (it.next_in_split(t)) {
          uint8_t* slot;
          uint32_t eb;
          if (!next_slot(oi, slot, eb)) {
            ok = false;
            break;
          }
          if (p.kv_fp8)
            attn_warp_tile<G_, true>(A, q, slot, slot + t.nr * rb, t.nr, -1, m_tok, sc, P, lane, t.r0, lo_m);
          else
            attn_warp_tile<G_, false>(A, q, slot, slot + t.nr * rb, t.nr, -1, m_tok, sc, P, lane, t.r0, lo_m);
          release(eb);
        }
      }
      // this call's own rows: the first warp of each token group attends to them (causally)
      if (ok && gi == 0 && nn > 0) {
        const uint8_t* kn = reinterpret_cast<const uint8_t*>(a.kvn);
        if (p.kv_fp8)
          attn_warp_tile<G_, true>(A, q, kn, kn + nn * rb, nn, nb - pos, m_tok, sc, P, lane);
        else
          attn_warp_tile<G_, false>(A, q, kn, kn + nn * rb, nn, nb - pos, m_tok, sc, P, lane);
      }
      // per-warp state -> shared memory; merge the warps of each token into the split partial
      float* mg = a.mg + warp * G * kPart;
#pragma unroll
      for (int h = 0; h < G_; ++h) {
        if (lane == 0) {
          mg[h * kPart] = A.mrun[h];
          mg[h * kPart + 1] = A.lrun[h];
        }
        // FP8 cache: the value codes were summed unscaled; sv is 1 for bf16
        *reinterpret_cast<float4*>(mg + h * kPart + 4 + lane * 4) =
            make_float4(A.o[h][0] * sv, A.o[h][1] * sv, A.o[h][2] * sv, A.o[h][3] * sv);
      }
      if (!consumer_all(ok)) return false;
      if (tid == 0) TRACE(p, oi, 3, gtimer());
      // the split's partial, every word tagged (the two pad words too: the merge polls the
      // (max, sum) pair as one 4-word item)
      uint64_t* part = lpart + (size_t)(head * ns + sidx) * sstride;
      for (int idx = tid; idx < MG * kPart; idx += kConsumerThreads) {
        const int mh = idx / kPart, e = idx % kPart;
        const int m = mh / G, h = mh % G;
        float val = 0.f;
        if (e != 2 && e != 3) {
          float mx = -INFINITY;
          for (int w = m; w < kConsumerWarps; w += M) mx = fmaxf(mx, a.mg[(w * G + h) * kPart]);
          float l = 0.f, o = 0.f;
          for (int w = m; w < kConsumerWarps; w += M) {
            const float mw = a.mg[(w * G + h) * kPart];
            const float f = mw == -INFINITY ? 0.f : exp2f(mw - mx);
            l += f * a.mg[(w * G + h) * kPart + 1];
            if (e >= 4) o += f * a.mg[(w * G + h) * kPart + e];
          }
          val = e == 0 ? mx : (e == 1 ? l : o);
        }
        st_tagged(part + mh * kPart + e, val, tag);
      }
      arrive(op.aux_ctr + head);
    }
    // Phase 2: the splits of a kv head merge its outputs together, each split a 1/ns slice
    // (log-sum-exp in base 2). One batch polls every split's (max, sum) of the slice's rows and
    // its share of the outputs. Every split of this CTA was published above before these polls,
    // so no CTA waits on one that waits on it.
    AttnIter it2;
    it2.init(p, blockIdx.x, warp, pos, M, P);
    for (; it2.j < it2.nsplit; it2.next_split()) {
      int head, sidx, p0, p1;
      split_range(it2.lo, it2.S, ns, it2.j, head, sidx, p0, p1);
      const uint64_t* hp = lpart + (size_t)(head * ns) * sstride;
      const int total = MG * 32;  // float4 outputs of this kv head
      const int o0 = (int)((long long)total * sidx / ns), o1 = (int)((long long)total * (sidx + 1) / ns);
      if (o0 >= o1) continue;
      const int mhA = o0 >> 5, mhB = (o1 - 1) >> 5;
      const int nrow = mhB - mhA + 1, nout = o1 - o0, per = nrow + nout;
      float4* outs = reinterpret_cast<float4*>(a.sc);  // [ns][nout]
      if (tid == 0) TRACE(p, oi, 10, gtimer());
      if (!wait_counter(op.aux_ctr + head, ns, oi, 13)) return false;
      if (tid == 0) TRACE(p, oi, 11, gtimer());
      bool ok = gather<4, 4>(
          ns * per,
          [&](int i) {
            const int q2 = i / per, k = i - q2 * per;
            const uint64_t* sp = hp + q2 * sstride;
            if (k < nrow) return sp + (mhA + k) * kPart;
            const int oo = o0 + k - nrow;
            return sp + (oo >> 5) * kPart + 4 + 4 * (oo & 31);
          },
          [&](int i, const float (&v)[4]) {
            const int q2 = i / per, k = i - q2 * per;
            if (k < nrow)
              a.ml[q2 * nrow + k] = make_float2(v[0], v[1]);
            else
              outs[q2 * nout + k - nrow] = make_float4(v[0], v[1], v[2], v[3]);
          },
          oi, 13);
      if (!consumer_all(ok)) return false;
      // weights of every split for each row of the slice (one warp per row)
      for (int r = warp; r < nrow; r += kConsumerWarps) {
        float* cw = a.cw + r * ns;
        float mx = -INFINITY;
        for (int q2 = lane; q2 < ns; q2 += 32) mx = fmaxf(mx, a.ml[q2 * nrow + r].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float l = 0.f;
        for (int q2 = lane; q2 < ns; q2 += 32) {
          const float2 ml = a.ml[q2 * nrow + r];
          const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mx);
          cw[q2] = w;
          l += w * ml.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        const float inv = 1.0f / l;
        for (int q2 = lane; q2 < ns; q2 += 32) cw[q2] *= inv;
      }
      consumer_sync();
      // each output vector: a warp sums the splits' weighted slices (lanes over splits, then a
      // fixed butterfly)
      for (int k = warp; k < nout; k += kConsumerWarps) {
        const int oo = o0 + k, mh = oo >> 5, d4 = oo & 31;
        const float* cw = a.cw + (mh - mhA) * ns;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q2 = lane; q2 < ns; q2 += 32) {
          const float w = cw[q2];
          const float4 v = outs[q2 * nout + k];
          o.x = fmaf(w, v.x, o.x);
          o.y = fmaf(w, v.y, o.y);
          o.z = fmaf(w, v.z, o.z);
          o.w = fmaf(w, v.w, o.w);
        }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) {
          o.x += __shfl_xor_sync(0xffffffffu, o.x, sh);
          o.y += __shfl_xor_sync(0xffffffffu, o.y, sh);
          o.z += __shfl_xor_sync(0xffffffffu, o.z, sh);
          o.w += __shfl_xor_sync(0xffffffffu, o.w, sh);
        }
        if (lane == 0) {
          const int m = mh / G, h = head * G + mh % G;
          st_tagged4(op.out + (size_t)m * p.n_q * 128 + h * 128 + d4 * 4, o, tag);
        }
      }
      consumer_sync();
    }
    return true;
  }

  // ---------------------------------------------------------------- main loop
  __device__ __forceinline__ bool run(int pos, int M) {
    for (int oi = p.op_begin; oi < p.op_end; ++oi) {
      {
        const int* src = reinterpret_cast<const int*>(p.ops + oi);
        int* dst = reinterpret_cast<int*>(s.op);
        for (int i = tid; i < (int)(sizeof(OpDesc) / 4); i += kConsumerThreads) dst[i] = __ldg(src + i);
        if (tid == 0) s.flags[kFlagLate] = 0;
      }
      consumer_sync();
      const OpDesc& op = *s.op;
      if (tid == 0) TRACE(p, oi, 0, gtimer());
      bool ok;
      if (op.type == OP_ATTN) {
        switch (p.G) {
          case 1: ok = attn_entry<1>(p, oi, pos, M); break;
          case 2: ok = attn_entry<2>(p, oi, pos, M); break;
          case 4: ok = attn_entry<4>(p, oi, pos, M); break;
          case 5: ok = attn_entry<5>(p, oi, pos, M); break;
          default: ok = attn_entry<8>(p, oi, pos, M); break;
        }
      } else {
        ok = gemv_prologue_entry(p, oi, M) && gemv_tiles_dispatch_entry(p, oi, M) && gemv_epilogue_entry(p, oi, M);
      }
      if (!ok) return false;
      if (op.type != OP_ROUTER) arrive(op.ctr);  // the router arrives before computing the routing
      else consumer_sync();
      if (tid == 0) TRACE(p, oi, 4, gtimer());
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

// ------------------------------------------------------------------ out-of-line entries
// Each op runs in a function of its own, and each tile loop in one more: every one rebuilds its
// Consumer in registers, so the register allocation of a hot loop is its own.
template <int WT, int MT, int NR, int NI>
__device__ __noinline__ bool gemv_tiles_entry(const KParams& p, int oi, const OpDesc& op, int M, float* xres, int a,
                                              float* accd) {
  Consumer c(p);
  const bool ok = c.gemv_op_t<WT, MT, NR, NI>(oi, op, M, xres, a, accd);
  c.save_tiles();
  return ok;
}

template <int WT, int MT, int NR, int NI>
__device__ __noinline__ bool gemv_csplit_entry(const KParams& p, int oi, const OpDesc& op, int M, int a, float* parts) {
  Consumer c(p);
  const bool ok = c.gemv_csplit_t<WT, MT, NR, NI>(oi, op, M, a, parts);
  c.save_tiles();
  return ok;
}

__device__ __noinline__ bool gemv_tc_entry(const KParams& p, int oi, const OpDesc& op, int M, float* xres, int a,
                                          float* parts) {
  Consumer c(p);
  const bool ok = c.gemv_tc_t(oi, op, M, xres, a, parts);
  c.save_tiles();
  return ok;
}

template <int MT, int NR, int NI>
__device__ __noinline__ bool gemv_xsplit_entry(const KParams& p, int oi, const OpDesc& op, int M, int a, float* parts) {
  Consumer c(p);
  const bool ok = c.gemv_xsplit_t<MT, NR, NI>(oi, op, M, a, parts);
  c.save_tiles();
  return ok;
}

template <int MT>
__device__ __noinline__ bool gemv_slot_entry(const KParams& p, int oi, const OpDesc& op, int sl, int M, int a,
                                             float* accd) {
  Consumer c(p);
  const bool ok = c.gemv_slot<MT>(oi, op, sl, M, a, accd);
  c.save_tiles();
  return ok;
}

__device__ __noinline__ bool gemv_prologue_entry(const KParams& p, int oi, int M) {
  Consumer c(p);
  return c.gemv_prologue(oi, *c.s.op, M);
}

__device__ __noinline__ bool gemv_tiles_dispatch_entry(const KParams& p, int oi, int M) {
  Consumer c(p);
  return c.gemv_tiles(oi, *c.s.op, M);
}

__device__ __noinline__ bool gemv_epilogue_entry(const KParams& p, int oi, int M) {
  Consumer c(p);
  return c.gemv_epilogue(oi, *c.s.op, M);
}

__device__ __noinline__ bool routing_entry(const KParams& p, int oi, int M) {
  Consumer c(p);
  return c.ensure_routing(*c.s.op, M, oi);
}

__device__ __noinline__ bool copy_act_entry(const KParams& p, int oi, float* dst, const uint64_t* src, int M, int K,
                                            int src_stride, int cw) {
  Consumer c(p);
  return c.copy_act(dst, src, M, K, src_stride, cw, oi);
}

template <int G_>
__device__ __noinline__ bool attn_entry(const KParams& p, int oi, int pos, int M) {
  Consumer c(p);
  const bool ok = c.attn_op<G_>(oi, *c.s.op, pos, M);
  c.save_tiles();
  return ok;
}

template <int G_>
__device__ __noinline__ bool attn_tc_entry(const KParams& p, int oi, int r0, int r1, int m_tok, int M, int lo_m) {
  Consumer c(p);
  const bool ok = c.attn_tc_t<G_>(oi, r0, r1, m_tok, M, lo_m);
  c.save_tiles();
  return ok;
}

// Consumers of a chained launch, between steps: the first thread waits (bounded) until the
// step state's epoch moves past this CTA's copy, which the last CTA of the step writes after the
// rest of the state, then copies the state in; every consumer thread learns the verdict.
__device__ __noinline__ bool next_step_state(const KParams& p) {
  bool ok = true;
  consumer_sync();  // every consumer thread is done with the old copy
  if (threadIdx.x == 0) {
    const uint32_t want = g_st.epoch + 1u;
    const volatile uint32_t* e = &p.state->epoch;
    const uint64_t t0 = gtimer();
    for (int it = 1; *e != want; ++it) {
      if ((it & 15) == 0) {
        if (aborted(p)) {
          ok = false;
          break;
        }
        if (gtimer() - t0 > p.timeout_ns) {
          raise_error(p, DEC_ERR_TIMEOUT, -1, 0xFFFFFFFDu, *e, want, 14);
          ok = false;
          break;
        }
      }
    }
    if (ok) {
      __threadfence();
      const uint32_t* src = reinterpret_cast<const uint32_t*>(p.state);
      uint32_t* dst = reinterpret_cast<uint32_t*>(&g_st);
      // every other field first; the epoch last, which the producer lanes poll
      constexpr int kEpochWord = (int)(offsetof(StepState, epoch) / 4);
      for (int i = 0; i < (int)(sizeof(StepState) / 4); ++i)
        if (i != kEpochWord) dst[i] = __ldcg(src + i);
      __threadfence_block();
      *reinterpret_cast<volatile uint32_t*>(&g_st.epoch) = __ldcg(src + kEpochWord);
    }
  }
  return consumer_all(ok);
}

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kThreads, 1) dec_megakernel(const __grid_constant__ KParams p) {
  Smem s = carve(smem_raw, p);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.state);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&g_st);
    for (int i = 0; i < (int)(sizeof(StepState) / 4); ++i) dst[i] = __ldcg(src + i);
    for (int i = 0; i < kConsumerWarps * kStages; ++i) {
      mbar_init(smem_addr(&s.full[i]), 1);
      mbar_init(smem_addr(&s.empty[i]), 1);
    }
    for (int w = 0; w < kConsumerWarps; ++w) s.ntiles[w] = 0;
    s.flags[kFlagRoute] = -1;
    mbar_init_fence();
  }
  __syncthreads();
  const int M = g_st.m;
  if (warp == kConsumerWarps) {
    Producer pr{p, s, g_st.pos, M, l2_policy_evict_first(), g_st.epoch};
    pr.run(lane);
    return;
  }
  for (int step = 0; step < steps_of(p); ++step) {
    // later steps of a chained launch: wait for the step end the last CTA announces, then take
    // the new state (its argmax as the token, the next position)
    if (step > 0 && !next_step_state(p)) return;
    const int pos = g_st.pos;
    // RoPE table of this call's positions (fp64 angle, then fp32 cos/sin).
    for (int t = tid; t < M * 64; t += kConsumerThreads) {
      const int m = t >> 6, i = t & 63;
      const double inv = pow((double)p.rope_base, -2.0 * (double)i / 128.0);
      double sn, cs;
      sincos((double)(pos + m) * inv, &sn, &cs);
      s.rope[t] = make_float2((float)cs, (float)sn);
    }
    consumer_sync();
    Consumer c(p);
    if (!c.run(pos, M)) return;
  }
}

}  // namespace decimpl

// ------------------------------------------------------------------ host launch
namespace {
// Largest dynamic shared-memory size the kernel has been allowed on each device so far.
decimpl::SmemAttrCache g_smem_attr;
}  // namespace

extern "C" cudaError_t dec_launch_megakernel(const decimpl::KParams* kp, int cooperative, cudaStream_t stream) {
  using namespace decimpl;
  const size_t smem = (size_t)kConsumerWarps * kStages * kp->slot_bytes + kp->act_bytes + kCommonBytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = (cudaError_t)g_smem_attr.ensure(dev, smem, [](size_t bytes) {
    return (int)cudaFuncSetAttribute(dec_megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  });
  if (e != cudaSuccess) return e;
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

// Common area plus the kernel's static shared memory, which the dynamic part must leave room for.
extern "C" int dec_megakernel_common_bytes(void) { return decimpl::kCommonBytes + 2048; }
