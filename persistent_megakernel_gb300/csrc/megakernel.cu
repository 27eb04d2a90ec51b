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
              kOffFlags = 7168, kOffRoute = 7232;
constexpr int kFlagTicket = 1;  // flags[kFlagTicket]: verdict of the last ticket
constexpr int kFlagRoute = 8;   // flags[kFlagRoute]: layer + 1 whose routing sits in `route`
static_assert(kConsumerWarps * kStages * 8 <= kOffEmpty - kOffFull, "full barriers");
static_assert(sizeof(OpDesc) <= kOffRed - kOffOp, "OpDesc copy");
static_assert(kOffRoute + sizeof(RouteBlock) <= kCommonBytes, "common area");

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
  s.slot_bytes = p.slot_bytes;
  return s;
}

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

// Poll n (1 or 4) tagged words at src until all carry `tag`; bounded like every wait.
__device__ __noinline__ bool poll_slow(const KParams& p, const uint64_t* src, int n, uint32_t tag, float* out,
                                       int op, uint32_t where) {
  const uint64_t t0 = gtimer();
  for (int it = 1;; ++it) {
    bool all = true;
    for (int i = 0; i < n; ++i) {
      const uint64_t w = ld_tagged(src + i);
      if (tag_of(w) == tag)
        out[i] = value_of(w);
      else
        all = false;
    }
    if (all) return true;
    if ((it & 7) == 0) {
      if (aborted(p)) return false;
      if (gtimer() - t0 > p.timeout_ns) {
        raise_error(p, DEC_ERR_TIMEOUT, op, 0x40000000u, tag_of(ld_tagged(src)), tag, where);
        return false;
      }
    }
  }
}

// Four tagged words at src (16-byte aligned).
__device__ __forceinline__ bool poll4(const KParams& p, const uint64_t* src, uint32_t tag, float4& v, int op,
                                      uint32_t where) {
  uint64_t a, b, c, d;
  ld_tagged2(src, a, b);
  ld_tagged2(src + 2, c, d);
  if (tag_of(a) == tag && tag_of(b) == tag && tag_of(c) == tag && tag_of(d) == tag) {
    v = make_float4(value_of(a), value_of(b), value_of(c), value_of(d));
    return true;
  }
  float o[4];
  const bool ok = poll_slow(p, src, 4, tag, o, op, where);
  v = make_float4(o[0], o[1], o[2], o[3]);
  return ok;
}

__device__ __forceinline__ bool poll1(const KParams& p, const uint64_t* src, uint32_t tag, float& v, int op,
                                      uint32_t where) {
  const uint64_t a = ld_tagged(src);
  if (tag_of(a) == tag) {
    v = value_of(a);
    return true;
  }
  return poll_slow(p, src, 1, tag, &v, op, where);
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
__device__ __forceinline__ void split_range(int S, int ns, int j, int& head, int& s, int& p0, int& p1) {
  head = j / ns;
  s = j % ns;
  p0 = (int)((long long)S * s / ns);
  p1 = (int)((long long)S * (s + 1) / ns);
}

// Warps serving token m of an M-token window: m, m + M, ...; this warp is number gi of ng.
__device__ __forceinline__ void token_group(int w, int M, int& m, int& gi, int& ng) {
  m = w % M;
  gi = w / M;
  ng = (kConsumerWarps - m + M - 1) / M;
}

__device__ __forceinline__ int bytes_per_col(int wtype) { return wtype == W_BF16 ? 2 : 1; }  // MXFP4: K/2 below

__device__ __forceinline__ int row_bytes(int wtype, int K) {
  return wtype == W_BF16 ? 2 * K : (wtype == W_FP8 ? K : K / 2);
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
                 // [kw0, kw1))
  int N, K, R, Kc;
  int aw, bw, s0, s1;
  int r, kc, sl;
  int kw0, kw1;
  const int* experts;  // expert id per slot (routed ops); null: expert id = mat_base + slot
  int mat_base;

  __device__ void init(const OpDesc& op, int C, int cta, int w, int n_slots, const int* expert_ids, int base) {
    mat_base = base;
    N = op.N;
    K = op.K;
    R = op.R;
    Kc = op.Kc;
    experts = expert_ids;
    mode = (op.type == OP_SHARED_GATEUP || op.type == OP_ROUTED_GATEUP) ? 1 : (op.type == OP_EXP_DOWN ? 2 : 0);
    if (op.csplit) mode = 3;
    s0 = 0;
    s1 = 1;
    if (mode == 1) {
      s0 = op.slot0;
      s1 = op.type == OP_SHARED_GATEUP ? op.slot1 : n_slots;
    } else if (mode == 2) {
      s1 = n_slots;
    }
    int a, b;
    cta_rows(mode == 1 ? (s1 - s0) * N : N, op.unit, C, cta, a, b);
    if (mode == 3) {
      aw = a;
      bw = b;
      kw0 = min(K, w * Kc);
      kw1 = w == kConsumerWarps - 1 ? K : min(K, kw0 + Kc);
    } else {
      warp_rows(a, b, op.unit, w, aw, bw);
      kw0 = kw1 = 0;
    }
    r = aw;
    kc = 0;
    sl = 0;
  }

  __device__ bool next(Tile& t) {
    if (mode == 3) {
      if (r >= bw || kw0 >= kw1) return false;
      t.mat = 0;
      t.sl = 0;
      t.r0 = r;
      t.nr = min(R, bw - r);
      t.kc = kw0;
      t.kn = kw1 - kw0;
      t.last_k = true;
      r += t.nr;
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
  int gi, ng;
  int j, q, qe, head;
  bool fresh;

  __device__ void init(const KParams& p, int cta, int w, int pos_, int M, int P_) {
    C = p.n_ctas;
    pos = pos_;
    S = pos + M;
    ns = p.ns_max;
    nsplit = p.n_kv * ns;
    P = P_;
    int m;
    token_group(w, M, m, gi, ng);
    j = cta;
    fresh = true;
  }

  __device__ void enter_split() {
    int s, p0, p1;
    split_range(S, ns, j, head, s, p0, p1);
    const int ce = max(p0, min(p1, pos));
    q = p0 + (int)((long long)(ce - p0) * gi / ng);
    qe = p0 + (int)((long long)(ce - p0) * (gi + 1) / ng);
    fresh = false;
  }

  // Next tile of the current split only (the consumer steps splits itself).
  __device__ bool next_in_split(Tile& t) {
    if (fresh) enter_split();
    if (q >= qe) return false;
    t.mat = head;
    t.sl = j;
    t.r0 = q;
    t.nr = min(P, qe - q);
    q += t.nr;
    return true;
  }

  __device__ bool next_split() {
    j += C;
    fresh = true;
    return j < nsplit;
  }

  // Producer: next tile across splits.
  __device__ bool next(Tile& t) {
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
struct LaneCursor {
  int oi, started;
  uint32_t n;  // tiles issued to this lane's warp
  GemvIter g;
  AttnIter a;
};

struct Producer {
  const KParams& p;
  Smem& s;
  int pos, M;

  // Expert ids of the current MoE layer's routing, once the consumers have published it.
  __device__ const int* routing(const OpDesc* op) {
    if (s.flags[kFlagRoute] != __ldg(&op->layer) + 1) return nullptr;
    __threadfence_block();
    return s.route->expert;
  }

  __device__ void copy_gemv(const OpDesc* op, const Tile& t, uint8_t* dst, uint32_t fb) {
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
      bulk_g2s(d, base + (size_t)t.r0 * rb, total, fb);
    } else {
      for (int i = 0; i < t.nr; ++i) bulk_g2s(d + i * cb, base + (size_t)(t.r0 + i) * rb + koff, (uint32_t)cb, fb);
    }
    if (sbytes) {
      const int K32 = K / 32;
      const char* sb = static_cast<const char*>(op->ws) + (size_t)t.mat * __ldg(&op->ws_mstride);
      const uint32_t d2 = d + ((total + 15u) & ~15u);
      if (t.kn == K) {
        bulk_g2s(d2, sb + (size_t)t.r0 * K32, sbytes, fb);
      } else {
        for (int i = 0; i < t.nr; ++i)
          bulk_g2s(d2 + i * (t.kn / 32), sb + (size_t)(t.r0 + i) * K32 + t.kc / 32, (uint32_t)(t.kn / 32), fb);
      }
    }
  }

  __device__ void copy_attn(const OpDesc* op, const Tile& t, uint8_t* dst, uint32_t fb) {
    const uint32_t bytes = (uint32_t)t.nr * 256u;
    const size_t off = ((size_t)t.mat * p.cap + t.r0) * kHeadDim;
    mbar_expect_tx(fb, 2u * bytes);
    const uint32_t d = smem_addr(dst);
    bulk_g2s(d, op->kc + off, bytes, fb);
    bulk_g2s(d + bytes, op->vc + off, bytes, fb);
  }

  // One attempt for this lane: returns true if the cursor moved (tile issued or op finished).
  __device__ bool step(LaneCursor& c, int w) {
    if (c.oi >= p.op_end) return false;
    const OpDesc* op = p.ops + c.oi;
    const int type = __ldg(&op->type);
    if (!c.started) {
      if (type == OP_ATTN) {
        c.a.init(p, blockIdx.x, w, pos, M, s.slot_bytes / 512);
      } else {
        const int* experts = nullptr;
        int n_slots = 0;
        if (type == OP_ROUTED_GATEUP || type == OP_EXP_DOWN) {
          experts = routing(op);
          if (!experts) return false;  // routing not computed yet
          n_slots = s.route->n_slots;
        }
        const OpDesc o = *op;
        c.g.init(o, p.n_ctas, blockIdx.x, w, n_slots, experts, type == OP_SHARED_GATEUP ? p.E : 0);
      }
      c.started = 1;
    }
    Tile t;
    AttnIter pa = c.a;
    GemvIter pg = c.g;
    const bool more = type == OP_ATTN ? pa.next(t) : pg.next(t);
    if (!more) {
      ++c.oi;
      c.started = 0;
      return true;
    }
    const uint32_t st = c.n % (uint32_t)kStages;
    const uint32_t parity = ((c.n / (uint32_t)kStages) & 1u) ^ 1u;
    if (!mbar_test_wait(smem_addr(&s.empty[w * kStages + st]), parity)) return false;
    const uint32_t fb = smem_addr(&s.full[w * kStages + st]);
    if (type == OP_ATTN) {
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
    return true;
  }

  __device__ void run(int lane) {
    if (lane >= kConsumerWarps) return;
    constexpr unsigned kMask = (1u << kConsumerWarps) - 1u;
    const int w = lane;
    LaneCursor c;
    c.oi = p.op_begin;
    c.started = 0;
    c.n = 0;
    uint64_t t_idle = 0;
    for (;;) {
      const bool moved = step(c, w);
      const bool done = c.oi >= p.op_end;
      if (__all_sync(kMask, done)) break;
      if (__any_sync(kMask, moved)) {
        t_idle = 0;
        continue;
      }
      // nothing could move: every live warp's slots are full or routing is pending; back off
      // so the spinning lanes leave the scheduler's issue slots to the consumers
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
//                            the merge products
//   mg    [warps][G][132]    per-warp (max, sum, -, -, output[128]) at the end of a split; reused
//                            for the splits' sums in the merge
//   kvn   bf16 [2][M][128]   this call's own keys / values (rotated, rounded)
//   cw    [M*G][ns]          merge weights
struct AttnScratch {
  float* q;
  float* sc;
  float* mg;
  uint16_t* kvn;
  float* cw;
};

__device__ __forceinline__ AttnScratch attn_scratch(const KParams& p, const Smem& s, int M, int P) {
  AttnScratch a;
  float* f = s.act;
  a.q = f;
  f += M * p.G * 128;
  {
    const int MG = M * p.G, ns = p.ns_max;
    const int prods = ((MG * 32 + ns - 1) / ns + 1) * ns * 4;  // merge products (float4) of one slice
    a.sc = f;
    f += max(kConsumerWarps * p.G * P, prods);
    f = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(f) + 15) & ~uintptr_t(15));
  }
  a.mg = f;
  f += kConsumerWarps * p.G * kPart;
  a.kvn = reinterpret_cast<uint16_t*>(f);
  f += 2 * kMmax * 128 / 2;
  a.cw = f;
  return a;
}

template <int G_>
struct AttnState {
  float mrun[G_], lrun[G_];
  float o[G_][4];  // this lane's dims 4*lane .. +3
};

// One tile of n rows (keys at kr, values at vr; 256 B per row) for the G_ heads of token m.
// vis_base < 0: all rows visible; else row j is this call's row vis_base + j, visible iff <= m.
template <int G_>
__device__ __forceinline__ void attn_warp_tile(AttnState<G_>& A, const float (&q)[G_][16], const uint8_t* kr,
                                               const uint8_t* vr, int n, int vis_base, int m, float* sc, int P,
                                               int lane) {
  const int grp = lane >> 3, sub = lane & 7;
  // scores: eight lanes per row, 16 dims each, four rows per step
  for (int j0 = 0; j0 < n; j0 += 4) {
    const int j = j0 + grp;
    float kf[16];
    if (j < n) {
      const uint4 k0 = *reinterpret_cast<const uint4*>(kr + (size_t)j * 256 + sub * 32);
      const uint4 k1 = *reinterpret_cast<const uint4*>(kr + (size_t)j * 256 + sub * 32 + 16);
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
        const bool vis = vis_base < 0 || vis_base + j <= m;
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
    const uint2 v = *reinterpret_cast<const uint2*>(vr + (size_t)j * 256 + lane * 8);
    const float2 v01 = make_float2(bf16_lo(v.x), bf16_hi(v.x));
    const float2 v23 = make_float2(bf16_lo(v.y), bf16_hi(v.y));
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
struct Consumer {
  const KParams& p;
  Smem& s;
  uint32_t epoch, tag;  // tag: the data tag of this step (epoch + 1; zeroed memory never matches)
  const StepState& st;
  int tid, warp, lane;
  uint32_t n_tiles;  // tiles consumed by this warp (ring position)

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

  // Arrive at ticket t (n arrivals per step); true in the last arrival (all consumers agree).
  __device__ bool ticket(int t, int n) {
    consumer_sync();
    if (tid == 0) {
      const uint32_t old = atom_add_acq_rel(&p.tickets[t], 1u);
      s.flags[kFlagTicket] = (old == (epoch + 1u) * (uint32_t)n - 1u) ? 1 : 0;
    }
    consumer_sync();
    return s.flags[kFlagTicket] != 0;
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
  __device__ __forceinline__ const uint16_t* x_bf16(const OpDesc& op, int m) const {
    return op.xsrc == X_EMBED ? static_cast<const uint16_t*>(op.x_src) + (size_t)st.tokens[m] * p.H
                              : static_cast<const uint16_t*>(st.hidden_in) + (size_t)m * p.H;
  }

  // Four consecutive elements 4*k4 .. +3 of token m's x (the op's residual / norm input).
  __device__ __forceinline__ bool load_x4(const OpDesc& op, int m, int k4, float4& v, int oi) {
    if (op.xsrc == X_F32) return poll4(p, p.hs + ((size_t)op.x_idx * p.Mmax + m) * p.H + 4 * k4, tag, v, oi, 7);
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(x_bf16(op, m)) + k4);
    v = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    return true;
  }

  __device__ __forceinline__ bool load_x1(const OpDesc& op, int m, int k, float& v, int oi) {
    if (op.xsrc == X_F32) return poll1(p, p.hs + ((size_t)op.x_idx * p.Mmax + m) * p.H + k, tag, v, oi, 8);
    v = __uint_as_float((uint32_t)__ldg(x_bf16(op, m) + k) << 16);
    return true;
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

  // act = RMSNorm(x_m) * gain (op.norm) or x_m, written in the quarter-plane layout of the op's
  // weight type; the sum of squares is reduced in a fixed order (lane partials, warp tree,
  // warps in order), identical in every CTA. Returns this thread's polling verdict.
  __device__ bool norm_prologue(const OpDesc& op, int M, const uint2 (&gpre)[kGainPre], int oi) {
    const int H = p.H, H4 = H / 4;
    const int cw = chunk_width(op.wtype), nvt = H / cw;
    bool ok = true;
    for (int m = 0; m < M; ++m) {
      float ss = 0.f;
      for (int i0 = tid; i0 < H4; i0 += 4 * kConsumerThreads) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * kConsumerThreads;
          x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (i < H4) ok &= load_x4(op, m, i, x[u], oi);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * kConsumerThreads;
          if (i < H4) *reinterpret_cast<float4*>(s.act + m * H + act_pos(4 * i, cw, nvt)) = x[u];
          ss = fmaf(x[u].x, x[u].x, ss);
          ss = fmaf(x[u].y, x[u].y, ss);
          ss = fmaf(x[u].z, x[u].z, ss);
          ss = fmaf(x[u].w, x[u].w, ss);
        }
      }
      if (op.norm) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s.red[warp] = ss;
        consumer_sync();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) tot += s.red[w];
        const float rstd = 1.0f / sqrtf(tot / (float)H + p.eps);
        auto scale = [&](int i, uint2 g) {
          float4* d = reinterpret_cast<float4*>(s.act + m * H + act_pos(4 * i, cw, nvt));
          float4 v = *d;
          v.x = v.x * rstd * bf16_lo(g.x);
          v.y = v.y * rstd * bf16_hi(g.x);
          v.z = v.z * rstd * bf16_lo(g.y);
          v.w = v.w * rstd * bf16_hi(g.y);
          *d = v;
        };
#pragma unroll
        for (int u = 0; u < kGainPre; ++u) {
          const int i = tid + u * kConsumerThreads;
          if (i < H4) scale(i, gpre[u]);
        }
        for (int i = tid + kGainPre * kConsumerThreads; i < H4; i += kConsumerThreads)
          scale(i, __ldg(reinterpret_cast<const uint2*>(op.gain) + i));
      }
      consumer_sync();
    }
    return ok;
  }

  // dst = M rows of K tagged words polled from global (row stride src_stride words), in the
  // quarter-plane layout of chunk width cw; four polls in flight per thread.
  __device__ bool copy_act(float* dst, const uint64_t* src, int M, int K, int src_stride, int cw, int oi) {
    const int K4 = K / 4, n4 = M * K4, nvt = K / cw;
    bool ok = true;
    for (int i0 = tid; i0 < n4; i0 += 4 * kConsumerThreads) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kConsumerThreads;
        x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n4) ok &= poll4(p, src + (size_t)(i / K4) * src_stride + 4 * (i % K4), tag, x[u], oi, 9);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kConsumerThreads;
        if (i < n4) *reinterpret_cast<float4*>(dst + (i / K4) * K + act_pos(4 * (i % K4), cw, nvt)) = x[u];
      }
    }
    return ok;
  }

  // xres[i][m] = x_m[a + i] for the CTA's rows [a, b): the residual input of the op.
  __device__ bool load_residual(const OpDesc& op, float* xres, int a, int b, int M, int oi) {
    bool ok = true;
    for (int t = tid; t < (b - a) * M; t += kConsumerThreads) {
      const int i = t / M, m = t % M;
      float v = 0.f;
      ok &= load_x1(op, m, a + i, v, oi);
      xres[t] = v;
    }
    return ok;
  }

  // ---------------------------------------------------------------- routing (MoE layers)
  // Every CTA computes the layer's routing itself from the router logits (op.act) it polls:
  // top-k per token (largest first, lower index on ties), softmax over the selected logits,
  // and the union of the window's experts (shared experts first). The producer lanes read it
  // from shared memory once flags[kFlagRoute] names the layer. Uses the start of s.act.
  __device__ __noinline__ bool ensure_routing(const OpDesc& op, int M, int oi) {
    if (s.flags[kFlagRoute] == op.layer + 1) return true;
    const int E = p.E, k = p.top_k;
    float* r = s.act;  // [M][E]
    bool ok = true;
    for (int i = tid; i < M * E; i += kConsumerThreads) {
      float v = 0.f;
      ok &= poll1(p, op.act + i, tag, v, oi, 10);
      r[i] = v;
    }
    if (!consumer_all(ok)) return false;
    RouteBlock* rb = s.route;
    for (int m = 0; m < M; ++m) {
      for (int kk = 0; kk < k; ++kk) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
        for (int e = tid; e < E; e += kConsumerThreads) {
          const float v = r[m * E + e];
          if (v > bv || (v == bv && e < bi)) {
            bv = v;
            bi = e;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oj = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oj < bi)) {
            bv = ov;
            bi = oj;
          }
        }
        if (lane == 0) {
          s.red[warp] = bv;
          s.resw[warp] = __int_as_float(bi);
        }
        consumer_sync();
        if (tid == 0) {
          float v = s.red[0];
          int i = __float_as_int(s.resw[0]);
          for (int w = 1; w < kConsumerWarps; ++w) {
            const int wi = __float_as_int(s.resw[w]);
            if (s.red[w] > v || (s.red[w] == v && wi < i)) {
              v = s.red[w];
              i = wi;
            }
          }
          rb->topk[m][kk] = i;
          rb->topk_w[m][kk] = v;  // the logit, replaced by its weight below
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
      __threadfence_block();
      s.flags[kFlagRoute] = op.layer + 1;  // the producer lanes may now read the expert ids
    }
    consumer_sync();
    if (blockIdx.x == 0) {  // a copy in global memory for inspection
      const int* src = reinterpret_cast<const int*>(rb);
      for (int i = tid; i < (int)(sizeof(RouteBlock) / 4); i += kConsumerThreads) op.route[i] = src[i];
    }
    return true;
  }

  // ---------------------------------------------------------------- matrix ops
  // This warp's tiles of a matrix op. Results of a row group land in lane j*MT + m (row j,
  // token m); tokens m >= M (MT = 4 serving a 2- or 3-token window) are computed on zero
  // activations and dropped.
  template <int WT, int MT, int NR>
  __device__ __noinline__ bool gemv_op_t(int oi, const OpDesc& op, int M, float* xres, int a, float* accd) {
    GemvIter it;
    const bool routed = op.type == OP_ROUTED_GATEUP || op.type == OP_EXP_DOWN;
    const int n_slots = routed ? s.route->n_slots : 0;
    it.init(op, p.n_ctas, blockIdx.x, warp, n_slots, routed ? s.route->expert : nullptr,
            op.type == OP_SHARED_GATEUP ? p.E : 0);
    Acc<NR, MT> A;
    acc_zero(A);
    float best_v = -INFINITY;
    int best_i = 0x7FFFFFFF;
    Tile t;
    bool ok = true;
    const int i = lane / MT, m = lane % MT;
    // one token, whole rows, activations that fit: keep them in registers for the whole op
    constexpr int NI = RegCfg<WT>::NI;
    const bool regs = MT == 1 && op.type != OP_EXP_DOWN && op.Kc == op.K && op.K <= 32 * NI * WCfg<WT>::CW;
    ActRegs<WT, (MT == 1 ? NI : 1)> AR;
    if constexpr (MT == 1)
      if (regs) act_regs_load(AR, s.act, op.K, 0, op.K, lane);
    while (it.next(t)) {
      uint8_t* slot;
      uint32_t eb;
      if (!next_slot(oi, slot, eb)) {
        ok = false;
        break;
      }
      const float* actp = (op.type == OP_EXP_DOWN && op.stage_all) ? s.act + (size_t)t.sl * M * op.K : s.act;
      if constexpr (MT == 1) {
        if (regs)
          warp_gemv_reg<WT, NR, NI>(slot, t.nr, t.kn, AR, A, lane);
        else
          warp_gemv<WT, MT, NR>(slot, t.nr, t.kn, t.kc, actp, op.K, M, A, lane);
      } else {
        warp_gemv<WT, MT, NR>(slot, t.nr, t.kn, t.kc, actp, op.K, M, A, lane);
      }
      release(eb);
      if (!t.last_k) continue;
      const float v = warp_rowsums<NR, MT>(A, t.nr, lane);
      acc_zero(A);
      const bool mine = lane < t.nr * MT && m < M;
      switch (op.type) {
        case OP_QKV:
        case OP_ROUTER:
          if (mine) st_tagged(op.out + (size_t)m * op.N + t.r0 + i, v, tag);
          break;
        case OP_OPROJ:
        case OP_DOWN:
          if (mine) st_tagged(op.x_out + (size_t)m * p.H + t.r0 + i, xres[(t.r0 + i - a) * M + m] + v, tag);
          break;
        case OP_GATEUP:
        case OP_SHARED_GATEUP:
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
  // activations in registers (one token) and leaves a partial sum per row; the warps' partials
  // are added in warp order afterwards (csplit_epilogue).
  template <int WT, int MT, int NR>
  __device__ __noinline__ bool gemv_csplit_t(int oi, const OpDesc& op, int M, int a, float* parts) {
    GemvIter it;
    it.init(op, p.n_ctas, blockIdx.x, warp, 0, nullptr, 0);
    Acc<NR, MT> A;
    constexpr int NI = RegCfg<WT>::NI;
    ActRegs<WT, (MT == 1 ? NI : 1)> AR;
    if constexpr (MT == 1)
      if (it.kw0 < it.kw1) act_regs_load(AR, s.act, op.K, it.kw0, it.kw1 - it.kw0, lane);
    const int rows = it.bw - it.aw;
    Tile t;
    while (it.next(t)) {
      uint8_t* slot;
      uint32_t eb;
      if (!next_slot(oi, slot, eb)) return false;
      acc_zero(A);
      if constexpr (MT == 1)
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
      return v;
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
      if (op.type == OP_OPROJ || op.type == OP_DOWN)
        st_tagged(op.x_out + (size_t)m * p.H + a + r, xres[t] + v, tag);
      else
        st_tagged(op.out + (size_t)m * op.N + a + r, v, tag);
    }
  }

  // Tile rows per warp-tile template: bf16 2/4/8, FP8 4/8, MXFP4 8 (the host's R fits).
  template <int MT>
  __device__ bool gemv_dispatch(int oi, const OpDesc& op, int M, float* xres, int a, float* accd) {
    if (op.csplit) {
      if (op.wtype == W_BF16) return gemv_csplit_t<W_BF16, MT, 8>(oi, op, M, a, accd);
      return gemv_csplit_t<W_FP8, MT, 8>(oi, op, M, a, accd);
    }
    if (op.wtype == W_BF16) {
      if (op.R <= 2) return gemv_op_t<W_BF16, MT, 2>(oi, op, M, xres, a, accd);
      if (op.R <= 4) return gemv_op_t<W_BF16, MT, 4>(oi, op, M, xres, a, accd);
      return gemv_op_t<W_BF16, MT, 8>(oi, op, M, xres, a, accd);
    }
    if (op.wtype == W_FP8) {
      if (op.R <= 4) return gemv_op_t<W_FP8, MT, 4>(oi, op, M, xres, a, accd);
      return gemv_op_t<W_FP8, MT, 8>(oi, op, M, xres, a, accd);
    }
    return gemv_op_t<W_MXFP4, MT, 8>(oi, op, M, xres, a, accd);
  }

  // Expert down, one slot (its hidden vectors staged in act by the caller).
  template <int MT>
  __device__ __noinline__ bool gemv_slot(int oi, const OpDesc& op, int sl, int M, int a, float* accd) {
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

  __device__ bool gemv_op(int oi, const OpDesc& op, int M, const uint2 (&gpre)[kGainPre]) {
    const int C = p.n_ctas, cta = blockIdx.x;
    const int cw = chunk_width(op.wtype);
    int a = 0, b = 0;
    float* xres = nullptr;
    float* accd = nullptr;
    bool ok = true;
    // prologue: poll the activations every tile multiplies, and the residual rows of this CTA
    switch (op.type) {
      case OP_OPROJ:
      case OP_DOWN:
        cta_rows(op.N, op.unit, C, cta, a, b);
        ok &= copy_act(s.act, op.act, M, op.K, op.K, cw, oi);
        xres = s.act + M * op.K;
        ok &= load_residual(op, xres, a, b, M, oi);
        if (op.csplit) accd = xres + (b - a) * M;  // per-warp partial sums
        break;
      case OP_EXP_DOWN: {
        if (!ensure_routing(op, M, oi)) return false;
        cta_rows(op.N, op.unit, C, cta, a, b);
        const int n_slots = s.route->n_slots;
        const int hfl = op.stage_all ? n_slots * M * op.K : M * op.K;
        xres = s.act + hfl;
        accd = xres + (b - a) * M;
        ok &= load_residual(op, xres, a, b, M, oi);
        for (int t = tid; t < (b - a) * M; t += kConsumerThreads) accd[t] = 0.f;
        if (op.stage_all)
          for (int sl = 0; sl < n_slots; ++sl)
            ok &= copy_act(s.act + (size_t)sl * M * op.K, op.eh + (size_t)sl * p.Mmax * op.K, M, op.K, op.K, cw, oi);
        break;
      }
      case OP_ROUTED_GATEUP:
        if (!ensure_routing(op, M, oi)) return false;
        ok &= norm_prologue(op, M, gpre, oi);
        break;
      default:
        ok &= norm_prologue(op, M, gpre, oi);
        if (op.csplit) {
          cta_rows(op.N, op.unit, C, cta, a, b);
          accd = s.act + M * op.K;  // per-warp partial sums
        }
        break;
    }
    if (!consumer_all(ok)) return false;
    if (tid == 0) {
      TRACE(p, oi, 1, gtimer());
      TRACE(p, oi, 2, gtimer());
    }
    if (op.type == OP_EXP_DOWN && !op.stage_all) {
      // one slot at a time: stage its hidden vectors, then every warp runs its rows of it
      const int n_slots = s.route->n_slots;
      for (int sl = 0; sl < n_slots; ++sl) {
        ok = copy_act(s.act, op.eh + (size_t)sl * p.Mmax * op.K, M, op.K, op.K, cw, oi);
        if (!consumer_all(ok)) return false;
        const bool r = M == 1 ? gemv_slot<1>(oi, op, sl, M, a, accd) : gemv_slot<4>(oi, op, sl, M, a, accd);
        if (!consumer_all(r)) return false;
      }
    } else {
      const bool r = M == 1 ? gemv_dispatch<1>(oi, op, M, xres, a, accd) : gemv_dispatch<4>(oi, op, M, xres, a, accd);
      if (!consumer_all(r)) return false;
    }
    if (tid == 0) TRACE(p, oi, 3, gtimer());
    if (op.csplit) csplit_epilogue(op, M, a, b, xres, accd);
    if (op.type == OP_EXP_DOWN) {
      for (int t = tid; t < (b - a) * M; t += kConsumerThreads) {
        const int i = t / M, m = t % M;
        st_tagged(op.x_out + (size_t)m * p.H + a + i, xres[t] + accd[t], tag);
      }
    }
    if (op.type == OP_ROUTER) {
      consumer_sync();  // s.act is reused for the logits
      return ensure_routing(op, M, oi);
    }
    if (op.type == OP_LMHEAD) lmhead_finish(op, M);
    return true;
  }

  // Per-warp bests -> per-CTA partial -> the last CTA reduces all partials (lowest index on ties).
  __device__ __noinline__ void lmhead_finish(const OpDesc& op, int M) {
    consumer_sync();
    const int MT = M == 1 ? 1 : 4;  // lane l of a warp tracked token l % MT
    if (tid < M) {
      float v = -INFINITY;
      int i = 0x7FFFFFFF;
      for (int w = 0; w < kConsumerWarps; ++w)
        for (int l = tid; l < 32; l += MT) {
          const float wv = s.resw[w * 64 + l];
          const int wi = reinterpret_cast<const int*>(s.resw)[w * 64 + 32 + l];
          if (wv > v || (wv == v && wi < i)) {
            v = wv;
            i = wi;
          }
        }
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
          if (cv > v || (cv == v && ci < i)) {
            v = cv;
            i = ci;
          }
        }
        p.am_out[tid] = i;
      }
    }
  }

  // ---------------------------------------------------------------- attention op
  template <int G_>
  __device__ __noinline__ bool attn_op(int oi, const OpDesc& op, int pos, int M) {
    const int P = s.slot_bytes / 512;
    const int G = G_, MG = M * G, ns = p.ns_max;
    const AttnScratch a = attn_scratch(p, s, M, P);
    const float qscale = 1.4426950408889634f / sqrtf(128.f);  // log2(e) / sqrt(d)
    int m_tok, gi, ng;
    token_group(warp, M, m_tok, gi, ng);
    AttnIter it;
    it.init(p, blockIdx.x, warp, pos, M, P);
    float* sc = a.sc + warp * G * P;
    const uint64_t* qkv = op.act;
    const size_t sstride = (size_t)p.Mmax * G * kPart;  // words per split partial
    uint64_t* lpart = p.part + (size_t)op.layer * p.n_kv * ns * sstride;
    for (; it.j < it.nsplit; it.next_split()) {
      int head, sidx, p0, p1;
      split_range(it.S, ns, it.j, head, sidx, p0, p1);
      // CTA prologue: rotated, scaled queries of the group; this call's own keys/values
      bool ok = true;
      for (int idx = tid; idx < MG * 64; idx += kConsumerThreads) {
        const int mh = idx >> 6, i = idx & 63;
        const int m = mh / G, h = head * G + mh % G;
        const uint64_t* qr = qkv + (size_t)m * p.qkv_rows + h * 128;
        float x1 = 0.f, x2 = 0.f;
        ok &= poll1(p, qr + i, tag, x1, oi, 11);
        ok &= poll1(p, qr + i + 64, tag, x2, oi, 11);
        const float2 cs = s.rope[m * 64 + i];
        a.q[mh * 128 + i] = (x1 * cs.x - x2 * cs.y) * qscale;
        a.q[mh * 128 + i + 64] = (x1 * cs.y + x2 * cs.x) * qscale;
      }
      const int nb = max(p0, pos), nn = max(0, p1 - nb);
      for (int idx = tid; idx < nn * 64; idx += kConsumerThreads) {
        const int r = idx >> 6, i = idx & 63;
        const int m = nb - pos + r;
        const uint64_t* kr = qkv + (size_t)m * p.qkv_rows + (p.n_q + head) * 128;
        const uint64_t* vr = qkv + (size_t)m * p.qkv_rows + (p.n_q + p.n_kv + head) * 128;
        float k1 = 0.f, k2 = 0.f, v1 = 0.f, v2 = 0.f;
        ok &= poll1(p, kr + i, tag, k1, oi, 12);
        ok &= poll1(p, kr + i + 64, tag, k2, oi, 12);
        ok &= poll1(p, vr + i, tag, v1, oi, 12);
        ok &= poll1(p, vr + i + 64, tag, v2, oi, 12);
        const float2 cs = s.rope[m * 64 + i];
        const uint16_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(k1 * cs.x - k2 * cs.y));
        const uint16_t b2 = __bfloat16_as_ushort(__float2bfloat16_rn(k1 * cs.y + k2 * cs.x));
        const uint16_t c1 = __bfloat16_as_ushort(__float2bfloat16_rn(v1));
        const uint16_t c2 = __bfloat16_as_ushort(__float2bfloat16_rn(v2));
        a.kvn[r * 128 + i] = b1;
        a.kvn[r * 128 + i + 64] = b2;
        a.kvn[(nn + r) * 128 + i] = c1;
        a.kvn[(nn + r) * 128 + i + 64] = c2;
        const size_t off = ((size_t)head * p.cap + pos + m) * kHeadDim;  // append to the KV history
        op.kc[off + i] = b1;
        op.kc[off + i + 64] = b2;
        op.vc[off + i] = c1;
        op.vc[off + i + 64] = c2;
      }
      if (!consumer_all(ok)) return false;
      if (tid == 0 && it.j == (int)blockIdx.x) {
        TRACE(p, oi, 1, gtimer());
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
#pragma unroll
      for (int h = 0; h < G_; ++h)
#pragma unroll
        for (int e = 0; e < 16; ++e) q[h][e] = a.q[(m_tok * G + h) * 128 + sub * 16 + e];
      Tile t;
      while (it.next_in_split(t)) {
        uint8_t* slot;
        uint32_t eb;
        if (!next_slot(oi, slot, eb)) {
          ok = false;
          break;
        }
        attn_warp_tile<G_>(A, q, slot, slot + t.nr * 256, t.nr, -1, m_tok, sc, P, lane);
        release(eb);
      }
      // this call's own rows: the first warp of each token group attends to them (causally)
      if (ok && gi == 0 && nn > 0) {
        const uint8_t* kn = reinterpret_cast<const uint8_t*>(a.kvn);
        attn_warp_tile<G_>(A, q, kn, kn + nn * 256, nn, nb - pos, m_tok, sc, P, lane);
      }
      // per-warp state -> shared memory; merge the warps of each token into the split partial
      float* mg = a.mg + warp * G * kPart;
#pragma unroll
      for (int h = 0; h < G_; ++h) {
        if (lane == 0) {
          mg[h * kPart] = A.mrun[h];
          mg[h * kPart + 1] = A.lrun[h];
        }
        *reinterpret_cast<float4*>(mg + h * kPart + 4 + lane * 4) =
            make_float4(A.o[h][0], A.o[h][1], A.o[h][2], A.o[h][3]);
      }
      if (!consumer_all(ok)) return false;
      if (tid == 0) TRACE(p, oi, 3, gtimer());
      uint64_t* part = lpart + (size_t)(head * ns + sidx) * sstride;
      for (int idx = tid; idx < MG * kPart; idx += kConsumerThreads) {
        const int mh = idx / kPart, e = idx % kPart;
        if (e == 2 || e == 3) continue;
        const int m = mh / G, h = mh % G;
        float mx = -INFINITY;
        for (int w = m; w < kConsumerWarps; w += M) mx = fmaxf(mx, a.mg[(w * G + h) * kPart]);
        float l = 0.f, o = 0.f;
        for (int w = m; w < kConsumerWarps; w += M) {
          const float mw = a.mg[(w * G + h) * kPart];
          const float f = mw == -INFINITY ? 0.f : exp2f(mw - mx);
          l += f * a.mg[(w * G + h) * kPart + 1];
          if (e >= 4) o += f * a.mg[(w * G + h) * kPart + e];
        }
        st_tagged(part + mh * kPart + e, e == 0 ? mx : (e == 1 ? l : o), tag);
      }
      consumer_sync();
    }
    // Phase 2: the splits of a kv head merge its outputs together, each split a 1/ns slice
    // (log-sum-exp in base 2), polling the head's tagged partials. Every split of this CTA was
    // published above before any of these polls, so no CTA waits on one that waits on it.
    AttnIter it2;
    it2.init(p, blockIdx.x, warp, pos, M, P);
    for (; it2.j < it2.nsplit; it2.next_split()) {
      int head, sidx, p0, p1;
      split_range(it2.S, ns, it2.j, head, sidx, p0, p1);
      const uint64_t* hp = lpart + (size_t)(head * ns) * sstride;
      const int total = MG * 32;  // float4 outputs of this kv head
      const int o0 = (int)((long long)total * sidx / ns), o1 = (int)((long long)total * (sidx + 1) / ns);
      if (o0 >= o1) continue;
      const int mhA = o0 >> 5, mhB = (o1 - 1) >> 5;
      bool ok = true;
      // weights of every split for the (m, h) rows of this slice (sums parked in mg)
      for (int mh = mhA + warp; mh <= mhB; mh += kConsumerWarps) {
        float* cw = a.cw + (mh - mhA) * ns;
        float* lw = a.mg + (mh - mhA) * ns;
        float mx = -INFINITY;
        for (int q2 = lane; q2 < ns; q2 += 32) {
          float mq = 0.f, lq = 0.f;
          ok &= poll1(p, hp + q2 * sstride + mh * kPart, tag, mq, oi, 13);
          ok &= poll1(p, hp + q2 * sstride + mh * kPart + 1, tag, lq, oi, 13);
          cw[q2] = mq;
          lw[q2] = lq;
          mx = fmaxf(mx, mq);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float l = 0.f;
        for (int q2 = lane; q2 < ns; q2 += 32) {
          const float mq = cw[q2];
          const float w = mq == -INFINITY ? 0.f : exp2f(mq - mx);
          cw[q2] = w;
          l += w * lw[q2];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        const float inv = 1.0f / l;
        for (int q2 = lane; q2 < ns; q2 += 32) cw[q2] *= inv;
      }
      if (!consumer_all(ok)) return false;
      // one (output, split) product per thread, then a fixed-order sum over the splits
      float4* prod = reinterpret_cast<float4*>(a.sc);
      const int n = (o1 - o0) * ns;
      for (int t = tid; t < n; t += kConsumerThreads) {
        const int oo = o0 + t / ns, q2 = t % ns;
        const int mh = oo >> 5, d4 = oo & 31;
        const float w = a.cw[(mh - mhA) * ns + q2];
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        ok &= poll4(p, hp + q2 * sstride + mh * kPart + 4 + 4 * d4, tag, v, oi, 14);
        prod[t] = make_float4(w * v.x, w * v.y, w * v.z, w * v.w);
      }
      if (!consumer_all(ok)) return false;
      for (int t = tid; t < o1 - o0; t += kConsumerThreads) {
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q2 = 0; q2 < ns; ++q2) {
          const float4 v = prod[t * ns + q2];
          o.x += v.x;
          o.y += v.y;
          o.z += v.z;
          o.w += v.w;
        }
        const int oo = o0 + t, mh = oo >> 5, d4 = oo & 31;
        const int m = mh / G, h = head * G + mh % G;
        st_tagged4(op.out + (size_t)m * p.n_q * 128 + h * 128 + d4 * 4, o, tag);
      }
      consumer_sync();
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
      if (tid == 0) TRACE(p, oi, 0, gtimer());
      uint2 gpre[kGainPre];
      load_gain(op, gpre);
      bool ok;
      if (op.type == OP_ATTN) {
        switch (p.G) {
          case 1: ok = attn_op<1>(oi, op, pos, M); break;
          case 2: ok = attn_op<2>(oi, op, pos, M); break;
          case 4: ok = attn_op<4>(oi, op, pos, M); break;
          case 5: ok = attn_op<5>(oi, op, pos, M); break;
          default: ok = attn_op<8>(oi, op, pos, M); break;
        }
      } else {
        ok = gemv_op(oi, op, M, gpre);
      }
      if (!ok) return false;
      consumer_sync();
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

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(kThreads, 1) dec_megakernel(const KParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem s = carve(smem_raw, p);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ StepState st;
  if (tid == 0) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.state);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&st);
    for (int i = 0; i < (int)(sizeof(StepState) / 4); ++i) dst[i] = __ldcg(src + i);
    for (int i = 0; i < kConsumerWarps * kStages; ++i) {
      mbar_init(smem_addr(&s.full[i]), 1);
      mbar_init(smem_addr(&s.empty[i]), 1);
    }
    s.flags[kFlagRoute] = -1;
    mbar_init_fence();
  }
  __syncthreads();
  const uint32_t epoch = st.epoch;
  const int pos = st.pos, M = st.m;
  if (warp == kConsumerWarps) {
    Producer pr{p, s, pos, M};
    pr.run(lane);
    return;
  }
  // RoPE table of this call's positions (fp64 angle, then fp32 cos/sin).
  for (int t = tid; t < M * 64; t += kConsumerThreads) {
    const int m = t >> 6, i = t & 63;
    const double inv = pow((double)p.rope_base, -2.0 * (double)i / 128.0);
    double sn, cs;
    sincos((double)(pos + m) * inv, &sn, &cs);
    s.rope[t] = make_float2((float)cs, (float)sn);
  }
  consumer_sync();
  Consumer c{p, s, epoch, epoch + 1u, st, tid, warp, lane, 0u};
  c.run(pos, M);
}

}  // namespace decimpl

// ------------------------------------------------------------------ host launch
extern "C" cudaError_t dec_launch_megakernel(const decimpl::KParams* kp, int cooperative, cudaStream_t stream) {
  using namespace decimpl;
  const size_t smem = (size_t)kConsumerWarps * kStages * kp->slot_bytes + kp->act_bytes + kCommonBytes;
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

// Common area plus the kernel's static shared memory, which the dynamic part must leave room for.
extern "C" int dec_megakernel_common_bytes(void) { return decimpl::kCommonBytes + 2048; }
