// Internal layout shared by the host runtime (api.cpp) and the megakernel (megakernel.cu).
//
// A decode step is a fixed list of ops (OpDesc). Every CTA of the persistent grid walks
// the whole list; for each op it takes its own share of the op's rows (or attention
// positions) and splits it among its consumer warps, in tiles that fit one ring slot. The
// producer warp streams every consumer warp's tiles of weights / KV history into that
// warp's slots with bulk asynchronous copies. Weights and cached KV never depend on the
// running step, so the producer runs ahead across op boundaries: the next op's weights are
// already in flight while the previous op is still being finished elsewhere (the
// multiprogramming argument of the Muse Spark Open megakernel article, section "the
// baseline nobody benchmarked", and its weight-prefetch ring, section "three bills").
// Activations travel as tagged words (value + step tag): a consumer reads the words it needs
// and re-reads any whose tag is not the current step's yet, so a writer never executes a fence
// (a fence would wait for the CTA's bulk copies in flight). Per-op arrival counters (relaxed
// atomics) remain as a build option that gates the reads on a count instead.
#pragma once
#include <cuda.h>  // CUtensorMap (a type only: the library does not link the driver API)
#include <cuda_runtime.h>
#include <stdint.h>

namespace decimpl {

// 7 consumer warps + 1 producer warp: two warps per scheduler, so a thread may hold up to 255
// registers (a ninth warp would put three on one scheduler and cap every thread at 168).
constexpr int kConsumerWarps = 7;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp (lane w serves consumer warp w)
#ifndef DEC_STAGES
#define DEC_STAGES 2
#endif
constexpr int kStages = DEC_STAGES;              // ring slots per consumer warp
constexpr int kRmax = 8;                         // rows one warp accumulates per tile
constexpr int kMmax = 4;                         // tokens per call (verify window)
constexpr int kHeadDim = 128;
constexpr int kMaxRouteSlots = 1 + 8 * kMmax;    // shared + union of routed experts
// Expert prefetch record of one MoE layer (int32 words): routed experts the layer's last routing
// shared with the one before it, slots of the last routing, then its expert ids (shared first).
constexpr int kXpfWords = 2 + kMaxRouteSlots + 1;  // padded to a multiple of 4 words
constexpr int kPart = 132;                       // attention partial: max, sum, 2 pad, output[128]
constexpr int kMaxSlotBytes = 16384;             // one warp's ring slot at most (attention rows <= 32)
constexpr int kSmemLimit = 232448;               // dynamic shared memory per CTA on sm_103a
constexpr int kNoAllocScratchBytes = 64 * 1024;  // static scratch of the allocation-free LM head
constexpr int kAttnTcRows = 16;                  // KV rows of one tensor-core attention tile
constexpr int kGemvTcRows = 16;                  // weight rows of one tensor-core GEMV tile
constexpr int kAttnTcBoxBytes = kAttnTcRows * 128;  // one 64-column box of a tile (swizzle span 128 B)

enum OpType : int32_t {
  OP_QKV = 0,           // a = RMSNorm(x); qkv = W_qkv a
  OP_ATTN = 1,          // split-K GQA attention (+ RoPE, KV append, log-sum-exp combine)
  OP_OPROJ = 2,         // x' = x + W_o o
  OP_GATEUP = 3,        // b = RMSNorm(x'); h = silu(W_g b) * (W_u b)   (pair-interleaved rows)
  OP_DOWN = 4,          // x'' = x' + W_d h
  OP_ROUTER = 5,        // b = RMSNorm(x'); r = W_r b (fp32); top-k + softmax (every CTA, locally)
  OP_ROUTED_GATEUP = 7, // h_e = SwiGLU gate/up of every slot: shared experts, then routed (MXFP4)
  OP_EXP_DOWN = 8,      // x'' = x' + sum_slots w * W_d,e h_e
  OP_LMHEAD = 9,        // logits = W_lm RMSNorm(x); argmax (block, then last CTA)
};

enum WType : int32_t { W_BF16 = 0, W_FP8 = 1, W_MXFP4 = 2 };
enum XSrc : int32_t { X_NONE = 0, X_F32 = 1, X_HIDDEN_IN = 2, X_EMBED = 3 };

struct OpDesc {
  int32_t type, wtype, layer, N;      // N: rows of one matrix (per expert for expert ops)
  int32_t K, R, Kc, pair;             // cols, rows per tile, columns per tile, gate/up pair rows
  int32_t ticket, ctr;                // ticket index (LM head argmax); this op's arrival counter
  int32_t wait_ctr, wait_n;           // counter of the op producing this op's input, arrivals / step
  int32_t aux_ctr, tc;                // attention: first per-kv-head counter; routed ops: router's;
                                      // tc: tensor-core tiles (multi-token lists: 16-row boxes by TMA)
  int32_t norm, xsrc;                 // input = RMSNorm(x) * gain; source of x
  int32_t slot0, slot1;               // expert slots [slot0, slot1) (slot1 < 0: up to n_slots)
  int32_t x_idx, unit;                // hidden-stream entry of x (X_F32); row granularity of the CTA split
  int32_t stage_all, csplit;          // expert down: all hidden vectors staged; column split across warps
                                      // (expert down: slot split, chunks of R rows per warp item)
  const void* w;                      // packed values (expert ops: expert 0)
  const void* ws;                     // scales plane (FP8 row scales / MXFP4 E8M0), else null
  int64_t w_mstride, ws_mstride;      // bytes between experts
  const uint16_t* gain;               // RMSNorm gain, bf16 [H]
  const void* x_src;                  // X_EMBED: embedding table bf16 [V][H]
  uint64_t* x_out;                    // residual output, tagged [Mmax][H]
  const uint64_t* act;                // plain input, tagged [Mmax][K] (o-proj: attention out; down: h;
                                      // attention: this layer's qkv)
  uint64_t* out;                      // output, tagged: qkv [Mmax][qkv], h [Mmax][F], router logits,
                                      // attention out [Mmax][n_q 128]
  float* logits;                      // LM head: fp32 logits [Mmax][V] (plain, for the caller)
  uint8_t* kc;                        // this layer's key cache   [n_kv][cap][128] bf16 or e4m3
  uint8_t* vc;                        // this layer's value cache [n_kv][cap][128] bf16 or e4m3
  const float* kv_scale;              // FP8 cache: this layer's scales [2][n_kv] (null: all 1)
  int32_t* route;                     // this layer's RouteBlock
  uint64_t* eh;                       // this layer's expert hidden, tagged [slots][Mmax][I]
  uint16_t* y_bf16;                   // residual ops: also store the output rounded to bf16 here,
                                      // [Mmax][H] (a layer run on its own hands its result back)
  int32_t* topk_idx_out;              // router: also store each token's top-k experts, [m][top_k]
  float* topk_w_out;                  // router: and their routing weights, [m][top_k]
  const CUtensorMap* tmap;            // tc ops: the weight matrix as a 2D tensor (K columns x N rows),
                                      // boxes of 64 columns x kGemvTcRows rows, 128-byte swizzle
  int32_t kw, pad1;                   // column split: columns per warp (0: Kc, in one tile)
  int32_t* xpf;                       // MoE ops: this layer's expert prefetch record (kXpfWords)
};

struct RouteBlock {
  int32_t n_slots;                    // n_shared + distinct routed experts
  int32_t expert[kMaxRouteSlots];     // expert id per slot (shared experts first: id >= E)
  float w[kMmax][kMaxRouteSlots];     // weight of slot for token m (1 for shared, pi or 0)
  int32_t topk[kMmax][8];             // per-token selection, best first
  float topk_w[kMmax][8];
};

struct StepState {
  uint32_t epoch;                     // completed steps; counters reach (epoch+1)*n during a step;
                                      // activation tags are epoch + 1
  int32_t pos;                        // position of the first token of this call
  int32_t m;                          // tokens in this call (1..kMmax)
  int32_t chain;                      // 1: at step end feed argmax back as the next token, pos += 1
  int32_t tokens[kMmax];
  const void* hidden_in;              // bf16 [m][H] when the step starts from a given hidden
  int32_t* gen_out;                   // chained generation: token i goes to gen_out[gen_idx++]
  int32_t gen_idx;
  int32_t pad[5];
};

struct Status {
  uint32_t abort;                     // set by the first failing CTA; every wait polls it
  uint32_t code;                      // dec_status of the failure
  int32_t op, cta;
  uint32_t counter, observed, target, where;
};

struct KParams {
  const OpDesc* ops;
  int32_t op_begin, op_end, n_ops, n_ctas;
  int32_t H, n_q, n_kv, G, qkv_rows, E, top_k, I, n_shared, V, cap, Mmax, L, ns_max;
  float eps, rope_base;
  uint64_t timeout_ns;
  int32_t slot_bytes, act_bytes;      // bytes of one warp's ring slot; shared-memory scratch
  int32_t kv_fp8;                     // 1: the KV cache holds e4m3 codes (128 B per row), else bf16
  int32_t xpf_mode;                   // expert prefetch while the routing is pending: 0 off, 1 the
                                      // shared experts, plus the last routing's experts when at least
                                      // half of them repeated the routing before it; 2 both always
  StepState* state;
  Status* status;
  uint32_t* tickets;
  uint32_t* ctr;                      // arrival counters: one per op, then one per (layer, kv head)
  uint64_t* part;                     // attention partials, tagged [n_kv][ns_max][Mmax*G][kPart]
  float* am_val;                      // argmax partials [n_ctas][Mmax]
  int32_t* am_idx;
  int32_t* am_out;                    // argmax [Mmax]
  int32_t step_ticket;                // ticket index of the step-end rendezvous
  int32_t n_steps, pad2;              // greedy steps this launch runs (> 1: chained in the kernel)
  uint64_t* hs;                       // hidden stream, tagged [2L + 1][Mmax][H]
  uint64_t* trace;                    // DEC_TRACE builds: [n_ctas][n_ops][kTraceFields] %globaltimer stamps
  int32_t attn_tc, attn_window;       // attn_window: 0 global, W > 0 the last W positions per token;
                                      // attn_tc 1: bf16 attention tiles come by TMA tensor copies (128-byte
                                      // swizzle) and run on the tensor cores
  CUtensorMap tmap_k, tmap_v;         // the bf16 key / value caches as 2D tensors: 128 columns x
                                      // (L n_kv cap) rows, boxes of 64 columns x kAttnTcRows rows
};

// Trace record of one (CTA, op), DEC_TRACE builds only (compiled out otherwise):
// consumer op start, input ready, prologue done, all warps' tiles done, op end;
// producer first issue, last issue, tiles issued; first thread's input loads done, input words
// found not yet visible (re-polled), attention merge start, attention merge inputs ready.
constexpr int kTraceFields = 12;
// DEC_TRACE builds also log the first kTileLog tiles of every consumer warp of CTA 0, in SM
// clock cycles (clock64): issued by the producer, consumer starts waiting, data landed,
// compute done, slot released (5 stamps + pad per tile).
constexpr int kTileLog = 1024;
constexpr int kTileStamps = 6;

#ifdef __CUDACC__
#define DEC_HD __host__ __device__
#else
#define DEC_HD
#endif

// Bytes of one cached key (or value) row, and the KV rows one ring slot takes (keys then values;
// at most 32: the softmax keeps one row per lane).
DEC_HD inline int kv_row_bytes(int kv_fp8) { return kv_fp8 ? 128 : 256; }
DEC_HD inline int attn_rows_per_slot(int slot_bytes, int kv_fp8) {
  const int r = slot_bytes / (2 * kv_row_bytes(kv_fp8));
  return r < 32 ? r : 32;
}

// Attention scratch inside a CTA's activation area, in floats from its (256-byte aligned) start;
// the kernel carves it and the host sizes the area with the same function. P: KV rows per
// ring slot; ns: splits per kv head.
struct AttnLayout {
  int q, sc, mg, kvn, cw, ml, raw, end;
};

DEC_HD inline AttnLayout attn_layout(int M, int G, int P, int ns) {
  auto up4 = [](int f) { return (f + 3) & ~3; };  // 16-byte boundary
  const int MG = M * G;
  const int prods = ((MG * 32 + ns - 1) / ns + 1) * ns * 4;  // the merge's output slices of every split
  AttnLayout l;
  l.q = 0;                                                      // [M*G][128] rotated queries
  l.sc = l.q + MG * 128;                                        // per-warp scores / merge slices
  l.mg = up4(l.sc + (kConsumerWarps * G * P > prods ? kConsumerWarps * G * P : prods));
  l.kvn = l.mg + kConsumerWarps * G * kPart;                    // per-warp split states
  l.cw = l.kvn + kMmax * 128;                                   // own keys / values ([2][M][128] bf16 or e4m3)
  l.ml = up4(l.cw + MG * ns);                                   // merge weights
  l.raw = up4(l.ml + 2 * MG * ns);                              // splits' (max, sum)
  l.end = l.raw + M * (G + 2) * 128;                            // polled q / k / v rows
  return l;
}

// Device address of the allocation-free LM head's static scratch on the current device
// (noalloc.cu); the first call on a device looks it up.
cudaError_t noalloc_scratch(void** ptr);

}  // namespace decimpl
