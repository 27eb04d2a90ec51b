// Internal layout shared by the host runtime (api.cpp) and the megakernel (megakernel.cu).
//
// A decode step is a fixed list of ops (OpDesc). Every CTA of the persistent grid walks
// the whole list; for each op it takes its own share of the op's rows (or attention
// positions), split into tiles that fit one shared-memory ring slot. A producer warp
// streams tiles of weights / KV history into the ring with bulk asynchronous copies;
// eight consumer warps wait on the op's input (a global counter), compute, and signal the
// op's own counter. Weights and cached KV never depend on the running step, so the
// producer runs ahead of the consumers across op boundaries: the next op's weights are
// already in flight while the previous op is still being finished elsewhere (the
// multiprogramming argument of the Muse Spark Open megakernel article, section "the
// baseline nobody benchmarked", and its weight-prefetch ring, section "three bills").
#pragma once
#include <stdint.h>

namespace decimpl {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kSlotBytes = 32768;                // one ring slot
constexpr int kMaxSlots = 8;                     // ring slots at most
constexpr int kRmax = 8;                         // rows one thread accumulates per tile
constexpr int kMmax = 4;                         // tokens per call (verify window)
constexpr int kHeadDim = 128;
constexpr int kAttnTilePos = 64;                 // positions per attention tile: 64 x 256 B x (K+V) = 32 KB
constexpr int kMaxRouteSlots = 1 + 8 * kMmax;    // shared + union of routed experts
constexpr int kSmemLimit = 232448;               // dynamic shared memory per CTA on sm_103a

enum OpType : int32_t {
  OP_QKV = 0,           // a = RMSNorm(x); qkv = W_qkv a
  OP_ATTN = 1,          // split-K GQA attention (+ RoPE, KV append, log-sum-exp combine)
  OP_OPROJ = 2,         // x' = x + W_o o
  OP_GATEUP = 3,        // b = RMSNorm(x'); h = silu(W_g b) * (W_u b)   (pair-interleaved rows)
  OP_DOWN = 4,          // x'' = x' + W_d h
  OP_ROUTER = 5,        // b = RMSNorm(x'); r = W_r b (fp32); top-k + softmax (last CTA)
  OP_SHARED_GATEUP = 6, // h_s = SwiGLU gate/up of the shared experts (MXFP4)
  OP_ROUTED_GATEUP = 7, // h_e = SwiGLU gate/up of the routed experts (MXFP4)
  OP_EXP_DOWN = 8,      // x'' = x' + sum_slots w * W_d,e h_e
  OP_LMHEAD = 9,        // logits = W_lm RMSNorm(x); argmax (block, then last CTA)
};

enum WType : int32_t { W_BF16 = 0, W_FP8 = 1, W_MXFP4 = 2 };
enum XSrc : int32_t { X_NONE = 0, X_F32 = 1, X_HIDDEN_IN = 2, X_EMBED = 3 };

struct OpDesc {
  int32_t type, wtype, layer, N;      // N: rows of one matrix (per expert for expert ops)
  int32_t K, rpt, tpr, pair;          // cols, rows per tile, threads per row group, pair rows
  int32_t wait_ctr, wait_n;           // consumer dependency: counter, contributions per step
  int32_t wait2_ctr, wait2_n;         // second dependency (-1: none)
  int32_t pwait_ctr, pwait_n;         // producer dependency (routing), -1: none
  int32_t sig_ctr, ticket;            // counter this op signals; ticket base (attention, router, head)
  int32_t norm, xsrc;                 // input = RMSNorm(x) * gain; source of x
  int32_t slot0, slot1;               // expert slots [slot0, slot1) (slot1 < 0: up to n_slots)
  int32_t x_idx, unit;                // hidden-stream entry of x (X_F32); row granularity of the CTA split
  const void* w;                      // packed values (expert ops: expert 0)
  const void* ws;                     // scales plane (FP8 row scales / MXFP4 E8M0), else null
  int64_t w_mstride, ws_mstride;      // bytes between experts
  const uint16_t* gain;               // RMSNorm gain, bf16 [H]
  const void* x_src;                  // X_EMBED: embedding table bf16 [V][H]
  float* x_out;                       // residual output fp32 [Mmax][H]
  const float* act;                   // plain input fp32 [Mmax][K] (o-proj: attention out; down: h)
  float* out;                         // output fp32: qkv [Mmax][qkv], h [Mmax][F], router logits, LM logits
  uint16_t* kc;                       // this layer's key cache  bf16 [n_kv][cap][128]
  uint16_t* vc;                       // this layer's value cache bf16 [n_kv][cap][128]
  int32_t* route;                     // this layer's RouteBlock
  float* eh;                          // this layer's expert hidden fp32 [slots][Mmax][I]
};

struct RouteBlock {
  int32_t n_slots;                    // n_shared + distinct routed experts
  int32_t expert[kMaxRouteSlots];     // expert id per slot (shared experts first: id >= E)
  float w[kMmax][kMaxRouteSlots];     // weight of slot for token m (1 for shared, pi or 0)
  int32_t topk[kMmax][8];             // per-token selection, best first
  float topk_w[kMmax][8];
};

struct StepState {
  uint32_t epoch;                     // completed steps; counters reach (epoch+1)*n during a step
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
  int32_t nslot, act_bytes;
  StepState* state;
  Status* status;
  uint32_t* ctr;
  uint32_t* tickets;
  float* part;                        // attention partials [n_kv][ns_max][Mmax*G][2 + 128]
  float* am_val;                      // argmax partials [n_ctas][Mmax]
  int32_t* am_idx;
  int32_t* am_out;                    // argmax [Mmax]
  int32_t step_ticket;                // ticket index of the step-end rendezvous
  float* hs;                          // hidden stream fp32 [2L + 1][Mmax][H]
};

}  // namespace decimpl
