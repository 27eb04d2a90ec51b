// Host side of the C ABI declared in include/dec.h: config validation, workspace layout,
// the step's op list, launch modes (persistent / per op / per-op CUDA graph) and the
// sticky device status.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/dec.h"
#include "dec_internal.h"

using namespace decimpl;

#ifndef DEC_ATTN_SPLIT_DIV
#define DEC_ATTN_SPLIT_DIV 1
#endif
#ifndef DEC_ATTN_TC
#define DEC_ATTN_TC 1  // bf16 attention on the tensor cores, its tiles by TMA tensor copies
#endif

extern "C" cudaError_t dec_launch_megakernel(const KParams* kp, int cooperative, cudaStream_t stream);
extern "C" int dec_megakernel_common_bytes(void);
extern "C" cudaError_t dec_launch_pack(int dtype, const uint16_t* a, const uint16_t* b, int rows, int cols,
                                       void* vals, void* scales, cudaStream_t stream);
extern "C" cudaError_t dec_launch_pack_kv_fp8(const uint16_t* v, size_t n, float s, uint8_t* out,
                                              cudaStream_t stream);

namespace {

thread_local std::string g_last_error;

dec_status fail(dec_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

#define CUDA_TRY(expr)                                                                     \
  do {                                                                                     \
    cudaError_t e_ = (expr);                                                               \
    if (e_ != cudaSuccess) return fail(DEC_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct LayerW {
  const void* attn_norm = nullptr;
  const void* wqkv = nullptr;
  const void* wo = nullptr;
  const void* ffn_norm = nullptr;
  const void* wgateup = nullptr;
  const void* wdown = nullptr;
  const void* wrouter = nullptr;
  const void* egu_v = nullptr;
  const void* egu_s = nullptr;
  const void* edn_v = nullptr;
  const void* edn_s = nullptr;
};

constexpr int kMaxSubOps = 8;  // ops of one layer (at most 7) or of the LM head alone

struct Layout {  // byte offsets into the workspace
  size_t state, status, tickets, ctr, ops, subops, wops, tmaps, hs, qkv, attn_out, hbuf, rlogits, route, xpf, eh, part, logits, am_val,
      am_idx, am_out, trace, total;
  int n_ops, n_tickets, n_ctas, ns_max, slot_bytes, act_bytes, exp_stage_all;
  int slot1_bytes, act1_bytes, exp_stage_all1;  // the one-token list's geometry
};

bool validate(const dec_config* c, std::string& why) {
  auto bad = [&](const char* m) { why = m; return false; };
  if (!c) return bad("null config");
  if (c->n_layers < 0 || c->hidden <= 0 || c->hidden % 64) return bad("hidden must be a positive multiple of 64");
  if (c->max_verify < 1 || c->max_verify > kMmax) return bad("max_verify must be 1..4");
  const bool attn = c->n_q > 0;
  if (c->n_layers > 0 && !attn && c->ffn == 0 && c->n_experts == 0) return bad("layers without blocks");
  if (attn) {
    if (c->head_dim != kHeadDim) return bad("head_dim must be 128");
    if (c->n_kv <= 0 || c->n_q % c->n_kv) return bad("n_q must be a multiple of n_kv");
    const int G = c->n_q / c->n_kv;
    if (G != 1 && G != 2 && G != 4 && G != 5 && G != 8) return bad("query heads per kv head must be 1, 2, 4, 5 or 8");
    if (c->kv_capacity < 1) return bad("kv_capacity must be positive");
  }
  if (c->ffn < 0 || c->ffn % 8) return bad("ffn must be a multiple of 8");
  if (c->ffn && c->n_experts) return bad("a layer is dense or MoE, not both");
  if (c->n_experts) {
    if (c->top_k < 1 || c->top_k > 8 || c->top_k > c->n_experts) return bad("top_k must be 1..min(8, E)");
    if (c->moe_inter <= 0 || c->moe_inter % 32) return bad("moe_inter must be a positive multiple of 32");
    if (c->n_shared < 0 || c->n_shared > 1) return bad("n_shared must be 0 or 1");
    if (c->expert_dtype != DEC_MXFP4) return bad("expert_dtype must be DEC_MXFP4");
    if ((2LL * c->moe_inter * (c->hidden / 32)) % 16 || (1LL * c->hidden * (c->moe_inter / 32)) % 16)
      return bad("MXFP4 scale planes of one expert must be multiples of 16 bytes");
  }
  if (c->vocab < 0) return bad("vocab must be >= 0");
  if (c->vocab && c->lm_head_dtype != DEC_BF16 && c->lm_head_dtype != DEC_FP8_E4M3_ROWSCALE)
    return bad("lm_head_dtype must be DEC_BF16 or DEC_FP8_E4M3_ROWSCALE");
  if (c->embedding && c->vocab <= 0) return bad("embedding needs a vocabulary");
  if (c->mode < DEC_MODE_PERSISTENT || c->mode > DEC_MODE_PER_OP_GRAPH) return bad("bad mode");
  if (c->num_ctas < 0) return bad("num_ctas must be >= 0");
  if (c->kv_dtype != DEC_BF16 && c->kv_dtype != DEC_FP8_E4M3) return bad("kv_dtype must be DEC_BF16 or DEC_FP8_E4M3");
  if (c->attn_window < 0 || (c->attn_window > 0 && c->attn_window < c->max_verify))
    return bad("attn_window must be 0 (global) or at least max_verify");
  if (!std::isfinite(c->rms_eps) || c->rms_eps < 0) return bad("rms_eps must be >= 0");
  return true;
}

// Attention runs on the tensor cores for a bf16 cache with at most 8 query heads per kv head.
bool attn_tc_for(const dec_config* c) {
  return DEC_ATTN_TC && c->n_q > 0 && c->kv_dtype == DEC_BF16 && c->n_q / c->n_kv <= 8;
}

int ctas_for(const dec_config* c) {
  if (c->num_ctas > 0) return c->num_ctas;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int count_ops(const dec_config* c) {
  int n = 0;
  for (int l = 0; l < c->n_layers; ++l) {
    if (c->n_q) n += 3;
    if (c->ffn) n += 2;
    if (c->n_experts) n += 3;
  }
  if (c->vocab) n += 1;
  return n;
}

int pow2_floor(int v) {
  int p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}

int gcd(int a, int b) { return b ? gcd(b, a % b) : a; }

// Tile geometry of a [N][K] matrix of dtype wt streamed through `slot`-byte warp slots:
// rows per tile R (nr * M <= 32 results per warp), columns per tile Kc, and the row
// granularity `unit` of the CTA / warp split (gate/up pairs; 16-byte MXFP4 scale copies).
void tile_geometry(int wt, int K, int pair, int slot, int Mmax, int& R, int& Kc, int& unit) {
  const double bpc = wt == W_BF16 ? 2.0 : (wt == W_FP8 ? 1.0 : 0.5 + 1.0 / 32.0);
  unit = pair ? 2 : 1;
  if (wt == W_MXFP4) {
    const int us = 16 / gcd(16, K / 32);
    unit = unit * us / gcd(unit, us);
  }
  const int rmax = std::min(kRmax, 32 / Mmax) / unit * unit;
  auto fits = [&](int r, int kc) {
    const size_t vb = wt == W_BF16 ? (size_t)2 * kc : (wt == W_FP8 ? (size_t)kc : (size_t)kc / 2);
    const size_t sb = wt == W_MXFP4 ? (size_t)kc / 32 : 0;
    return ((size_t)r * vb + 15) / 16 * 16 + (size_t)r * sb <= (size_t)slot;
  };
  if (fits(unit, K)) {
    int r = rmax;
    while (r > unit && !fits(r, K)) r -= unit;
    R = r;
    Kc = K;
    return;
  }
  // a row does not fit: split the columns; two rows per tile share each activation load
  R = std::max(unit, std::min(2, rmax));
  const int gran = wt == W_BF16 ? 256 : 512;
  int kc = (int)((double)slot / (R * bpc)) / gran * gran;
  while (kc > gran && !fits(R, kc)) kc -= gran;
  Kc = kc;
}

bool compute_layout(const dec_config* c, Layout& L, std::string& why) {
  const int C = ctas_for(c);
  if (C <= 0) {
    why = "no CUDA device to size the grid (set num_ctas)";
    return false;
  }
  const int M = c->max_verify, H = c->hidden, nl = c->n_layers;
  const int G = c->n_q ? c->n_q / c->n_kv : 1;
  const int qkv_rows = c->n_q ? (c->n_q + 2 * c->n_kv) * kHeadDim : 0;
  L.n_ctas = C;
  L.n_ops = count_ops(c);
  // attention splits per kv head: every CTA takes one split (fewer, longer splits: knob)
  L.ns_max = c->n_q ? std::max(1, C / c->n_kv / DEC_ATTN_SPLIT_DIV) : 1;
  L.n_tickets = 2;  // LM-head argmax, step end

  // Shared-memory geometry of a list whose calls carry up to Mg tokens: the scratch ("act") its
  // largest op needs, in floats (a multi-token list's tensor-core ops stage their inputs in
  // kMmax tokens' bytes whatever the window), and the ring slots the rest leaves.
  const int rows_cta = (H + C - 1) / C + 16;
  auto geometry = [&](int Mg, int& slot_bytes, int& act_bytes, int& stage_all) -> bool {
    const int Ma = Mg > 1 ? kMmax : 1;
    size_t act = (size_t)Ma * H;
    act = std::max(act, (size_t)2 * kConsumerThreads);
    if (c->n_q) {
      act = std::max(act, (size_t)Ma * c->n_q * kHeadDim + (size_t)rows_cta * Mg * (1 + kConsumerWarps));
      // the attention scratch the kernel carves (at most 32 KV rows per ring slot)
      act = std::max(act, (size_t)attn_layout(Mg, G, kMaxSlotBytes / 512, L.ns_max).end);
    }
    if (c->ffn) act = std::max(act, (size_t)Ma * c->ffn + (size_t)rows_cta * Mg * (1 + kConsumerWarps));
    act = std::max(act, (size_t)Ma * H + (size_t)2 * (rows_cta + 1) * Mg * kConsumerWarps);  // column-split partials
    stage_all = 0;
    if (c->n_experts) {
      act = std::max(act, (size_t)Mg * c->n_experts);
      const size_t per_slot = (size_t)Mg * c->moe_inter + 2 * (size_t)rows_cta * Mg;
      // every slot's hidden vectors, the residual rows and one set of partial sums per warp
      const size_t all =
          (size_t)(c->n_shared + c->top_k * Mg) * Mg * c->moe_inter + (1 + kConsumerWarps) * (size_t)rows_cta * Mg;
      if (all <= std::max(act, (size_t)7168)) {
        act = std::max(act, all);
        stage_all = 1;
      } else {
        act = std::max(act, per_slot);
      }
    }
    act = align_up(act * 4, 256);
    const int common = dec_megakernel_common_bytes();
    const long long room = (long long)kSmemLimit - (long long)act - common;
    // ring slots: 256-byte multiples, 1024 when tensor copies with a 128-byte swizzle land in them
    const int slot_align = (attn_tc_for(c) || c->max_verify > 1) ? 1024 : 256;
    long long slot = room / (kConsumerWarps * kStages) / slot_align * slot_align;
    slot = std::min<long long>(slot, kMaxSlotBytes);
    if (slot < 4096) return false;
    slot_bytes = (int)slot;
    act_bytes = (int)act;
    return true;
  };
  // multi-token calls (and the layer-level entry points) use the max_verify geometry; one-token
  // steps run a list of their own with the smaller scratch of one token and larger ring slots
  if (!geometry(M, L.slot_bytes, L.act_bytes, L.exp_stage_all) ||
      !geometry(1, L.slot1_bytes, L.act1_bytes, L.exp_stage_all1)) {
    why = "shapes need more shared memory than a CTA has";
    return false;
  }

  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.state = take(sizeof(StepState));
  L.status = take(sizeof(Status));
  L.tickets = take((size_t)L.n_tickets * 4);
  L.ctr = take((size_t)(std::max(1, L.n_ops) + (c->n_q ? nl * c->n_kv : 0)) * 4);
  L.ops = take((size_t)std::max(1, L.n_ops) * sizeof(OpDesc));
  L.subops = take((size_t)kMaxSubOps * sizeof(OpDesc));  // a layer or the LM head run on its own
  // multi-token calls (max_verify > 1): their own op list, and a tensor map per tensor-core op
  L.wops = take((size_t)(c->max_verify > 1 ? std::max(1, L.n_ops) : 0) * sizeof(OpDesc));
  L.tmaps = take((size_t)(c->max_verify > 1 ? std::max(1, L.n_ops) : 0) * sizeof(CUtensorMap));
  // activations handed between CTAs are tagged 8-byte words (see ptx.cuh), one buffer per
  // layer so that no word is written twice in a step
  L.hs = take((size_t)(2 * nl + 1) * M * H * 8);
  L.qkv = take((size_t)nl * M * qkv_rows * 8);
  L.attn_out = take((size_t)nl * M * c->n_q * kHeadDim * 8);
  L.hbuf = take((size_t)nl * M * c->ffn * 8);
  L.rlogits = take((size_t)nl * M * c->n_experts * 8);
  L.route = take((size_t)(c->n_experts ? nl : 0) * sizeof(RouteBlock));
  L.xpf = take((size_t)(c->n_experts ? nl : 0) * kXpfWords * 4);
  L.eh = take((size_t)(c->n_experts ? nl : 0) * kMaxRouteSlots * M * c->moe_inter * 8);
  L.part = take((size_t)(c->n_q ? nl * c->n_kv : 0) * L.ns_max * M * G * kPart * 8);
  L.logits = take((size_t)M * c->vocab * 4);
  L.am_val = take((size_t)C * kMmax * 4);
  L.am_idx = take((size_t)C * kMmax * 4);
  L.am_out = take((size_t)kMmax * 4);
#ifdef DEC_TRACE
  L.trace = take((size_t)C * std::max(1, L.n_ops) * kTraceFields * 8 + (size_t)kConsumerWarps * kTileLog * kTileStamps * 8);
#else
  L.trace = 0;
#endif
  L.total = o;
  return true;
}

}  // namespace

struct dec_ctx {
  dec_config cfg;
  cudaStream_t stream;
  uint8_t* ws;
  Layout lay;
  std::vector<LayerW> layers;
  const void* embed = nullptr;
  const void* final_norm = nullptr;
  const void* lm_v = nullptr;
  const void* lm_s = nullptr;
  uint8_t* kc = nullptr;   // bf16 or e4m3 rows (kv_row_bytes)
  uint8_t* vc = nullptr;
  const float* kv_scales = nullptr;  // FP8 cache: [n_layers][2][n_kv] (null: all 1)
  bool ops_dirty = true;
  std::vector<OpDesc> ops;
  KParams kp;
  bool sticky = false;
  dec_status sticky_code = DEC_OK;
  cudaGraphExec_t graph = nullptr;
  int attn_tc = 0;                   // tensor-core attention (tensor maps below encoded)
  int xpf_mode = 0;                  // expert prefetch (DEC_EXPERT_PREFETCH: 0 off, 1 adaptive, 2 always)
  std::vector<OpDesc> wops;          // the op list of multi-token calls (max_verify > 1)
  KParams wkp;
  std::vector<CUtensorMap> tmaps_host;  // the tensor maps of its tensor-core ops
  const void* tmap_kc = nullptr;     // the caches the tensor maps describe
  const void* tmap_vc = nullptr;
  CUtensorMap tmap_k, tmap_v;
  int last_launches = 0;
  int drop_op = -1;  // failure injection: the next per-op call skips launching this op
};

namespace {

template <class T>
T* wsp(dec_ctx* c, size_t off) {
  return reinterpret_cast<T*>(c->ws + off);
}

dec_status check_layer(dec_ctx* c, int l) {
  const dec_config& g = c->cfg;
  const LayerW& w = c->layers[l];
  if (g.n_q && (!w.attn_norm || !w.wqkv || !w.wo)) return fail(DEC_ERR_STATE, "layer %d: attention weights missing", l);
  if ((g.ffn || g.n_experts) && !w.ffn_norm) return fail(DEC_ERR_STATE, "layer %d: ffn_norm missing", l);
  if (g.ffn && (!w.wgateup || !w.wdown)) return fail(DEC_ERR_STATE, "layer %d: dense FFN weights missing", l);
  if (g.n_experts && (!w.wrouter || !w.egu_v || !w.egu_s || !w.edn_v || !w.edn_s))
    return fail(DEC_ERR_STATE, "layer %d: MoE weights missing", l);
  if (g.n_q && (!c->kc || !c->vc)) return fail(DEC_ERR_STATE, "KV cache not set");
  return DEC_OK;
}

dec_status check_head(dec_ctx* c) {
  const dec_config& g = c->cfg;
  if (g.vocab && (!c->lm_v || (g.final_norm && !c->final_norm))) return fail(DEC_ERR_STATE, "LM head missing");
  if (g.vocab && g.lm_head_dtype == DEC_FP8_E4M3_ROWSCALE && !c->lm_s) return fail(DEC_ERR_STATE, "LM head scales missing");
  return DEC_OK;
}

dec_status check_weights(dec_ctx* c) {
  const dec_config& g = c->cfg;
  for (int l = 0; l < g.n_layers; ++l) {
    const dec_status st = check_layer(c, l);
    if (st != DEC_OK) return st;
  }
  if (g.embedding && !c->embed) return fail(DEC_ERR_STATE, "embedding missing");
  return check_head(c);
}

// The driver's tensor-map encoder, looked up once through the runtime (no link against the driver
// library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

constexpr int kLmHeadTicket = 0;  // tickets: the LM head's argmax, then the step end
constexpr int kStepTicket = 1;

// Op-list builder: the ops of a layer or of the LM head, appended to a list. The state
// carries what the next block reads (its input's source and hidden-stream entry) and the op
// producing it (for the counted-read build option).
struct ListBuilder {
  dec_ctx* c;
  std::vector<OpDesc>& ops;
  int xsrc, x_idx, prev;
  bool window = false;               // a multi-token list: bf16 matrices on tensor-core tiles
  int gm;                            // tokens the list's geometry serves: 1, or max_verify
  int slot, act, stage_all;          // its ring slot and scratch bytes, expert-down staging
  dec_status err = DEC_OK;

  ListBuilder(dec_ctx* c_, std::vector<OpDesc>& ops_, int xsrc_, bool one_token = false)
      : c(c_), ops(ops_), xsrc(xsrc_), x_idx(0), prev(-1) {
    const Layout& L = c->lay;
    gm = one_token ? 1 : c->cfg.max_verify;
    slot = one_token ? L.slot1_bytes : L.slot_bytes;
    act = one_token ? L.act1_bytes : L.act_bytes;
    stage_all = one_token ? L.exp_stage_all1 : L.exp_stage_all;
  }

  OpDesc blank(int type) const {
    OpDesc o;
    std::memset(&o, 0, sizeof(o));
    o.type = type;
    o.ctr = (int)ops.size();
    o.wait_ctr = prev;
    o.wait_n = c->lay.n_ctas;
    o.aux_ctr = -1;
    o.xsrc = xsrc;
    o.x_idx = x_idx;
    o.x_src = c->embed;
    o.slot1 = -1;
    return o;
  }

  void geom(OpDesc& o) {
    const Layout& L = c->lay;
    const int M = gm;
    if (window && o.wtype == W_BF16 && o.K % 64 == 0 && o.N % kGemvTcRows == 0 &&
        slot >= kGemvTcRows * 2 * 64) {
      // tensor-core tiles: kGemvTcRows rows x Kc columns in boxes of 64 columns (128-byte swizzle)
      o.tc = 1;
      o.R = kGemvTcRows;
      o.unit = kGemvTcRows;
      int kc = (slot / (kGemvTcRows * 2 * 64)) * 64;
      o.Kc = std::min(o.K, kc);
      o.csplit = 0;
      o.kw = 0;
      // fewer row groups per CTA than warps: split the columns across the warps instead (the
      // partial sums of the CTA's rows must fit next to the staged inputs)
      const int C = L.n_ctas, groups = (o.N / kGemvTcRows + C - 1) / C;
      const size_t parts = (size_t)kConsumerWarps * groups * kGemvTcRows * M;
      const size_t staged = (size_t)kMmax * o.K + (o.type == OP_OPROJ || o.type == OP_DOWN ? (size_t)groups * kGemvTcRows * M : 0);
      if (o.type != OP_LMHEAD && groups < kConsumerWarps && (staged + parts) * 4 <= (size_t)act) {
        o.csplit = 1;
        o.kw = ((o.K + kConsumerWarps - 1) / kConsumerWarps + 63) / 64 * 64;
      }
      encode_tmap(o);
      return;
    }
    tile_geometry(o.wtype, o.K, o.pair, slot, M, o.R, o.Kc, o.unit);
    // rows too wide for one slot (or for activations in registers): split the columns across
    // the CTA's warps instead of its rows (bf16 / FP8 matrices without expert slots)
    const int cw = o.wtype == W_BF16 ? 8 : (o.wtype == W_FP8 ? 16 : 32);
    const int ni = o.wtype == W_BF16 ? 10 : (o.wtype == W_FP8 ? 5 : 3);
    const bool experts = o.type == OP_ROUTED_GATEUP || o.type == OP_EXP_DOWN;
    if (!experts && o.type != OP_LMHEAD && o.wtype != W_MXFP4 && (o.Kc < o.K || o.K > 32 * ni * cw)) {
      const int kw = ((o.K + kConsumerWarps - 1) / kConsumerWarps + cw - 1) / cw * cw;
      const int bpc = o.wtype == W_BF16 ? 2 : 1;
      int r = std::min(kRmax, 32 / M);
      while (r > o.unit && (size_t)r * kw * bpc > (size_t)slot) r -= o.unit;
      if ((size_t)r * kw * bpc <= (size_t)slot && kw <= 32 * ni * cw) {
        o.csplit = 1;
        o.Kc = kw;
        o.R = r / o.unit * o.unit;
      }
    }
  }

  // The op's bf16 weight matrix as a 2D tensor map (K columns x N rows, boxes of 64 columns x
  // kGemvTcRows rows, 128-byte swizzle), kept on the host and uploaded with the list.
  void encode_tmap(OpDesc& o) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    CUtensorMap m;
    std::memset(&m, 0, sizeof(m));
    if (!enc) {
      err = fail(DEC_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    } else {
      const cuuint64_t dims[2] = {(cuuint64_t)o.K, (cuuint64_t)o.N};
      const cuuint64_t strides[1] = {(cuuint64_t)o.K * 2};
      const cuuint32_t box[2] = {64, (cuuint32_t)kGemvTcRows};
      const cuuint32_t estr[2] = {1, 1};
      const CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(o.w), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) err = fail(DEC_ERR_CUDA, "encoding a weight tensor map failed (CUresult %d)", (int)r);
    }
    o.tmap = reinterpret_cast<const CUtensorMap*>(c->ws + c->lay.tmaps) + c->tmaps_host.size();
    c->tmaps_host.push_back(m);
  }

  uint64_t* hs_at(int idx) const {  // tagged [Mmax][H]
    return wsp<uint64_t>(c, c->lay.hs) + (size_t)idx * c->cfg.max_verify * c->cfg.hidden;
  }

  // The ops of decoder layer l: attention block (QKV, attention, o-proj), then the dense FFN
  // (gate/up, down) or the MoE FFN (router, shared and routed gate/up, expert down).
  void layer(int l) {
    const dec_config& g = c->cfg;
    const Layout& L = c->lay;
    const int M = g.max_verify, H = g.hidden;
    const int qkv_rows = g.n_q ? (g.n_q + 2 * g.n_kv) * kHeadDim : 0;
    const LayerW& w = c->layers[l];
    if (g.n_q) {
      OpDesc q = blank(OP_QKV);
      q.layer = l;
      q.wtype = W_BF16;
      q.N = qkv_rows;
      q.K = H;
      q.norm = 1;
      q.gain = static_cast<const uint16_t*>(w.attn_norm);
      q.w = w.wqkv;
      q.out = wsp<uint64_t>(c, L.qkv) + (size_t)l * M * qkv_rows;
      geom(q);
      ops.push_back(q);
      prev = q.ctr;

      OpDesc a = blank(OP_ATTN);
      a.layer = l;
      a.act = q.out;
      a.out = wsp<uint64_t>(c, L.attn_out) + (size_t)l * M * g.n_q * kHeadDim;
      a.aux_ctr = L.n_ops + l * g.n_kv;  // per-kv-head counters of the splits' partials
      const size_t kv_layer = (size_t)l * g.n_kv * g.kv_capacity * kv_row_bytes(g.kv_dtype == DEC_FP8_E4M3);
      a.kc = c->kc + kv_layer;
      a.vc = c->vc + kv_layer;
      a.kv_scale = c->kv_scales ? c->kv_scales + (size_t)l * 2 * g.n_kv : nullptr;
      ops.push_back(a);
      prev = a.ctr;

      OpDesc o = blank(OP_OPROJ);
      o.layer = l;
      o.wtype = W_BF16;
      o.N = H;
      o.K = g.n_q * kHeadDim;
      o.w = w.wo;
      o.act = a.out;
      o.x_out = hs_at(2 * l + 1);
      geom(o);
      ops.push_back(o);
      prev = o.ctr;
      xsrc = X_F32;
      x_idx = 2 * l + 1;
    }
    if (g.ffn) {
      OpDesc u = blank(OP_GATEUP);
      u.layer = l;
      u.wtype = W_BF16;
      u.N = 2 * g.ffn;
      u.K = H;
      u.pair = 1;
      u.norm = 1;
      u.gain = static_cast<const uint16_t*>(w.ffn_norm);
      u.w = w.wgateup;
      u.out = wsp<uint64_t>(c, L.hbuf) + (size_t)l * M * g.ffn;
      geom(u);
      ops.push_back(u);
      prev = u.ctr;

      OpDesc d = blank(OP_DOWN);
      d.layer = l;
      d.wtype = W_BF16;
      d.N = H;
      d.K = g.ffn;
      d.w = w.wdown;
      d.act = u.out;
      d.x_out = hs_at(2 * l + 2);
      geom(d);
      ops.push_back(d);
      prev = d.ctr;
      xsrc = X_F32;
      x_idx = 2 * l + 2;
    }
    if (g.n_experts) {
      const int I = g.moe_inter, E = g.n_experts;
      int32_t* route = reinterpret_cast<int32_t*>(wsp<uint8_t>(c, L.route) + (size_t)l * sizeof(RouteBlock));
      int32_t* xpf = wsp<int32_t>(c, L.xpf) + (size_t)l * kXpfWords;
      uint64_t* eh = wsp<uint64_t>(c, L.eh) + (size_t)l * kMaxRouteSlots * M * I;
      uint64_t* rlogits = wsp<uint64_t>(c, L.rlogits) + (size_t)l * M * E;
      const int64_t gu_v = (int64_t)2 * I * (H / 2), gu_s = (int64_t)2 * I * (H / 32);
      const int64_t dn_v = (int64_t)H * (I / 2), dn_s = (int64_t)H * (I / 32);

      OpDesc r = blank(OP_ROUTER);
      r.layer = l;
      r.wtype = W_BF16;
      r.N = E;
      r.K = H;
      r.norm = 1;
      r.gain = static_cast<const uint16_t*>(w.ffn_norm);
      r.w = w.wrouter;
      r.out = rlogits;
      r.act = rlogits;  // routing ops read the layer's router logits
      r.route = route;
      r.xpf = xpf;
      r.aux_ctr = r.ctr;  // the routing waits for every CTA's logits
      geom(r);
      ops.push_back(r);
      const int x_ready = r.wait_ctr;  // the experts' gate/up reads x' like the router

      OpDesc rg = blank(OP_ROUTED_GATEUP);
      rg.layer = l;
      rg.wtype = W_MXFP4;
      rg.N = 2 * I;
      rg.K = H;
      rg.pair = 1;
      rg.norm = 1;
      rg.gain = static_cast<const uint16_t*>(w.ffn_norm);
      rg.w = w.egu_v;
      rg.ws = w.egu_s;
      rg.w_mstride = gu_v;
      rg.ws_mstride = gu_s;
      rg.slot0 = 0;  // every slot: the shared experts first, then the routed ones
      rg.slot1 = -1;
      rg.eh = eh;
      rg.route = route;
      rg.xpf = xpf;
      rg.act = rlogits;
      rg.wait_ctr = x_ready;  // its own input is x'; its routing waits for the router (aux)
      rg.aux_ctr = r.ctr;
      geom(rg);
      ops.push_back(rg);

      OpDesc dn = blank(OP_EXP_DOWN);
      dn.layer = l;
      dn.wtype = W_MXFP4;
      dn.N = H;
      dn.K = I;
      dn.w = w.edn_v;
      dn.ws = w.edn_s;
      dn.w_mstride = dn_v;
      dn.ws_mstride = dn_s;
      dn.eh = eh;
      dn.route = route;
      dn.xpf = xpf;
      dn.act = rlogits;
      dn.wait_ctr = rg.ctr;  // routed (and, earlier in every CTA, shared) expert hidden vectors
      dn.aux_ctr = r.ctr;
      dn.x_out = hs_at(2 * l + 2);
      dn.stage_all = stage_all;
      geom(dn);
      if (dn.stage_all && dn.Kc == dn.K) {
        // slot split: the CTA's rows of each slot in about two chunks, one chunk per warp item
        const int C = L.n_ctas, units = (H / dn.unit + C - 1) / C;
        const int nr_max = gm == 1 ? 10 : 8;  // the kernel's tile rows for one token / a window
        int R = (units + 1) / 2 * dn.unit;
        const size_t row_b = (size_t)I / 2 + I / 32;
        while (R > dn.unit && (R > nr_max || (size_t)R * row_b + 16 > (size_t)slot)) R -= dn.unit;
        dn.R = R;
        dn.csplit = 1;
      }
      ops.push_back(dn);
      prev = dn.ctr;
      xsrc = X_F32;
      x_idx = 2 * l + 2;
    }
  }

  // The final norm and the LM head (logits to `logits`, argmax through the LM-head ticket).
  void head(float* logits) {
    const dec_config& g = c->cfg;
    const int H = g.hidden;
    if (g.vocab) {
      OpDesc h = blank(OP_LMHEAD);
      h.wtype = g.lm_head_dtype == DEC_FP8_E4M3_ROWSCALE ? W_FP8 : W_BF16;
      h.N = g.vocab;
      h.K = H;
      h.norm = g.final_norm ? 1 : 0;
      h.gain = static_cast<const uint16_t*>(c->final_norm);
      h.w = c->lm_v;
      h.ws = c->lm_s;
      h.logits = logits;
      h.ticket = kLmHeadTicket;
      geom(h);
      ops.push_back(h);
    }
  }
};

// Kernel parameters of an op list of n_ops ops at byte offset ops_off of the workspace, built
// with the one-token geometry or the max_verify one.
void fill_params(dec_ctx* c, KParams& k, size_t ops_off, int n_ops, bool one_token) {
  const dec_config& g = c->cfg;
  const Layout& L = c->lay;
  const int M = g.max_verify, H = g.hidden, C = L.n_ctas;
  const int qkv_rows = g.n_q ? (g.n_q + 2 * g.n_kv) * kHeadDim : 0;
  std::memset(&k, 0, sizeof(k));
  k.ops = wsp<OpDesc>(c, ops_off);
  k.n_ops = n_ops;
  k.op_begin = 0;
  k.op_end = k.n_ops;
  k.n_ctas = C;
  k.H = H;
  k.n_q = g.n_q;
  k.n_kv = g.n_kv;
  k.G = g.n_q ? g.n_q / g.n_kv : 1;
  k.qkv_rows = qkv_rows;
  k.E = g.n_experts;
  k.top_k = g.top_k;
  k.I = g.moe_inter;
  k.n_shared = g.n_shared;
  k.V = g.vocab;
  k.cap = g.kv_capacity;
  k.Mmax = M;
  k.L = g.n_layers;
  k.ns_max = L.ns_max;
  k.eps = g.rms_eps;
  k.rope_base = g.rope_base;
  k.timeout_ns = g.spin_timeout_ns ? g.spin_timeout_ns : 2000000000ull;
  k.slot_bytes = one_token ? L.slot1_bytes : L.slot_bytes;
  k.act_bytes = one_token ? L.act1_bytes : L.act_bytes;
  k.kv_fp8 = g.kv_dtype == DEC_FP8_E4M3 ? 1 : 0;
  k.xpf_mode = c->xpf_mode;
  k.attn_tc = c->attn_tc && k.slot_bytes >= 4 * kAttnTcBoxBytes;  // a tile of keys and values fits a slot
  k.attn_window = g.attn_window;
  k.tmap_k = c->tmap_k;
  k.tmap_v = c->tmap_v;
  k.state = wsp<StepState>(c, L.state);
  k.status = wsp<Status>(c, L.status);
  k.tickets = wsp<uint32_t>(c, L.tickets);
  k.ctr = wsp<uint32_t>(c, L.ctr);
  k.part = wsp<uint64_t>(c, L.part);
  k.am_val = wsp<float>(c, L.am_val);
  k.am_idx = wsp<int32_t>(c, L.am_idx);
  k.am_out = wsp<int32_t>(c, L.am_out);
  k.step_ticket = kStepTicket;
  k.n_steps = 1;
  k.hs = wsp<uint64_t>(c, L.hs);
#ifdef DEC_TRACE
  k.trace = wsp<uint64_t>(c, L.trace);
#endif
}

// The whole step: every layer, then the LM head.
dec_status build_ops(dec_ctx* c) {
  const dec_config& g = c->cfg;
  c->ops.clear();
  // one-token calls (every call when max_verify is 1): the one-token geometry
  ListBuilder b(c, c->ops, g.embedding ? X_EMBED : X_HIDDEN_IN, true);
  for (int l = 0; l < g.n_layers; ++l) b.layer(l);
  if (g.vocab) b.head(wsp<float>(c, c->lay.logits));
  fill_params(c, c->kp, c->lay.ops, (int)c->ops.size(), true);
  // multi-token calls: the same step with the bf16 matrices on tensor-core tiles (one-token
  // calls keep the CUDA-core list above)
  c->wops.clear();
  c->tmaps_host.clear();
  if (g.max_verify > 1) {
    ListBuilder w(c, c->wops, g.embedding ? X_EMBED : X_HIDDEN_IN);
    w.window = true;
    for (int l = 0; l < g.n_layers; ++l) w.layer(l);
    if (g.vocab) w.head(wsp<float>(c, c->lay.logits));
    if (w.err != DEC_OK) return w.err;
    fill_params(c, c->wkp, c->lay.wops, (int)c->wops.size(), false);
  }
  return DEC_OK;
}

// Tensor maps of the bf16 key and value caches for tensor-core attention: each cache a 2D tensor
// of 128 bf16 columns by (n_layers n_kv kv_capacity) rows of 256 bytes, read in boxes of 64
// columns x kAttnTcRows rows with a 128-byte swizzle (the tensor-core tile's shared layout).
dec_status ensure_tmaps(dec_ctx* c) {
  const dec_config& g = c->cfg;
  // a tile of keys and values (four boxes) must fit a ring slot: large multi-token staging
  // areas leave smaller slots, and those contexts keep the CUDA-core attention tiles
  if (!attn_tc_for(&g) || std::max(c->lay.slot_bytes, c->lay.slot1_bytes) < 4 * kAttnTcBoxBytes) {
    c->attn_tc = 0;
    return DEC_OK;
  }
  if (c->attn_tc && c->tmap_kc == c->kc && c->tmap_vc == c->vc) return DEC_OK;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return fail(DEC_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)g.n_layers * g.n_kv * g.kv_capacity};
  const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kAttnTcRows};
  const cuuint32_t estr[2] = {1, 1};
  for (int which = 0; which < 2; ++which) {
    CUresult r = enc(which ? &c->tmap_v : &c->tmap_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, which ? c->vc : c->kc, dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DEC_ERR_CUDA, "encoding the KV cache tensor map failed (CUresult %d)", (int)r);
  }
  c->tmap_kc = c->kc;
  c->tmap_vc = c->vc;
  c->attn_tc = 1;
  return DEC_OK;
}

dec_status prepare(dec_ctx* c) {
  if (c->sticky) return fail(DEC_ERR_STATE, "a device error is pending (code %d): call dec_reset", (int)c->sticky_code);
  if (!c->ops_dirty) return DEC_OK;
  dec_status st = check_weights(c);
  if (st != DEC_OK) return st;
  st = ensure_tmaps(c);
  if (st != DEC_OK) return st;
  st = build_ops(c);
  if (st != DEC_OK) return st;
  CUDA_TRY(cudaMemcpyAsync(c->ws + c->lay.ops, c->ops.data(), c->ops.size() * sizeof(OpDesc), cudaMemcpyHostToDevice,
                           c->stream));
  if (!c->wops.empty()) {
    CUDA_TRY(cudaMemcpyAsync(c->ws + c->lay.wops, c->wops.data(), c->wops.size() * sizeof(OpDesc),
                             cudaMemcpyHostToDevice, c->stream));
    CUDA_TRY(cudaMemcpyAsync(c->ws + c->lay.tmaps, c->tmaps_host.data(), c->tmaps_host.size() * sizeof(CUtensorMap),
                             cudaMemcpyHostToDevice, c->stream));
  }
  CUDA_TRY(cudaStreamSynchronize(c->stream));
  if (c->graph) {
    cudaGraphExecDestroy(c->graph);
    c->graph = nullptr;
  }
  c->ops_dirty = false;
  return DEC_OK;
}

// Launch an op list in the context's mode. The CUDA graph of the per-op-graph mode holds the
// whole step's list; other lists (a layer or the LM head on its own) run as plain per-op launches
// in that mode. Persistent mode with n_steps > 1: n chained greedy steps in one launch.
dec_status launch_list(dec_ctx* c, const KParams& k0, bool whole_step, int n_steps = 1) {
  KParams k = k0;
  dec_mode mode = c->cfg.mode;
  if (mode == DEC_MODE_PER_OP_GRAPH && !whole_step) mode = DEC_MODE_PER_OP;
  if (mode == DEC_MODE_PERSISTENT) {
    k.n_steps = n_steps;
    CUDA_TRY(dec_launch_megakernel(&k, 1, c->stream));
    c->last_launches = 1;
    return DEC_OK;
  }
  if (mode == DEC_MODE_PER_OP_GRAPH) {
    if (!c->graph) {
      cudaGraph_t g;
      CUDA_TRY(cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
      cudaError_t err = cudaSuccess;
      for (int i = 0; i < k.n_ops && err == cudaSuccess; ++i) {
        KParams ki = k;
        ki.op_begin = i;
        ki.op_end = i + 1;
        err = dec_launch_megakernel(&ki, 0, c->stream);
      }
      cudaError_t e2 = cudaStreamEndCapture(c->stream, &g);
      if (err != cudaSuccess) return fail(DEC_ERR_CUDA, "graph capture launch: %s", cudaGetErrorString(err));
      if (e2 != cudaSuccess) return fail(DEC_ERR_CUDA, "graph capture: %s", cudaGetErrorString(e2));
      CUDA_TRY(cudaGraphInstantiate(&c->graph, g, 0));
      cudaGraphDestroy(g);
    }
    CUDA_TRY(cudaGraphLaunch(c->graph, c->stream));
    c->last_launches = k.n_ops;
    return DEC_OK;
  }
  const int drop = whole_step ? c->drop_op : -1;
  if (whole_step) c->drop_op = -1;
  int launched = 0;
  for (int i = 0; i < k.n_ops; ++i) {
    if (i == drop) continue;  // injected failure: this op's outputs are never written
    KParams ki = k;
    ki.op_begin = i;
    ki.op_end = i + 1;
    CUDA_TRY(dec_launch_megakernel(&ki, 0, c->stream));
    ++launched;
  }
  c->last_launches = launched;
  return DEC_OK;
}

// Host-written part of the step state (everything after `epoch`, which the device owns).
dec_status write_state(dec_ctx* c, int32_t pos, int m, const int32_t* tokens, const void* hidden, int chain,
                       int32_t* gen_out) {
  StepState s;
  std::memset(&s, 0, sizeof(s));
  s.pos = pos;
  s.m = m;
  s.chain = chain;
  for (int i = 0; i < m; ++i) s.tokens[i] = tokens ? tokens[i] : 0;
  s.hidden_in = hidden;
  s.gen_out = gen_out;
  s.gen_idx = 0;
  const size_t off = offsetof(StepState, pos);
  CUDA_TRY(cudaMemcpyAsync(c->ws + c->lay.state + off, reinterpret_cast<const uint8_t*>(&s) + off,
                           sizeof(StepState) - off, cudaMemcpyHostToDevice, c->stream));
  return DEC_OK;
}

dec_status read_status(dec_ctx* c) {
  Status s;
  CUDA_TRY(cudaMemcpyAsync(&s, c->ws + c->lay.status, sizeof(s), cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(cudaStreamSynchronize(c->stream));
  if (s.code != 0) {
    c->sticky = true;
    c->sticky_code = (dec_status)s.code;
    return fail((dec_status)s.code, "device wait timed out: op %d, cta %d, counter %u observed %u target %u (site %u)",
                s.op, s.cta, s.counter, s.observed, s.target, s.where);
  }
  return DEC_OK;
}

dec_status check_call(dec_ctx* c, int32_t pos, int m, const int32_t* tokens, const void* hidden) {
  const dec_config& g = c->cfg;
  if (m < 1 || m > g.max_verify) return fail(DEC_ERR_INVALID_ARG, "window of %d tokens (max_verify %d)", m, g.max_verify);
  if (pos < 0) return fail(DEC_ERR_INVALID_ARG, "negative position");
  if (g.n_q && (long long)pos + m > g.kv_capacity)
    return fail(DEC_ERR_CAPACITY, "positions %d..%d exceed kv_capacity %d", pos, pos + m - 1, g.kv_capacity);
  if (g.embedding) {
    if (!tokens) return fail(DEC_ERR_INVALID_ARG, "tokens required");
    for (int i = 0; i < m; ++i)
      if (tokens[i] < 0 || tokens[i] >= g.vocab) return fail(DEC_ERR_CAPACITY, "token %d outside the vocabulary", tokens[i]);
  } else if (g.n_layers > 0 || g.vocab) {
    if (!hidden) return fail(DEC_ERR_INVALID_ARG, "hidden_dev required (config without embedding)");
    if (reinterpret_cast<uintptr_t>(hidden) % 16) return fail(DEC_ERR_INVALID_ARG, "hidden_dev must be 16-byte aligned");
  }
  return DEC_OK;
}

dec_status run_call(dec_ctx* c, int32_t pos, int m, const int32_t* tokens, const void* hidden, float* logits_dev,
                    int32_t* argmax_host) {
  dec_status st = prepare(c);
  if (st != DEC_OK) return st;
  st = check_call(c, pos, m, tokens, hidden);
  if (st != DEC_OK) return st;
  st = write_state(c, pos, m, tokens, hidden, 0, nullptr);
  if (st != DEC_OK) return st;
  // several tokens: the multi-token list (bf16 matrices on the tensor cores)
  st = (m > 1 && !c->wops.empty()) ? launch_list(c, c->wkp, false) : launch_list(c, c->kp, true);
  if (st != DEC_OK) return st;
  if (logits_dev && c->cfg.vocab)
    CUDA_TRY(cudaMemcpyAsync(logits_dev, c->ws + c->lay.logits, (size_t)m * c->cfg.vocab * 4, cudaMemcpyDeviceToDevice,
                             c->stream));
  if (argmax_host) {
    CUDA_TRY(cudaMemcpyAsync(argmax_host, c->ws + c->lay.am_out, (size_t)m * 4, cudaMemcpyDeviceToHost, c->stream));
    return read_status(c);
  }
  return DEC_OK;
}

// Run an op list of its own (a layer or the LM head) from the given hidden vectors: the list
// goes to the workspace's second op region and runs in the context's mode. argmax_host
// (nullable) receives the list's argmaxes and makes the call wait and check the status word.
dec_status run_sub(dec_ctx* c, const std::vector<OpDesc>& ops, int32_t pos, int m, const void* hidden,
                   int32_t* argmax_host) {
  const bool one_token = m == 1;  // the builder chose the geometry the same way
  if ((int)ops.size() > kMaxSubOps) return fail(DEC_ERR_STATE, "%zu ops exceed the sub-list region", ops.size());
  CUDA_TRY(cudaMemcpyAsync(c->ws + c->lay.subops, ops.data(), ops.size() * sizeof(OpDesc), cudaMemcpyHostToDevice,
                           c->stream));
  KParams k;
  fill_params(c, k, c->lay.subops, (int)ops.size(), one_token);
  dec_status st = write_state(c, pos, m, nullptr, hidden, 0, nullptr);
  if (st != DEC_OK) return st;
  st = launch_list(c, k, false);
  if (st != DEC_OK) return st;
  if (argmax_host) {
    CUDA_TRY(cudaMemcpyAsync(argmax_host, c->ws + c->lay.am_out, (size_t)m * 4, cudaMemcpyDeviceToHost, c->stream));
    return read_status(c);
  }
  return DEC_OK;
}

bool aligned16(const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; }

}  // namespace

extern "C" {

const char* dec_last_error(void) { return g_last_error.c_str(); }

size_t dec_workspace_bytes(const dec_config* cfg) {
  std::string why;
  if (!validate(cfg, why)) {
    fail(DEC_ERR_INVALID_ARG, "invalid config: %s", why.c_str());
    return 0;
  }
  Layout L;
  if (!compute_layout(cfg, L, why)) {
    fail(DEC_ERR_SHAPE, "%s", why.c_str());
    return 0;
  }
  return L.total;
}

dec_status dec_init(const dec_config* cfg, void* cuda_stream, void* workspace_dev, dec_ctx** out) {
  if (!out) return fail(DEC_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  std::string why;
  if (!validate(cfg, why)) return fail(DEC_ERR_INVALID_ARG, "invalid config: %s", why.c_str());
  if (!workspace_dev) return fail(DEC_ERR_INVALID_ARG, "workspace is null");
  if (reinterpret_cast<uintptr_t>(workspace_dev) % 256) return fail(DEC_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  Layout L;
  if (!compute_layout(cfg, L, why)) return fail(DEC_ERR_SHAPE, "%s", why.c_str());
  dec_ctx* c = new dec_ctx();
  c->cfg = *cfg;
  c->stream = static_cast<cudaStream_t>(cuda_stream);
  c->ws = static_cast<uint8_t*>(workspace_dev);
  c->lay = L;
  c->layers.resize(cfg->n_layers);
  if (const char* v = std::getenv("DEC_EXPERT_PREFETCH")) {
    const int m = std::atoi(v);
    c->xpf_mode = m < 0 ? 0 : (m > 2 ? 2 : m);
  }
  cudaError_t e = cudaMemsetAsync(c->ws, 0, L.total, c->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) {
    delete c;
    return fail(DEC_ERR_CUDA, "clearing the workspace: %s", cudaGetErrorString(e));
  }
  *out = c;
  return DEC_OK;
}

dec_status dec_load_weights(dec_ctx* c, const dec_tensor* t, int n) {
  if (!c || (!t && n > 0) || n < 0) return fail(DEC_ERR_INVALID_ARG, "null context or tensors");
  const dec_config& g = c->cfg;
  const int H = g.hidden;
  for (int i = 0; i < n; ++i) {
    const dec_tensor& x = t[i];
    if (!x.values || reinterpret_cast<uintptr_t>(x.values) % 16)
      return fail(DEC_ERR_INVALID_ARG, "tensor %d: values null or not 16-byte aligned", i);
    const bool head = x.kind == DEC_T_EMBED || x.kind == DEC_T_FINAL_NORM || x.kind == DEC_T_LM_HEAD;
    if (!head && (x.layer < 0 || x.layer >= g.n_layers)) return fail(DEC_ERR_SHAPE, "tensor %d: layer %d", i, x.layer);
    auto want = [&](dec_dtype dt, int r, int cc) -> dec_status {
      if (x.dtype != dt) return fail(DEC_ERR_DTYPE, "tensor %d (kind %d): dtype %d, expected %d", i, x.kind, x.dtype, dt);
      if (x.rows != r || x.cols != cc)
        return fail(DEC_ERR_SHAPE, "tensor %d (kind %d): shape %dx%d, expected %dx%d", i, x.kind, x.rows, x.cols, r, cc);
      if (dt != DEC_BF16 && (!x.scales || reinterpret_cast<uintptr_t>(x.scales) % 16))
        return fail(DEC_ERR_INVALID_ARG, "tensor %d: scales null or not 16-byte aligned", i);
      return DEC_OK;
    };
    dec_status st = DEC_OK;
    LayerW* w = head ? nullptr : &c->layers[x.layer];
    const int qkv_rows = (g.n_q + 2 * g.n_kv) * kHeadDim;
    switch (x.kind) {
      case DEC_T_EMBED:
        if (!g.embedding) return fail(DEC_ERR_STATE, "config has no embedding");
        st = want(DEC_BF16, g.vocab, H);
        if (st == DEC_OK) c->embed = x.values;
        break;
      case DEC_T_ATTN_NORM:
      case DEC_T_FFN_NORM:
      case DEC_T_FINAL_NORM:
        if (x.rows * x.cols != H || x.dtype != DEC_BF16) return fail(DEC_ERR_SHAPE, "tensor %d: a norm gain is bf16 [H]", i);
        if (x.kind == DEC_T_ATTN_NORM) w->attn_norm = x.values;
        else if (x.kind == DEC_T_FFN_NORM) w->ffn_norm = x.values;
        else c->final_norm = x.values;
        break;
      case DEC_T_WQKV:
        if (!g.n_q) return fail(DEC_ERR_STATE, "config has no attention");
        st = want(DEC_BF16, qkv_rows, H);
        if (st == DEC_OK) w->wqkv = x.values;
        break;
      case DEC_T_WO:
        if (!g.n_q) return fail(DEC_ERR_STATE, "config has no attention");
        st = want(DEC_BF16, H, g.n_q * kHeadDim);
        if (st == DEC_OK) w->wo = x.values;
        break;
      case DEC_T_WGATEUP:
        if (!g.ffn) return fail(DEC_ERR_STATE, "config has no dense FFN");
        st = want(DEC_BF16, 2 * g.ffn, H);
        if (st == DEC_OK) w->wgateup = x.values;
        break;
      case DEC_T_WDOWN:
        if (!g.ffn) return fail(DEC_ERR_STATE, "config has no dense FFN");
        st = want(DEC_BF16, H, g.ffn);
        if (st == DEC_OK) w->wdown = x.values;
        break;
      case DEC_T_WROUTER:
        if (!g.n_experts) return fail(DEC_ERR_STATE, "config has no MoE");
        st = want(DEC_BF16, g.n_experts, H);
        if (st == DEC_OK) w->wrouter = x.values;
        break;
      case DEC_T_EXPERT_GATEUP:
        if (!g.n_experts) return fail(DEC_ERR_STATE, "config has no MoE");
        st = want(DEC_MXFP4, 2 * g.moe_inter, H);
        if (st == DEC_OK) { w->egu_v = x.values; w->egu_s = x.scales; }
        break;
      case DEC_T_EXPERT_DOWN:
        if (!g.n_experts) return fail(DEC_ERR_STATE, "config has no MoE");
        st = want(DEC_MXFP4, H, g.moe_inter);
        if (st == DEC_OK) { w->edn_v = x.values; w->edn_s = x.scales; }
        break;
      case DEC_T_LM_HEAD:
        if (!g.vocab) return fail(DEC_ERR_STATE, "config has no LM head");
        st = want(g.lm_head_dtype, g.vocab, H);
        if (st == DEC_OK) { c->lm_v = x.values; c->lm_s = x.scales; }
        break;
      default:
        return fail(DEC_ERR_INVALID_ARG, "tensor %d: unknown kind %d", i, (int)x.kind);
    }
    if (st != DEC_OK) return st;
  }
  c->ops_dirty = true;
  return DEC_OK;
}

dec_status dec_set_kv_cache(dec_ctx* c, void* k_dev, void* v_dev) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  if (!c->cfg.n_q) return fail(DEC_ERR_STATE, "config has no attention");
  if (!k_dev || !v_dev || reinterpret_cast<uintptr_t>(k_dev) % 256 || reinterpret_cast<uintptr_t>(v_dev) % 256)
    return fail(DEC_ERR_INVALID_ARG, "KV cache pointers must be non-null and 256-byte aligned");
  c->kc = static_cast<uint8_t*>(k_dev);
  c->vc = static_cast<uint8_t*>(v_dev);
  c->ops_dirty = true;
  return DEC_OK;
}

dec_status dec_set_kv_scales(dec_ctx* c, const float* scales_dev) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  if (!c->cfg.n_q || c->cfg.kv_dtype != DEC_FP8_E4M3) return fail(DEC_ERR_STATE, "config has no FP8 KV cache");
  if (scales_dev && reinterpret_cast<uintptr_t>(scales_dev) % 4)
    return fail(DEC_ERR_INVALID_ARG, "KV scales must be 4-byte aligned");
  c->kv_scales = scales_dev;
  c->ops_dirty = true;
  return DEC_OK;
}

dec_status dec_step(dec_ctx* c, int32_t token, const void* hidden_dev, int32_t pos, float* logits_dev,
                    int32_t* argmax_host) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  return run_call(c, pos, 1, &token, hidden_dev, logits_dev, argmax_host);
}

dec_status dec_verify(dec_ctx* c, const int32_t* tokens_host, const void* hidden_dev, int k, int32_t pos,
                      float* logits_dev, int32_t* argmax_host, int32_t* n_accepted) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  int32_t am[kMmax] = {0, 0, 0, 0};
  const bool need_am = argmax_host || n_accepted;
  dec_status st = run_call(c, pos, k, tokens_host, hidden_dev, logits_dev, need_am ? am : nullptr);
  if (st != DEC_OK) return st;
  if (argmax_host)
    for (int i = 0; i < k; ++i) argmax_host[i] = am[i];
  if (n_accepted) {
    int j = 0;
    while (tokens_host && j + 1 < k && tokens_host[j + 1] == am[j]) ++j;
    *n_accepted = j + 1;
  }
  return DEC_OK;
}

dec_status dec_run_layer(dec_ctx* c, int layer, const void* h_in, int m, int32_t pos, void* h_out,
                         int32_t* topk_idx_dev, float* topk_w_dev) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  const dec_config& g = c->cfg;
  if (c->sticky) return fail(DEC_ERR_STATE, "a device error is pending (code %d): call dec_reset", (int)c->sticky_code);
  if (layer < 0 || layer >= g.n_layers) return fail(DEC_ERR_SHAPE, "layer %d outside 0..%d", layer, g.n_layers - 1);
  if (m < 1 || m > g.max_verify) return fail(DEC_ERR_INVALID_ARG, "window of %d tokens (max_verify %d)", m, g.max_verify);
  if (!h_in || !aligned16(h_in) || !h_out || !aligned16(h_out))
    return fail(DEC_ERR_INVALID_ARG, "h_in and h_out must be non-null and 16-byte aligned");
  if ((topk_idx_dev || topk_w_dev) && !g.n_experts) return fail(DEC_ERR_STATE, "top-k outputs need a MoE layer");
  if (pos < 0) return fail(DEC_ERR_INVALID_ARG, "negative position");
  if (g.n_q && (long long)pos + m > g.kv_capacity)
    return fail(DEC_ERR_CAPACITY, "positions %d..%d exceed kv_capacity %d", pos, pos + m - 1, g.kv_capacity);
  dec_status st = check_layer(c, layer);
  if (st != DEC_OK) return st;
  st = ensure_tmaps(c);
  if (st != DEC_OK) return st;
  std::vector<OpDesc> ops;
  ListBuilder b(c, ops, X_HIDDEN_IN, m == 1);
  b.layer(layer);
  ops.back().y_bf16 = static_cast<uint16_t*>(h_out);  // the layer's last op writes its residual output
  for (OpDesc& o : ops)
    if (o.type == OP_ROUTER) {
      o.topk_idx_out = topk_idx_dev;
      o.topk_w_out = topk_w_dev;
    }
  return run_sub(c, ops, pos, m, h_in, nullptr);
}

dec_status dec_lm_head(dec_ctx* c, const void* h_in, int m, float* logits_dev, int32_t* argmax_host) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  const dec_config& g = c->cfg;
  if (c->sticky) return fail(DEC_ERR_STATE, "a device error is pending (code %d): call dec_reset", (int)c->sticky_code);
  if (!g.vocab) return fail(DEC_ERR_STATE, "config has no LM head");
  if (m < 1 || m > g.max_verify) return fail(DEC_ERR_INVALID_ARG, "window of %d tokens (max_verify %d)", m, g.max_verify);
  if (!h_in || !aligned16(h_in)) return fail(DEC_ERR_INVALID_ARG, "h_in must be non-null and 16-byte aligned");
  dec_status st = check_head(c);
  if (st != DEC_OK) return st;
  std::vector<OpDesc> ops;
  ListBuilder b(c, ops, X_HIDDEN_IN, m == 1);
  b.head(logits_dev ? logits_dev : wsp<float>(c, c->lay.logits));
  return run_sub(c, ops, 0, m, h_in, argmax_host);
}

dec_status dec_generate(dec_ctx* c, int32_t token, int32_t pos, int n, int32_t* tokens_dev) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  if (n < 0) return fail(DEC_ERR_INVALID_ARG, "negative step count");
  if (!c->cfg.embedding || !c->cfg.vocab) return fail(DEC_ERR_STATE, "chained generation needs an embedding and an LM head");
  dec_status st = prepare(c);
  if (st != DEC_OK) return st;
  if (n == 0) return DEC_OK;
  st = check_call(c, pos, 1, &token, nullptr);
  if (st != DEC_OK) return st;
  if (c->cfg.n_q && (long long)pos + n > c->cfg.kv_capacity)
    return fail(DEC_ERR_CAPACITY, "positions %d..%d exceed kv_capacity %d", pos, pos + n - 1, c->cfg.kv_capacity);
  st = write_state(c, pos, 1, &token, nullptr, 1, tokens_dev);
  if (st != DEC_OK) return st;
  if (c->cfg.mode == DEC_MODE_PERSISTENT) {
    // the whole chain in one launch: the kernel feeds each step's argmax to the next step
    return launch_list(c, c->kp, true, n);
  }
  int launches = 0;
  for (int i = 0; i < n; ++i) {
    st = launch_list(c, c->kp, true);
    if (st != DEC_OK) return st;
    launches += c->last_launches;
  }
  c->last_launches = launches;
  return DEC_OK;
}

dec_status dec_debug_buffers(dec_ctx* c, const uint64_t** hidden, const uint64_t** qkv, const int32_t** routing) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  if (hidden) *hidden = wsp<uint64_t>(c, c->lay.hs);
  if (qkv) *qkv = wsp<uint64_t>(c, c->lay.qkv);
  if (routing) *routing = reinterpret_cast<const int32_t*>(c->ws + c->lay.route);
  return DEC_OK;
}

dec_status dec_trace_buffer(dec_ctx* c, const uint64_t** records, int* n_ctas, int* n_ops) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
#ifdef DEC_TRACE
  if (records) *records = wsp<uint64_t>(c, c->lay.trace);
#else
  if (records) *records = nullptr;
#endif
  if (n_ctas) *n_ctas = c->lay.n_ctas;
  if (n_ops) *n_ops = c->lay.n_ops;
  return DEC_OK;
}

dec_status dec_reset(dec_ctx* c) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  // the whole workspace restarts from zero: tickets, status, the device-owned epoch, and every
  // tagged activation (their tags restart with the epoch, so no stale word may survive)
  CUDA_TRY(cudaStreamSynchronize(c->stream));
  CUDA_TRY(cudaMemsetAsync(c->ws, 0, c->lay.total, c->stream));
  CUDA_TRY(cudaStreamSynchronize(c->stream));
  c->ops_dirty = true;  // the op list lives in the workspace too
  c->sticky = false;
  c->sticky_code = DEC_OK;
  return DEC_OK;
}

dec_status dec_sync(dec_ctx* c) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  if (c->sticky) return fail(DEC_ERR_STATE, "a device error is pending (code %d): call dec_reset", (int)c->sticky_code);
  return read_status(c);
}

int dec_last_launch_count(dec_ctx* c) { return c ? c->last_launches : 0; }

dec_status dec_debug_drop_op(dec_ctx* c, int op) {
  if (!c) return fail(DEC_ERR_INVALID_ARG, "null context");
  if (c->cfg.mode != DEC_MODE_PER_OP) return fail(DEC_ERR_STATE, "ops can be dropped only in DEC_MODE_PER_OP");
  if (op < -1 || op >= count_ops(&c->cfg)) return fail(DEC_ERR_INVALID_ARG, "op %d outside the step's %d ops", op,
                                                       count_ops(&c->cfg));
  c->drop_op = op;
  return DEC_OK;
}

dec_status dec_lm_head_noalloc(int hidden, int vocab, dec_dtype dtype, int m, float rms_eps, const void* hidden_dev,
                               const void* final_norm_dev, const void* w_values_dev, const void* w_scales_dev,
                               float* logits_dev, int32_t* argmax_dev, void* cuda_stream) {
  auto misaligned = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 != 0; };
  if (hidden <= 0 || hidden % 64) return fail(DEC_ERR_SHAPE, "hidden must be a positive multiple of 64");
  if (vocab <= 0) return fail(DEC_ERR_SHAPE, "vocab must be positive");
  if (m < 1 || m > kMmax) return fail(DEC_ERR_SHAPE, "m must be 1..%d", kMmax);
  if (dtype != DEC_BF16 && dtype != DEC_FP8_E4M3_ROWSCALE)
    return fail(DEC_ERR_DTYPE, "dtype must be DEC_BF16 or DEC_FP8_E4M3_ROWSCALE");
  if (!std::isfinite(rms_eps) || rms_eps < 0) return fail(DEC_ERR_INVALID_ARG, "rms_eps must be >= 0");
  if (!hidden_dev || misaligned(hidden_dev)) return fail(DEC_ERR_INVALID_ARG, "hidden_dev null or not 16-byte aligned");
  if (!w_values_dev || misaligned(w_values_dev)) return fail(DEC_ERR_INVALID_ARG, "w_values_dev null or not 16-byte aligned");
  if (dtype == DEC_FP8_E4M3_ROWSCALE && (!w_scales_dev || misaligned(w_scales_dev)))
    return fail(DEC_ERR_INVALID_ARG, "w_scales_dev null or not 16-byte aligned");
  if (final_norm_dev && misaligned(final_norm_dev)) return fail(DEC_ERR_INVALID_ARG, "final_norm_dev not 16-byte aligned");
  if (!logits_dev || !argmax_dev) return fail(DEC_ERR_INVALID_ARG, "logits_dev and argmax_dev are required");

  int dev = 0, C = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&C, cudaDevAttrMultiProcessorCount, dev));
  // scratch: step state, status word, tickets, arrival counter, the op, per-CTA argmax partials
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t off_state = take(sizeof(StepState)), off_status = take(sizeof(Status)), off_tickets = take(2 * 4),
               off_ctr = take(4), off_op = take(sizeof(OpDesc)), off_val = take((size_t)C * kMmax * 4),
               off_idx = take((size_t)C * kMmax * 4);
  if (o > (size_t)kNoAllocScratchBytes)
    return fail(DEC_ERR_CAPACITY, "the allocation-free LM head needs %zu bytes of scratch for %d SMs; it has %d", o, C,
                kNoAllocScratchBytes);
  void* scratch_ptr = nullptr;
  CUDA_TRY(noalloc_scratch(&scratch_ptr));
  uint8_t* scratch = static_cast<uint8_t*>(scratch_ptr);

  // shared memory: the same sizing as a context holding only an LM head
  const int rows_cta = (hidden + C - 1) / C + 16;
  size_t act = std::max((size_t)m * hidden, (size_t)2 * kConsumerThreads);
  act = std::max(act, (size_t)m * hidden + (size_t)2 * (rows_cta + 1) * m * kConsumerWarps);
  act = align_up(act * 4, 256);
  long long slot = ((long long)kSmemLimit - (long long)act - dec_megakernel_common_bytes()) / (kConsumerWarps * kStages);
  slot = std::min<long long>(slot / 256 * 256, kMaxSlotBytes);
  if (slot < 4096) return fail(DEC_ERR_SHAPE, "hidden %d needs more shared memory than a CTA has", hidden);

  OpDesc h;
  std::memset(&h, 0, sizeof(h));
  h.type = OP_LMHEAD;
  h.wtype = dtype == DEC_FP8_E4M3_ROWSCALE ? W_FP8 : W_BF16;
  h.N = vocab;
  h.K = hidden;
  h.ticket = 0;
  h.ctr = 0;
  h.wait_ctr = -1;
  h.wait_n = C;
  h.aux_ctr = -1;
  h.norm = final_norm_dev ? 1 : 0;
  h.xsrc = X_HIDDEN_IN;
  h.slot1 = -1;
  h.gain = static_cast<const uint16_t*>(final_norm_dev);
  h.w = w_values_dev;
  h.ws = w_scales_dev;
  h.logits = logits_dev;
  tile_geometry(h.wtype, h.K, 0, (int)slot, m, h.R, h.Kc, h.unit);

  StepState st;
  std::memset(&st, 0, sizeof(st));
  st.m = m;
  st.hidden_in = hidden_dev;

  KParams k;
  std::memset(&k, 0, sizeof(k));
  k.ops = reinterpret_cast<const OpDesc*>(scratch + off_op);
  k.op_begin = 0;
  k.op_end = k.n_ops = 1;
  k.n_ctas = C;
  k.H = hidden;
  k.G = 1;
  k.V = vocab;
  k.Mmax = m;
  k.ns_max = 1;
  k.eps = rms_eps;
  k.timeout_ns = 2000000000ull;
  k.slot_bytes = (int)slot;
  k.act_bytes = (int)act;
  k.state = reinterpret_cast<StepState*>(scratch + off_state);
  k.status = reinterpret_cast<Status*>(scratch + off_status);
  k.tickets = reinterpret_cast<uint32_t*>(scratch + off_tickets);
  k.ctr = reinterpret_cast<uint32_t*>(scratch + off_ctr);
  k.am_val = reinterpret_cast<float*>(scratch + off_val);
  k.am_idx = reinterpret_cast<int32_t*>(scratch + off_idx);
  k.am_out = argmax_dev;
  k.step_ticket = 1;
  k.n_steps = 1;

  // the scratch keeps the previous call's contents: everything the kernel counts from starts at zero
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  CUDA_TRY(cudaMemsetAsync(scratch, 0, o, stream));
  CUDA_TRY(cudaMemcpyAsync(scratch + off_op, &h, sizeof(h), cudaMemcpyHostToDevice, stream));
  CUDA_TRY(cudaMemcpyAsync(scratch + off_state, &st, sizeof(st), cudaMemcpyHostToDevice, stream));
  CUDA_TRY(dec_launch_megakernel(&k, 1, stream));
  Status sw;
  CUDA_TRY(cudaMemcpyAsync(&sw, scratch + off_status, sizeof(sw), cudaMemcpyDeviceToHost, stream));
  CUDA_TRY(cudaStreamSynchronize(stream));
  if (sw.code != 0)
    return fail((dec_status)sw.code, "device wait timed out in the allocation-free LM head (cta %d, site %u)", sw.cta,
                sw.where);
  return DEC_OK;
}

static dec_status pack_device(dec_dtype dtype, const uint16_t* a, const uint16_t* b, int rows, int cols, void* vals,
                              void* scales, void* stream) {
  size_t vb = 0, sb = 0;
  const dec_status st = dec_packed_bytes(dtype, rows, cols, &vb, &sb);
  if (st != DEC_OK) return fail(st, "cannot pack dtype %d as a [%d][%d] matrix", (int)dtype, rows, cols);
  if (!a || !vals || (dtype != DEC_BF16 && !scales)) return fail(DEC_ERR_INVALID_ARG, "null device pointer");
  const auto misaligned = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) != 0; };
  if (misaligned(a, 16) || (b && misaligned(b, 16)) || misaligned(vals, 16) ||
      (dtype == DEC_FP8_E4M3_ROWSCALE && misaligned(scales, 4)))
    return fail(DEC_ERR_INVALID_ARG, "device packer: inputs and values must be 16-byte aligned (FP8 scales 4-byte)");
  CUDA_TRY(dec_launch_pack((int)dtype, a, b, rows, cols, vals, scales, static_cast<cudaStream_t>(stream)));
  return DEC_OK;
}

dec_status dec_pack_device(dec_dtype dtype, const uint16_t* bf16_dev, int rows, int cols, void* out_values,
                           void* out_scales, void* stream) {
  return pack_device(dtype, bf16_dev, nullptr, rows, cols, out_values, out_scales, stream);
}

dec_status dec_pack_pair_device(dec_dtype dtype, const uint16_t* a_dev, const uint16_t* b_dev, int rows, int cols,
                                void* out_values, void* out_scales, void* stream) {
  if (!b_dev) return fail(DEC_ERR_INVALID_ARG, "null device pointer");
  return pack_device(dtype, a_dev, b_dev, rows, cols, out_values, out_scales, stream);
}

dec_status dec_pack_kv_fp8_device(const uint16_t* v, size_t n, float scale, uint8_t* out, void* stream) {
  if (n && (!v || !out)) return fail(DEC_ERR_INVALID_ARG, "null device pointer");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(DEC_ERR_INVALID_ARG, "KV scale must be positive and finite");
  CUDA_TRY(dec_launch_pack_kv_fp8(v, n, scale, out, static_cast<cudaStream_t>(stream)));
  return DEC_OK;
}

void dec_free(dec_ctx* c) {
  if (!c) return;
  if (c->graph) cudaGraphExecDestroy(c->graph);
  delete c;
}

}  // extern "C"
