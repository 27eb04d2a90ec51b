/*
 * dec.h -- C ABI of the GB300 batch-1 decode step (persistent megakernel).
 *
 * What the library computes is one autoregressive decode step of a pre-norm
 * transformer at batch 1, or a verify window of up to 4 tokens:
 *   x <- E[token] (or a given hidden vector)
 *   per layer: a = RMSNorm(x); [q;k;v] = W_qkv a; RoPE(q, k, pos); cache[pos] <- bf16(k, v);
 *              o = GQA attention over cache[0..pos]; x += W_o o;
 *              b = RMSNorm(x); x += SwiGLU(b) (dense) or shared + top-k routed experts (MoE)
 *   logits = W_lm RMSNorm(x); token = argmax(logits)
 * Sources: batch-1 decode as matrix-vector weight streaming (Kog, "3k tokens/s
 * per request", section "what limits decode speed on GPUs"); one resident
 * kernel chaining the ops instead of one launch per op (Muse Spark Open
 * megakernel article, sections "the baseline nobody benchmarked" and "where
 * the kernel boundary sits"); MoE top-8 of 512 + 1 shared expert in MXFP4, a
 * dynamic FP8 LM head and a k-token verify window (Ling-3.0-flash on DGX Spark,
 * sections "model and baseline configuration", "optimisation 1/2/3").
 *
 * Conventions for every call:
 *   - No exception crosses the ABI: every call returns a dec_status; the text of
 *     the last error of the calling thread is dec_last_error().
 *   - Device memory is owned by the caller (weights, KV cache, workspace). The
 *     library keeps pointers, never frees them and allocates no device memory.
 *   - Work is ordered on the CUDA stream given to dec_init. A call synchronises
 *     the host only where it copies a result to a host pointer.
 *   - A device-side failure (a dependency wait that ran out of time) is sticky:
 *     later calls return DEC_ERR_STATE until dec_reset.
 *   - Matrices are logical [rows = out_features][cols = in_features], row-major.
 */
#ifndef DEC_H
#define DEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DEC_OK = 0,
  DEC_ERR_INVALID_ARG = 1, /* null pointer, misaligned pointer, bad enum */
  DEC_ERR_SHAPE = 2,       /* dimension not supported or inconsistent with the config */
  DEC_ERR_DTYPE = 3,       /* tensor dtype tag does not match the config */
  DEC_ERR_STATE = 4,       /* call out of order, missing weights, or sticky device error */
  DEC_ERR_CUDA = 5,        /* a CUDA runtime call failed */
  DEC_ERR_TIMEOUT = 6,     /* a device dependency wait ran out of time (sticky) */
  DEC_ERR_CAPACITY = 7,    /* pos + window exceeds the KV capacity, or token >= vocab */
} dec_status;

typedef enum {
  DEC_BF16 = 0,            /* bfloat16 values, 2 B per weight */
  DEC_FP8_E4M3_ROWSCALE = 1, /* e4m3fn codes, 1 B per weight, plus one fp32 scale per row */
  DEC_MXFP4 = 2,           /* e2m1 codes (2 per byte, even element low nibble) plus one
                              E8M0 scale byte per 32 consecutive weights of a row */
  DEC_FP8_E4M3 = 3,        /* KV cache: e4m3fn codes, 1 B per element, value = s * e4m3(q)
                              with one fp32 scale s per (layer, keys or values, kv head) */
} dec_dtype;

typedef enum {
  DEC_MODE_PERSISTENT = 0, /* one cooperative launch per step; ops chained through tagged data */
  DEC_MODE_PER_OP = 1,     /* the same kernel launched once per op (launch-per-op comparison) */
  DEC_MODE_PER_OP_GRAPH = 2, /* the per-op launches of one step replayed as a CUDA graph */
} dec_mode;

typedef struct {
  int n_layers;      /* decoder layers (0: LM head only) */
  int hidden;        /* H, multiple of 64 */
  int n_q, n_kv;     /* attention heads (n_q = 0: no attention block); n_q % n_kv == 0 */
  int head_dim;      /* must be 128 */
  int ffn;           /* dense SwiGLU width F (0: no dense FFN), multiple of 8 */
  int n_experts;     /* routed experts E (0: no MoE FFN) */
  int top_k;         /* routed experts per token, 1..8 */
  int moe_inter;     /* expert intermediate I, multiple of 32 */
  int n_shared;      /* shared experts (weight 1), 0..1 */
  int vocab;         /* V (0: no LM head) */
  int kv_capacity;   /* positions the KV cache holds */
  int max_verify;    /* largest window (tokens per call), 1..4. Above 1 the context keeps a
                        second op list for multi-token calls (bf16 matrices on the tensor
                        cores); one-token calls keep a list of their own, as fast
                        as in a max_verify = 1 context */
  int embedding;     /* 1: a step starts from E[token]; 0: from a given hidden vector */
  int final_norm;    /* 1: RMSNorm before the LM head */
  float rms_eps;     /* RMSNorm epsilon */
  float rope_base;   /* RoPE base (rotate-half pairing (i, i + d/2)) */
  dec_dtype lm_head_dtype; /* DEC_BF16 or DEC_FP8_E4M3_ROWSCALE */
  dec_dtype expert_dtype;  /* DEC_MXFP4 */
  dec_mode mode;
  uint64_t spin_timeout_ns; /* limit of every device wait (0: 2 s) */
  int num_ctas;      /* persistent CTAs (0: one per SM) */
  dec_dtype kv_dtype; /* KV cache: DEC_BF16 (0) or DEC_FP8_E4M3 */
  int attn_window;   /* 0: global attention; W > 0: the token at position p attends to positions
                        p - W + 1 .. p only (sliding-window attention, the Muse Spark Open megakernel
                        article, section "where the kernel boundary sits"), W >= max_verify */
} dec_config;

typedef struct dec_ctx dec_ctx;

/* Kinds of weight tensors passed to dec_load_weights. Packed layouts are the
   ones dec_pack / dec_pack_pair write. */
typedef enum {
  DEC_T_EMBED = 0,       /* [V][H] bf16 (embedding = 1 only) */
  DEC_T_ATTN_NORM = 1,   /* [H] bf16 gain */
  DEC_T_WQKV = 2,        /* [(n_q + 2 n_kv) d][H] bf16: q heads, then k heads, then v heads */
  DEC_T_WO = 3,          /* [H][n_q d] bf16 */
  DEC_T_FFN_NORM = 4,    /* [H] bf16 gain */
  DEC_T_WGATEUP = 5,     /* [2F][H] bf16, rows interleaved gate_0, up_0, gate_1, ... (dec_pack_pair) */
  DEC_T_WDOWN = 6,       /* [H][F] bf16 */
  DEC_T_WROUTER = 7,     /* [E][H] bf16 */
  DEC_T_EXPERT_GATEUP = 8, /* all experts of a layer: E + n_shared matrices [2I][H] MXFP4 pair-
                              interleaved; values contiguous per expert, scales contiguous per
                              expert; expert e >= E is shared expert e - E */
  DEC_T_EXPERT_DOWN = 9, /* all experts of a layer: E + n_shared matrices [H][I] MXFP4 */
  DEC_T_FINAL_NORM = 10, /* [H] bf16 gain */
  DEC_T_LM_HEAD = 11,    /* [V][H] bf16, or FP8 codes + fp32 row scales */
} dec_tensor_kind;

typedef struct {
  dec_tensor_kind kind;
  int layer;             /* layer index, 0 for head tensors */
  dec_dtype dtype;       /* tag checked against the config */
  int rows, cols;        /* logical shape of one matrix (per expert for expert tensors) */
  const void* values;    /* device pointer, 16-byte aligned */
  const void* scales;    /* device pointer of the scale plane (FP8, MXFP4), else NULL */
} dec_tensor;

/* Bytes of device workspace dec_init needs for this config (0 on an invalid config). */
size_t dec_workspace_bytes(const dec_config* cfg);

/* Validate cfg, bind the CUDA stream (cudaStream_t, NULL = legacy default) and the
   caller's workspace (dec_workspace_bytes long, 256-byte aligned, any contents: it is
   cleared here), and create a context on the current device. The environment variable
   DEC_EXPERT_PREFETCH, read here, sets the MoE expert prefetch (the Muse Spark Open
   megakernel article prefetches the experts the previous step routed to): while a layer's
   routing is pending, ask L2 for 0: nothing (the default), 1: the shared experts, plus the
   experts the layer's last routing chose when at least half of them had been chosen by the
   routing before it, 2: both, always. Results do not depend on it. */
dec_status dec_init(const dec_config* cfg, void* cuda_stream, void* workspace_dev, dec_ctx** out);

/* Register packed weight tensors (device pointers, caller-owned and kept alive until
   dec_free). Tags and shapes are checked against the config; may be called repeatedly. */
dec_status dec_load_weights(dec_ctx* ctx, const dec_tensor* tensors, int n);

/* Register the KV cache: k_dev and v_dev are [n_layers][n_kv][kv_capacity][head_dim], bf16, or
   e4m3fn codes (1 byte) when kv_dtype = DEC_FP8_E4M3; caller-owned device memory, each 256-byte
   aligned (DEC_ERR_INVALID_ARG otherwise). Positions below the step's pos must hold the cached
   (already rotated) keys and values; a step writes its own rows at pos.. before attending over
   them (the Muse Spark Open megakernel article, section "three bills": the layer's KV write
   comes before the attention that reads it; the Kimi-K3 8xB300 benchmark page reads the
   long-context cache this way). DEC_ERR_STATE for a config without attention. */
dec_status dec_set_kv_cache(dec_ctx* ctx, void* k_dev, void* v_dev);

/* Scales of an FP8 KV cache (kv_dtype = DEC_FP8_E4M3; the Kimi-K3 8xB300 benchmark, section on
   its log warnings: fp8_e4m3 caches whose scaling factor defaults to 1.0): scales_dev is fp32
   [n_layers][2][n_kv] on the device (index 0 keys, 1 values), caller-owned; NULL (the state
   after dec_init) makes every scale 1.0. A new key or value x is stored as
   e4m3fn(round-to-nearest-even of x / s in fp32, saturated to +-448). */
dec_status dec_set_kv_scales(dec_ctx* ctx, const float* scales_dev);

/* One decode step of `token` at position `pos` (embedding configs), or of the given hidden
   vector hidden_dev (bf16 [H], device, 16-byte aligned; non-embedding configs, token ignored):
   the whole step of the file header in one persistent launch (Kog, "3k tokens/s per
   request", section on the monokernel: embedding row, every layer, LM head and greedy argmax
   without returning to the host; Muse Spark Open megakernel article, "the baseline nobody
   benchmarked", for the launch count it removes).
   Writes the new key/value at pos. logits_dev (nullable, fp32 [V], device) receives the
   logits; argmax_host (nullable) receives the greedy token (lowest index among equal
   maxima) and makes the call wait and check the device status word.
   Errors: DEC_ERR_CAPACITY when pos >= kv_capacity or token >= vocab, DEC_ERR_INVALID_ARG on
   a missing or misaligned hidden_dev, DEC_ERR_STATE while a device error is pending. */
dec_status dec_step(dec_ctx* ctx, int32_t token, const void* hidden_dev, int32_t pos,
                    float* logits_dev, int32_t* argmax_host);

/* One decoder layer on its own, from and to bf16 hidden vectors (device memory the caller
   owns, 16-byte aligned): h_out[m][H] = layer `layer` applied to h_in[m][H] for the m tokens at
   positions pos .. pos + m - 1 (1 <= m <= max_verify), with the layer's own weights and KV cache
   slice (its rows at pos .. are written, as in a step). The layer runs exactly as inside a
   step (pre-norm attention block, then the dense SwiGLU or the MoE block of the file header;
   Kog, "3k tokens/s per request", for the decoder layer; Ling-3.0-flash on DGX Spark, "model
   and baseline configuration", for the MoE block); only its result is rounded to bf16 where it
   leaves the library. MoE layers: topk_idx_dev (nullable, int32 [m][top_k]) receives each
   token's routed experts, best first (lowest index among equal logits), and topk_w_dev
   (nullable, fp32 [m][top_k]) their weights, the softmax over the selected router logits.
   Ordered on the context's stream; does not wait. Errors: DEC_ERR_SHAPE for a layer outside
   the config, DEC_ERR_CAPACITY past kv_capacity, DEC_ERR_STATE for top-k outputs on a layer
   without MoE, missing weights or a pending device error, DEC_ERR_INVALID_ARG on null or
   misaligned hidden pointers. */
dec_status dec_run_layer(dec_ctx* ctx, int layer, const void* h_in, int m, int32_t pos, void* h_out,
                         int32_t* topk_idx_dev, float* topk_w_dev);

/* The final norm (when the config has one) and the LM head on their own, from given bf16
   hidden vectors h_in[m][H] (device, 16-byte aligned): logits_dev (nullable, fp32 [m][V],
   device; NULL keeps them in the workspace) and argmax_host (nullable, int32 [m], host: the
   greedy token of each row, lowest index among equal maxima; makes the call wait and check the
   device status word). Same kernel as a step's LM head: bf16, or FP8 e4m3 codes times a per-row
   scale (Ling-3.0-flash on DGX Spark, section "optimisation 2: online FP8 LM head").
   DEC_ERR_STATE for a config without an LM head. */
dec_status dec_lm_head(dec_ctx* ctx, const void* h_in, int m, float* logits_dev, int32_t* argmax_host);

/* n greedy steps chained on the device: step i feeds the argmax of step i-1 (the first one
   feeds `token`) at position pos + i. No host synchronisation between steps.
   tokens_dev (nullable, int32 [n], device) receives the n generated tokens. */
dec_status dec_generate(dec_ctx* ctx, int32_t token, int32_t pos, int n, int32_t* tokens_dev);

/* Verify window (Ling-3.0-flash on DGX Spark, section "optimisation 3": the MTP verify pass
   that scores the drafted tokens in one forward and keeps the correct prefix):
   tokens_host[i] (i < k <= max_verify) is fed at pos + i in one pass, each
   seeing positions 0..pos+i (causal inside the window); weights are streamed once for all k. logits_dev (nullable, fp32 [k][V]); argmax_host (nullable,
   [k]); n_accepted (nullable): the longest j with tokens[i+1] == argmax[i] for all i < j,
   plus one (the model's own next token). Non-embedding configs pass hidden_dev (bf16 [k][H])
   and tokens_host may be NULL. Keys/values of all k positions are written. */
dec_status dec_verify(dec_ctx* ctx, const int32_t* tokens_host, const void* hidden_dev, int k,
                      int32_t pos, float* logits_dev, int32_t* argmax_host, int32_t* n_accepted);

/* Device pointers of the activations the last call handed between SMs, as tagged 64-bit
   words: the fp32 value in the low 32 bits, the step's tag in the high 32 bits. hidden: the
   residual stream [2 n_layers + 1][max_verify][H] (entry 2l+1 after the attention block of
   layer l, entry 2l+2 after its FFN; entry 0 is unused, the input comes from the embedding
   or hidden_dev); qkv: the projections [n_layers][max_verify][qkv rows]; routing: one
   routing block per MoE layer, 920 bytes each, laid out as
     int32 n_slots;          n_shared + the distinct routed experts of the call (<= 33)
     int32 expert[33];       expert id per slot, shared experts first (id >= n_experts)
     float w[4][33];         weight of each slot for token m (1 for shared, pi or 0)
     int32 topk[4][8];       token m's routed experts, best first
     float topk_w[4][8];     their weights pi
   For inspection and tests; valid until the next call on the stream. */
dec_status dec_debug_buffers(dec_ctx* ctx, const uint64_t** hidden, const uint64_t** qkv,
                             const int32_t** routing);

/* Self-timing records of the last call (builds compiled with DEC_TRACE; *records is NULL
   otherwise): uint64 [n_ctas][n_ops][12] per (CTA, op): %globaltimer nanoseconds of consumer
   op start, input ready, prologue done, all warps' tiles done, op end; producer first issue,
   last issue, the count of tiles issued; first thread's input loads done, the count of input
   words re-read because their tag was not current yet, attention merge start, attention merge
   inputs ready. Zero the region between calls to read one call. */
dec_status dec_trace_buffer(dec_ctx* ctx, const uint64_t** records, int* n_ctas, int* n_ops);

/* Clear a sticky device error: zeroes the whole workspace (step counters, status word and
   every handed-over activation) after waiting for the stream. Weights and KV cache are kept.
   The bounded waits it recovers from are this library's own failure detection (the pages'
   kernels spin on flags without a limit; Muse Spark Open megakernel article, "three bills"). */
dec_status dec_reset(dec_ctx* ctx);

/* Wait for the context's stream; returns a sticky device error if one was raised. */
dec_status dec_sync(dec_ctx* ctx);

/* Failure injection for tests (host side only): the next call of a DEC_MODE_PER_OP context
   skips launching op `op` of the step (0-based, in list order; -1 cancels), so its outputs are
   never written. The op that reads them waits spin_timeout_ns, records the failure in the status
   word and raises the abort flag; every later wait of the step returns at once. The call
   returns DEC_ERR_TIMEOUT (sticky until dec_reset) and the GPU context stays usable.
   DEC_ERR_STATE in other modes; DEC_ERR_INVALID_ARG for an op outside the step. */
dec_status dec_debug_drop_op(dec_ctx* ctx, int op);

/* Number of kernel launches the last dec_step / dec_verify issued (1 in persistent mode). */
int dec_last_launch_count(dec_ctx* ctx);

/* LM head without any allocation, for callers that cannot allocate device memory: code that
   runs inside a memory pool or arena it does not own, or under an allocator it may not call
   (cudaMalloc / cudaFree can synchronise the device and fail inside some capture or
   callback contexts). The paper has no counterpart; it is this library's own addition.
   logits_dev[m][vocab] (fp32) = W_lm RMSNorm(hidden_dev[i]) (RMSNorm with final_norm_dev when
   it is non-NULL, eps rms_eps; plain hidden otherwise) and argmax_dev[m] (int32, lowest index
   among equal maxima), computed by the same kernel a context runs for its LM head.
   hidden_dev bf16 [m][hidden]; w_values_dev / w_scales_dev the dec_pack layout of dtype
   (DEC_BF16: scales unused, may be NULL; DEC_FP8_E4M3_ROWSCALE: fp32 row scales [vocab]).
   All pointers are device memory the caller owns; inputs and weights 16-byte aligned.
   Its scratch (step state, argmax partials, status) is a static device array of 64 KiB in
   the library, which every GPU that loads the library keeps until the process exits; a call
   needs about 256 * 5 + 32 * (SM count) bytes of it and returns DEC_ERR_CAPACITY beyond that.
   The first call on a device looks up the array's device address. The call synchronises the
   stream it is given (it waits for the result), so it must not be issued on a stream that is
   being captured. Every call clears and reuses the same array: calls that overlap on the GPU
   (other streams, other threads) race, so serialise them. Returns a device error if the
   kernel raised one.
   m: 1..4; hidden a multiple of 64. */
dec_status dec_lm_head_noalloc(int hidden, int vocab, dec_dtype dtype, int m, float rms_eps, const void* hidden_dev,
                               const void* final_norm_dev, const void* w_values_dev, const void* w_scales_dev,
                               float* logits_dev, int32_t* argmax_dev, void* cuda_stream);

/* Text of the last error raised on the calling thread ("" if none). */
const char* dec_last_error(void);

void dec_free(dec_ctx* ctx);

/* ---------------------------------------------------------------- packer (host)
   Quantise / lay out one logical bf16 matrix [rows][cols] (host memory) into the packed
   layout the kernels stream. Sizes: dec_packed_bytes. Rules:
   - DEC_BF16: values copied as is.
   - DEC_FP8_E4M3_ROWSCALE (Ling-3.0-flash DGX Spark article, "optimisation 2: online FP8 LM
     head"): per row s = amax / 448 in IEEE fp32 (zero row: s = 1), code =
     e4m3fn(round-to-nearest-even of w / s, fp32 division), saturated to +-448.
   - DEC_MXFP4 (OCP MX v1.0): per 32 weights along a row, E8M0 e = floor(log2 amax) - 2 + 127
     clamped to [0, 254] (all-zero block: e = 0); code = e2m1(round-to-nearest-even of
     w / 2^(e-127)) saturated to +-6, sign bit = sign of w; values plane [rows][cols/2]
     then scales plane [rows][cols/32].
   out_scales may be NULL for DEC_BF16. */
dec_status dec_packed_bytes(dec_dtype dtype, int rows, int cols, size_t* values_bytes,
                            size_t* scales_bytes);
dec_status dec_pack(dec_dtype dtype, const uint16_t* bf16_host, int rows, int cols,
                    void* out_values, void* out_scales);
/* Interleave two [rows][cols] matrices row by row (a_0, b_0, a_1, b_1, ...) into a packed
   [2 rows][cols] matrix: the gate/up layout of DEC_T_WGATEUP and DEC_T_EXPERT_GATEUP. */
dec_status dec_pack_pair(dec_dtype dtype, const uint16_t* a_host, const uint16_t* b_host, int rows,
                         int cols, void* out_values, void* out_scales);

/* ---------------------------------------------------------------- packer (device)
   dec_pack / dec_pack_pair on device memory, for weights too large to stage through the host
   (the MoE stack holds 67 GB of MXFP4 experts). Same rules and the same bytes as the host
   packer: both run one set of encoders. bf16_dev (a_dev, b_dev): bf16 [rows][cols] on the
   device; out_values / out_scales: device buffers of dec_packed_bytes. Inputs and out_values
   16-byte aligned, FP8 out_scales 4-byte aligned (DEC_ERR_INVALID_ARG otherwise). The kernel is queued on `stream` (a cudaStream_t; NULL:
   the legacy default stream) and the call returns without waiting; launch errors come back as
   DEC_ERR_CUDA. The packer has no counterpart in the pages beyond the formats it writes. */
dec_status dec_pack_device(dec_dtype dtype, const uint16_t* bf16_dev, int rows, int cols,
                           void* out_values, void* out_scales, void* stream);
dec_status dec_pack_pair_device(dec_dtype dtype, const uint16_t* a_dev, const uint16_t* b_dev,
                                int rows, int cols, void* out_values, void* out_scales,
                                void* stream);

/* FP8 KV-cache entries from bf16 values: out[i] = e4m3fn(RNE of v[i] / scale in fp32, saturated
   to +-448), the rule the kernel applies to new rows; n elements, host or device memory. The
   device form is queued on `stream` and returns without waiting. */
dec_status dec_pack_kv_fp8(const uint16_t* bf16_host, size_t n, float scale, uint8_t* out_host);
dec_status dec_pack_kv_fp8_device(const uint16_t* bf16_dev, size_t n, float scale, uint8_t* out_dev,
                                  void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DEC_H */
