"""The whole decode step and the verify window, composed from ``ops``; fp64 throughout.

Test infrastructure only (see the package docstring).

One decode step of token ``x0`` at position ``pos`` (Muse Spark Open megakernel
article, "where the kernel boundary sits": a layer is attention over the KV
history plus this token's qkv projection and KV write; Ling-3.0-flash DGX Spark
article, "model and baseline configuration": MoE layers with 8 routed + 1
shared expert, LM head 2560 -> 157184):

    x <- x0
    for each layer:
        a = RMSNorm(x, g_attn);  [q; k; v] = W_qkv a;  q, k <- RoPE(q, k, pos)
        cache[pos] <- (bf16(k), bf16(v));  o = GQA-attention(q, cache[0..pos])
        x <- x + W_o o
        b = RMSNorm(x, g_ffn);  x <- x + FFN(b)      (dense SwiGLU or MoE)
    f = RMSNorm(x, g_final);  logits = W_lm f;  token = argmax(logits)

Weights enter as their stored values: bf16 exactly; an FP8 head as s_r * e4m3(q);
MXFP4 experts as e2m1(q) * 2^(e-127), each quantised here by ``formats``.
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from . import ops


def bf16_to_f64_fast(bits) -> np.ndarray:
    """bf16 codes -> fp64 by placing the 16 bits atop an fp32 word (bf16 is fp32's upper half).
    Exact; pinned against ``formats.bf16_to_f64`` over all 65536 codes."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class OracleModel:
    """fp64 decode of one model.

    shape      : synth.ModelShape (dims, eps, rope base, head dtype)
    layers     : list of dicts of logical bf16 weights per layer (``synth.model.layer_weights``)
    head       : dict with ``embed`` / ``final_norm`` / ``w_lm`` bf16 arrays (``head_weights``)
    experts    : callable (layer, expert) -> (gate, up, down) bf16, for MoE layers
    kv         : list of (K, V) bf16 prefilled caches [n_kv, n_prefill, d] per layer
    capacity   : positions the oracle's own cache can hold
    """

    def __init__(self, shape, layers, head, experts=None, kv=None, capacity=None, cache_weights=False,
                 kv_scales=None):
        self.s = shape
        self.layers = layers
        self.head = head
        self.experts_bf16 = experts
        self.cache_weights = cache_weights
        self._w = {}
        self._experts = {}
        self._lm = None
        cap = capacity if capacity is not None else shape.kv_prefill + 8
        # FP8 cache (shape.kv_dtype == "fp8"): e4m3 codes, fp32 scales [layer][K, V][kv head];
        # the engines' fallback scale 1.0 when none is given
        self.kv_fp8 = getattr(shape, "kv_dtype", "bf16") == "fp8"
        self.kv_scales = (np.ones((max(shape.n_layers, 1), 2, max(shape.n_kv, 1)), np.float32) if kv_scales is None
                          else np.asarray(kv_scales, np.float32))
        self.K, self.V = [], []
        if shape.attn:
            for l in range(shape.n_layers):
                K = np.zeros((shape.n_kv, cap, shape.head_dim), np.uint8 if self.kv_fp8 else np.uint16)
                V = np.zeros_like(K)
                if kv is not None:
                    n = kv[l][0].shape[1]
                    if self.kv_fp8:
                        # the prefilled bf16 history is stored quantised, like every new row
                        K[:, :n] = F.quantize_kv_fp8(bf16_to_f64_fast(kv[l][0]), self._kv_scale(l, 0, 3))
                        V[:, :n] = F.quantize_kv_fp8(bf16_to_f64_fast(kv[l][1]), self._kv_scale(l, 1, 3))
                    else:
                        K[:, :n] = kv[l][0]
                        V[:, :n] = kv[l][1]
                self.K.append(K)
                self.V.append(V)

    def _kv_scale(self, l, kv, ndim):
        """Scales of layer l's keys (kv = 0) or values (1), one per kv head, shaped to broadcast
        against an [n_kv, ...] array of ndim dimensions."""
        return self.kv_scales[l, kv].reshape((-1,) + (1,) * (ndim - 1))

    # ---------------------------------------------------------------- weights
    def w(self, l, name):
        key = (l, name)
        if key in self._w:
            return self._w[key]
        v = bf16_to_f64_fast(self.layers[l][name])
        if self.cache_weights:
            self._w[key] = v
        return v

    def expert(self, l, e):
        """fp64 (gate, up, down) of expert e in layer l as stored in MXFP4."""
        key = (l, e)
        if key in self._experts:
            return self._experts[key]
        g, u, d = self.experts_bf16(l, e)
        out = tuple(F.dequant_mxfp4(*F.quantize_mxfp4(m)) for m in (g, u, d))
        if self.cache_weights:
            self._experts[key] = out
        return out

    def lm_head(self):
        if self._lm is not None:
            return self._lm
        W = self.head["w_lm"]
        if self.s.lm_head_dtype == "fp8":
            W64 = F.dequant_fp8_rows(*F.quantize_fp8_rows(W))
        else:
            W64 = bf16_to_f64_fast(W)
        if self.cache_weights:
            self._lm = W64
        return W64

    # ---------------------------------------------------------------- blocks
    def attention_block(self, l, x, pos):
        s = self.s
        d = s.head_dim
        a = ops.rmsnorm(x, bf16_to_f64_fast(self.layers[l]["attn_norm"]), s.rms_eps)
        qkv = ops.gemv(self.w(l, "w_qkv"), a)
        q = qkv[: s.n_q * d].reshape(s.n_q, d)
        k = qkv[s.n_q * d:(s.n_q + s.n_kv) * d].reshape(s.n_kv, d)
        v = qkv[(s.n_q + s.n_kv) * d:].reshape(s.n_kv, d)
        q = ops.rope(q, pos, s.rope_base)
        k = ops.rope(k, pos, s.rope_base)
        # the cache holds bf16 (or FP8 codes): the new row is stored rounded, then read back (R4)
        # sliding-window attention (Muse Spark Open megakernel article: most of that model's layers
        # attend over the last 2,048 tokens only): the token at pos sees positions
        # pos - W + 1 .. pos; W = 0 is global attention over 0 .. pos
        W = getattr(s, "attn_window", 0)
        lo = max(0, pos - W + 1) if W > 0 else 0
        if self.kv_fp8:
            self.K[l][:, pos] = F.quantize_kv_fp8(k, self._kv_scale(l, 0, 2))
            self.V[l][:, pos] = F.quantize_kv_fp8(v, self._kv_scale(l, 1, 2))
            Kc = F.dequant_kv_fp8(self.K[l][:, lo: pos + 1], self._kv_scale(l, 0, 3))
            Vc = F.dequant_kv_fp8(self.V[l][:, lo: pos + 1], self._kv_scale(l, 1, 3))
        else:
            self.K[l][:, pos] = F.f64_to_bf16(k)
            self.V[l][:, pos] = F.f64_to_bf16(v)
            Kc = bf16_to_f64_fast(self.K[l][:, lo: pos + 1])
            Vc = bf16_to_f64_fast(self.V[l][:, lo: pos + 1])
        o = ops.attention(q, Kc, Vc)
        return x + ops.gemv(self.w(l, "w_o"), o.reshape(-1))

    def ffn_block(self, l, x, info):
        s = self.s
        b = ops.rmsnorm(x, bf16_to_f64_fast(self.layers[l]["ffn_norm"]), s.rms_eps)
        if s.moe:
            shared = [s.n_experts + i for i in range(s.n_shared)]
            y, S, pi = ops.moe_ffn(b, self.w(l, "w_router"), lambda e: self.expert(l, e), s.top_k, shared)
            info.setdefault("topk", []).append(S)
            info.setdefault("topk_w", []).append(pi)
            return x + y
        return x + ops.swiglu_ffn(b, self.w(l, "w_gate"), self.w(l, "w_up"), self.w(l, "w_down"))

    def logits(self, x):
        f = ops.rmsnorm(x, bf16_to_f64_fast(self.head["final_norm"]), self.s.rms_eps) if self.s.final_norm else x
        return ops.gemv(self.lm_head(), f)

    # ---------------------------------------------------------------- step
    def embed(self, token):
        return bf16_to_f64_fast(self.head["embed"][token])

    def step(self, x0, pos):
        """One decode step from hidden x0 (fp64) at position pos. Returns a dict with
        ``hidden`` (the residual stream after every block, fp64), ``logits``, ``token``,
        and for MoE layers ``topk`` / ``topk_w``."""
        s = self.s
        x = np.asarray(x0, np.float64)
        info = {"hidden": []}
        for l in range(s.n_layers):
            if s.attn:
                x = self.attention_block(l, x, pos)
                info["hidden"].append(x)
            if s.ffn or s.moe:
                x = self.ffn_block(l, x, info)
                info["hidden"].append(x)
        if s.vocab:
            lg = self.logits(x)
            info["logits"] = lg
            info["token"] = ops.argmax_first(lg)
        info["x_out"] = x
        return info

    def step_token(self, token, pos):
        return self.step(self.embed(token), pos)

    def verify(self, tokens, pos):
        """Verify window (Ling-3.0-flash DGX Spark article, "optimisation 3"): tokens[i] sits at
        pos+i and sees positions 0..pos+i. Evaluated as len(tokens) causal steps, which is the
        definition of one causal pass over the window. Returns (per-token infos, n_accepted)."""
        infos = [self.step_token(int(t), pos + i) for i, t in enumerate(tokens)]
        am = [inf["token"] for inf in infos]
        return infos, ops.accepted_prefix(list(tokens), am)

    def greedy(self, token, pos, n):
        """n greedy steps from ``token`` at ``pos``: returns the list of step infos."""
        out = []
        for i in range(n):
            inf = self.step_token(token, pos + i)
            out.append(inf)
            token = inf["token"]
        return out
