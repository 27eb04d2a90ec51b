"""Load a model into the library: pack weights, place them in device memory, register them.

PyTorch is used for device memory and the stream only; every step of the decode runs in the
library's kernels. Weights arrive as logical bfloat16 bits (numpy ``uint16``, matrices
[out_features, in_features]); packing follows ``dec_pack`` / ``dec_pack_pair``.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import binding as B

_DTYPE = {"bf16": B.DEC_BF16, "fp8": B.DEC_FP8_E4M3_ROWSCALE, "mxfp4": B.DEC_MXFP4}
_MODE = {"persistent": B.DEC_MODE_PERSISTENT, "per_op": B.DEC_MODE_PER_OP, "graph": B.DEC_MODE_PER_OP_GRAPH}


def make_config(shape, capacity: int, max_verify: int = 1, mode: str = "persistent", num_ctas: int = 0,
                timeout_ns: int = 0) -> B.DecConfig:
    c = B.DecConfig()
    c.n_layers = shape.n_layers
    c.hidden = shape.hidden
    c.n_q = shape.n_q
    c.n_kv = shape.n_kv
    c.head_dim = shape.head_dim
    c.ffn = shape.ffn
    c.n_experts = shape.n_experts
    c.top_k = shape.top_k
    c.moe_inter = shape.moe_inter
    c.n_shared = shape.n_shared
    c.vocab = shape.vocab
    c.kv_capacity = capacity
    c.max_verify = max_verify
    c.embedding = 1 if shape.embedding else 0
    c.final_norm = 1 if shape.final_norm else 0
    c.rms_eps = shape.rms_eps
    c.rope_base = shape.rope_base
    c.lm_head_dtype = _DTYPE[shape.lm_head_dtype]
    c.expert_dtype = B.DEC_MXFP4
    c.mode = _MODE[mode]
    c.spin_timeout_ns = timeout_ns
    c.num_ctas = num_ctas
    c.attn_window = getattr(shape, "attn_window", 0)
    c.kv_dtype = B.DEC_FP8_E4M3 if getattr(shape, "kv_dtype", "bf16") == "fp8" else B.DEC_BF16
    return c


def _dev(a: np.ndarray, device) -> torch.Tensor:
    """numpy array -> device tensor with the same bytes (uint16 bits travel as int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def pack_host(dtype: int, w: np.ndarray, pair_with: np.ndarray | None = None):
    """Pack one logical bf16 matrix (or two, interleaved row by row) on the host."""
    rows, cols = w.shape
    out_rows = rows * (2 if pair_with is not None else 1)
    vb, sb = B.dec_packed_bytes(dtype, out_rows, cols)
    vals = np.empty(vb, np.uint8)
    scales = np.empty(max(sb, 1), np.uint8)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    if pair_with is None:
        B.dec_pack(dtype, w, rows, cols, vals, scales if sb else None)
    else:
        B.dec_pack_pair(dtype, w, np.ascontiguousarray(pair_with, dtype=np.uint16), rows, cols, vals,
                        scales if sb else None)
    return vals, (scales[:sb] if sb else None)


def pack_device(dtype: int, w: torch.Tensor, pair_with: torch.Tensor | None = None):
    """Pack one logical bf16 matrix held on the device (2-byte elements, [rows, cols]), or two
    interleaved row by row, with the library's device packer on the current stream."""
    rows, cols = w.shape
    out_rows = rows * (2 if pair_with is not None else 1)
    vb, sb = B.dec_packed_bytes(dtype, out_rows, cols)
    vals = torch.empty(vb, dtype=torch.uint8, device=w.device)
    scales = torch.empty(max(sb, 1), dtype=torch.uint8, device=w.device) if sb else None
    stream = torch.cuda.current_stream(w.device).cuda_stream
    if pair_with is None:
        B.dec_pack_device(dtype, w, rows, cols, vals, scales, stream)
    else:
        B.dec_pack_pair_device(dtype, w, pair_with, rows, cols, vals, scales, stream)
    return vals, scales


def pack_kv_host(x: np.ndarray, head_scales: np.ndarray) -> np.ndarray:
    """e4m3 codes of a bf16 cache block [n_kv, n, d] (numpy uint16), head g under head_scales[g]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    out = np.empty(x.shape, np.uint8)
    for g in range(x.shape[0]):
        B.dec_pack_kv_fp8(x[g], x[g].size, float(head_scales[g]), out[g])
    return out


class Decoder:
    """One model instance on one GPU: workspace, packed weights, KV cache, context.

    shape      : a ModelShape (dims, eps, RoPE base, head dtype, embedding)
    layers     : per-layer dicts of logical bf16 weights (attn_norm, w_qkv, w_o, ffn_norm,
                 w_gate, w_up, w_down, w_router): numpy uint16 arrays (packed on the host) or
                 2-byte device tensors (packed on the device)
    head       : dict with embed / final_norm / w_lm
    experts    : callable (layer, expert) -> (gate, up, down) bf16 for MoE layers; experts
                 shape.n_experts .. + n_shared - 1 are the shared ones
    kv         : list of (K, V) bf16 prefills [n_kv, n, d] per layer, or None (the caller may
                 fill ``k_cache`` / ``v_cache`` itself before the first step); an FP8 cache
                 (shape.kv_dtype == "fp8") stores them as e4m3 codes
    kv_scales  : FP8 cache scales [n_layers, 2 (keys, values), n_kv] (None: all 1.0)
    packed_experts : instead of ``experts``, callable layer -> (gate/up values, gate/up scales,
                 down values, down scales), the MXFP4 planes of all the layer's experts already
                 packed (host arrays or device tensors)
    """

    def __init__(self, shape, layers, head, experts=None, kv=None, capacity=None, max_verify=1, mode="persistent",
                 num_ctas=0, timeout_ns=0, device="cuda:0", packed_experts=None, kv_scales=None):
        self.shape = shape
        self.device = torch.device(device)
        # a stream of its own: CUDA-graph capture cannot use the legacy default stream
        self.stream = torch.cuda.Stream(self.device)
        self.capacity = capacity if capacity is not None else max(1, shape.kv_prefill + 8)
        self.max_verify = max_verify
        self.cfg = make_config(shape, self.capacity, max_verify, mode, num_ctas, timeout_ns)
        nbytes = B.dec_workspace_bytes(self.cfg)
        if nbytes == 0:
            raise B.DecError(B.DEC_ERR_INVALID_ARG, B.dec_last_error())
        self.workspace = torch.zeros(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.workspace.data_ptr()) % 256
        self.ws = self.workspace[off:off + nbytes]
        torch.cuda.synchronize(self.device)
        self.ctx = B.dec_init(self.cfg, self.stream.cuda_stream, self.ws)
        self._keep = []
        tensors = []

        def reg(kind, layer, dtype, rows, cols, vals, scales=None):
            v = vals if isinstance(vals, torch.Tensor) else _dev(vals, self.device)
            s = None if scales is None else (scales if isinstance(scales, torch.Tensor) else _dev(scales, self.device))
            self._keep += [v, s]
            tensors.append(B.DecTensor(kind, layer, dtype, rows, cols, v.data_ptr(),
                                       s.data_ptr() if s is not None else None))

        s = shape
        H = s.hidden
        for l, w in enumerate(layers):
            if s.attn:
                reg(B.DEC_T_ATTN_NORM, l, B.DEC_BF16, H, 1, w["attn_norm"])
                reg(B.DEC_T_WQKV, l, B.DEC_BF16, s.qkv_rows, H, w["w_qkv"])
                reg(B.DEC_T_WO, l, B.DEC_BF16, H, s.n_q * s.head_dim, w["w_o"])
            if s.ffn or s.moe:
                reg(B.DEC_T_FFN_NORM, l, B.DEC_BF16, H, 1, w["ffn_norm"])
            if s.ffn:
                pack = pack_device if isinstance(w["w_gate"], torch.Tensor) else pack_host
                vals, _ = pack(B.DEC_BF16, w["w_gate"], w["w_up"])
                reg(B.DEC_T_WGATEUP, l, B.DEC_BF16, 2 * s.ffn, H, vals)
                reg(B.DEC_T_WDOWN, l, B.DEC_BF16, H, s.ffn, w["w_down"])
            if s.moe:
                reg(B.DEC_T_WROUTER, l, B.DEC_BF16, s.n_experts, H, w["w_router"])
                if packed_experts is not None:
                    gu_v, gu_s, dn_v, dn_s = packed_experts(l)
                else:
                    gu_v, gu_s, dn_v, dn_s = self._pack_experts(experts, l)
                reg(B.DEC_T_EXPERT_GATEUP, l, B.DEC_MXFP4, 2 * s.moe_inter, H, gu_v, gu_s)
                reg(B.DEC_T_EXPERT_DOWN, l, B.DEC_MXFP4, H, s.moe_inter, dn_v, dn_s)
        if s.embedding:
            reg(B.DEC_T_EMBED, 0, B.DEC_BF16, s.vocab, H, head["embed"])
        if s.vocab:
            if s.final_norm:
                reg(B.DEC_T_FINAL_NORM, 0, B.DEC_BF16, H, 1, head["final_norm"])
            if s.lm_head_dtype == "fp8":
                pack = pack_device if isinstance(head["w_lm"], torch.Tensor) else pack_host
                vals, scales = pack(B.DEC_FP8_E4M3_ROWSCALE, head["w_lm"])
                reg(B.DEC_T_LM_HEAD, 0, B.DEC_FP8_E4M3_ROWSCALE, s.vocab, H, vals, scales)
            else:
                reg(B.DEC_T_LM_HEAD, 0, B.DEC_BF16, s.vocab, H, head["w_lm"])
        B.dec_load_weights(self.ctx, tensors)
        self._tensors = tensors

        self.kv_fp8 = getattr(s, "kv_dtype", "bf16") == "fp8"
        self.kv_scales = None
        if s.attn:
            dt = torch.uint8 if self.kv_fp8 else torch.int16
            self.k_cache = torch.zeros((s.n_layers, s.n_kv, self.capacity, s.head_dim), dtype=dt, device=self.device)
            self.v_cache = torch.zeros_like(self.k_cache)
            sc = (np.ones((s.n_layers, 2, s.n_kv), np.float32) if kv_scales is None
                  else np.ascontiguousarray(kv_scales, np.float32))
            if kv is not None:
                for l, (k, v) in enumerate(kv):
                    n = k.shape[1]
                    if self.kv_fp8:
                        # the prefilled bf16 history is stored as e4m3 codes under each head's scale
                        k, v = pack_kv_host(k, sc[l, 0]), pack_kv_host(v, sc[l, 1])
                    self.k_cache[l, :, :n] = _dev(k, self.device)
                    self.v_cache[l, :, :n] = _dev(v, self.device)
            B.dec_set_kv_cache(self.ctx, self.k_cache, self.v_cache)
            if self.kv_fp8:
                self.kv_scales = torch.from_numpy(sc).to(self.device)
                B.dec_set_kv_scales(self.ctx, self.kv_scales)
        torch.cuda.synchronize(self.device)
        self.logits = torch.empty((max_verify, max(s.vocab, 1)), dtype=torch.float32, device=self.device)

    def context(self, mode: str):
        """Another context over the same packed weights and KV cache (e.g. another launch mode).
        Returns (ctx, workspace); the caller frees ctx with binding.dec_free."""
        cfg = make_config(self.shape, self.capacity, self.max_verify, mode, self.cfg.num_ctas, self.cfg.spin_timeout_ns)
        nbytes = B.dec_workspace_bytes(cfg)
        ws_all = torch.zeros(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-ws_all.data_ptr()) % 256
        torch.cuda.synchronize(self.device)
        ctx = B.dec_init(cfg, self.stream.cuda_stream, ws_all[off:off + nbytes])
        B.dec_load_weights(ctx, self._tensors)
        if self.shape.attn:
            B.dec_set_kv_cache(ctx, self.k_cache, self.v_cache)
            if self.kv_scales is not None:
                B.dec_set_kv_scales(ctx, self.kv_scales)
        return ctx, ws_all

    def _pack_experts(self, experts, l):
        s = self.shape
        n = s.n_experts + s.n_shared
        H, I = s.hidden, s.moe_inter
        gu_v = np.empty((n, 2 * I * H // 2), np.uint8)
        gu_s = np.empty((n, 2 * I * H // 32), np.uint8)
        dn_v = np.empty((n, H * I // 2), np.uint8)
        dn_s = np.empty((n, H * I // 32), np.uint8)
        for e in range(n):
            g, u, d = experts(l, e)
            B.dec_pack_pair(B.DEC_MXFP4, np.ascontiguousarray(g), np.ascontiguousarray(u), I, H, gu_v[e], gu_s[e])
            B.dec_pack(B.DEC_MXFP4, np.ascontiguousarray(d), H, I, dn_v[e], dn_s[e])
        return gu_v, gu_s, dn_v, dn_s

    # ------------------------------------------------------------------ calls
    def _order(self):
        # inputs written on the caller's stream must land before the library's stream reads them
        self.stream.wait_stream(torch.cuda.current_stream(self.device))

    def step(self, token: int = 0, pos: int = 0, hidden: torch.Tensor | None = None, logits: bool = True) -> int:
        self._order()
        return B.dec_step(self.ctx, token, hidden, pos, self.logits if logits else None)

    def verify(self, tokens, pos: int, hidden: torch.Tensor | None = None, k: int | None = None):
        self._order()
        k = k if k is not None else len(tokens)
        return B.dec_verify(self.ctx, tokens, hidden, k, pos, self.logits)

    def run_layer(self, layer: int, h_in: torch.Tensor, pos: int, topk: bool = False):
        """One decoder layer on its own: bf16 [m, H] in (2-byte elements on the device), bf16
        [m, H] out; with topk (MoE layers) also the [m, top_k] expert ids and weights."""
        m = h_in.shape[0]
        h_out = torch.empty_like(h_in)
        s = self.shape
        idx = torch.empty((m, s.top_k), dtype=torch.int32, device=self.device) if topk else None
        w = torch.empty((m, s.top_k), dtype=torch.float32, device=self.device) if topk else None
        self._order()
        B.dec_run_layer(self.ctx, layer, h_in, m, pos, h_out, idx, w)
        torch.cuda.current_stream(self.device).wait_stream(self.stream)
        return (h_out, idx, w) if topk else h_out

    def lm_head(self, h_in: torch.Tensor):
        """The final norm and LM head on their own: logits into ``self.logits[:m]``; returns the
        m argmaxes."""
        self._order()
        return B.dec_lm_head(self.ctx, h_in, h_in.shape[0], self.logits)

    def generate(self, token: int, pos: int, n: int, out: torch.Tensor | None = None) -> torch.Tensor:
        out = out if out is not None else torch.empty(n, dtype=torch.int32, device=self.device)
        self._order()
        B.dec_generate(self.ctx, token, pos, n, out)
        return out

    def sync(self):
        B.dec_sync(self.ctx)
        torch.cuda.current_stream(self.device).wait_stream(self.stream)

    def reset(self):
        B.dec_reset(self.ctx)

    def launches(self) -> int:
        return B.dec_last_launch_count(self.ctx)

    def hidden_stream(self) -> torch.Tensor:
        """fp32 [2L + 1, max_verify, H] copy of the residual stream of the last call (the low
        halves of its tagged words)."""
        h, _, _ = B.dec_debug_buffers(self.ctx)
        s = self.shape
        n = (2 * s.n_layers + 1) * self.max_verify * s.hidden
        off = h - self.ws.data_ptr()
        words = self.ws[off:off + 8 * n].view(torch.float32).view(n, 2)
        return words[:, 0].contiguous().view(2 * s.n_layers + 1, self.max_verify, s.hidden)

    # routing block of dec_debug_buffers (include/dec.h): int32 n_slots, int32 expert[33],
    # float w[4][33], int32 topk[4][8], float topk_w[4][8]
    ROUTE_SLOTS, ROUTE_TOKENS, ROUTE_K = 33, 4, 8
    ROUTE_WORDS = 1 + ROUTE_SLOTS + ROUTE_TOKENS * ROUTE_SLOTS + 2 * ROUTE_TOKENS * ROUTE_K

    def routing(self, layer: int) -> dict:
        """Routing block of a MoE layer after the last call (slots, per-token top-k)."""
        _, _, r = B.dec_debug_buffers(self.ctx)
        off = r - self.ws.data_ptr()
        S, T, K = self.ROUTE_SLOTS, self.ROUTE_TOKENS, self.ROUTE_K
        sz = 4 * self.ROUTE_WORDS
        raw = self.ws[off + layer * sz: off + (layer + 1) * sz].cpu().numpy()
        i32 = raw.view(np.int32)
        f32 = raw.view(np.float32)
        n = int(i32[0])
        w0 = 1 + S                      # float w[T][S]
        t0 = w0 + T * S                 # int32 topk[T][K]
        tw0 = t0 + T * K                # float topk_w[T][K]
        return {"n_slots": n, "expert": i32[1:1 + n].tolist(),
                "w": f32[w0:t0].reshape(T, S)[:, :n],
                "topk": i32[t0:tw0].reshape(T, K),
                "topk_w": f32[tw0:tw0 + T * K].reshape(T, K)}

    def close(self):
        if self.ctx:
            B.dec_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
