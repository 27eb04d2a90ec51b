"""Roofline arithmetic of batch-1 decode.

First-order bound (Kog, "3k tokens/s per request", section "what limits decode
speed on GPUs"): every active weight and the KV cache cross HBM once per token,
so tokens/s <= bandwidth / (beta * active_weight_bytes + kv_bytes), with
beta >= 1 counting re-loaded tiles. Launch overhead model (same post, section
"where standard inference stacks lose microseconds"): per-token overhead =
launch cost x kernels per layer x layers.

``algorithmic_bytes`` is the per-token byte count of this library's path for
a model shape: bf16 weights 2 B per parameter, FP8-e4m3 rows 1 B per parameter
plus a 4-byte scale per row, MXFP4 17 B per 32 parameters (16 B of e2m1 codes
+ 1 E8M0 scale), plus the KV rows read (2 B per element, keys and values).
"""
from __future__ import annotations


def bound_tokens_per_s(bw_bytes_per_s: float, weight_bytes: float, kv_bytes: float = 0.0, beta: float = 1.0) -> float:
    return bw_bytes_per_s / (beta * weight_bytes + kv_bytes)


def launch_overhead_us(launch_us: float, kernels_per_layer: float, layers: int) -> float:
    return launch_us * kernels_per_layer * layers


def ceiling_tokens_per_s(overhead_us: float) -> float:
    return 1e6 / overhead_us


def budget_us(tokens_per_s: float) -> float:
    return 1e6 / tokens_per_s


def mxfp4_bytes(rows: int, cols: int) -> int:
    return rows * (cols // 2 + cols // 32)


def fp8_row_bytes(rows: int, cols: int) -> int:
    return rows * cols + 4 * rows


def layer_weight_bytes(s, n_routed_active: int | None = None) -> int:
    """Weight bytes one token streams through one layer (routed experts: the distinct
    experts the token(s) selected; ``top_k`` when not given)."""
    H, d = s.hidden, s.head_dim
    b = 0
    if s.attn:
        b += 2 * (s.qkv_rows * H + H * s.n_q * d) + 2 * H      # qkv, o-proj, norm gain
    if s.ffn:
        b += 2 * 3 * s.ffn * H + 2 * H
    if s.moe:
        n = s.top_k if n_routed_active is None else n_routed_active
        per_expert = mxfp4_bytes(2 * s.moe_inter, H) + mxfp4_bytes(H, s.moe_inter)
        b += 2 * s.n_experts * H + 2 * H                          # router, norm gain
        b += (n + s.n_shared) * per_expert
    return b


def head_bytes(s) -> int:
    if not s.vocab:
        return 0
    w = fp8_row_bytes(s.vocab, s.hidden) if s.lm_head_dtype == "fp8" else 2 * s.vocab * s.hidden
    return w + (2 * s.hidden if s.final_norm else 0) + (2 * s.hidden if s.embedding else 0)


def kv_bytes(s, pos: int, m: int = 1) -> int:
    """KV bytes one step reads: keys and values of positions [lo, pos + m) of every layer
    (the window's own new rows included; lo = 0, or pos - W + 1 with a sliding window of W
    positions), bf16 (2 B) or FP8 e4m3 (1 B) per element."""
    if not s.attn:
        return 0
    eb = 1 if getattr(s, "kv_dtype", "bf16") == "fp8" else 2
    w = getattr(s, "attn_window", 0)
    lo = max(0, pos - w + 1) if w > 0 else 0
    return s.n_layers * 2 * s.n_kv * s.head_dim * eb * (pos + m - lo)


def algorithmic_bytes(s, pos: int, m: int = 1, n_routed_active: int | None = None) -> int:
    return s.n_layers * layer_weight_bytes(s, n_routed_active) + head_bytes(s) + kv_bytes(s, pos, m)
