"""Seeded synthetic weights, KV-cache prefill and inputs for a :class:`ModelShape`.

Everything is returned as logical (unpacked) bfloat16 bits in numpy ``uint16``
arrays, matrices laid out [out_features, in_features] row-major:

* matrices ~ N(0, w_std) (0.02 in every workload);
* RMSNorm gains ~ 1 + N(0, 0.02), so a dropped gain multiply is visible;
* cached keys/values of prefilled positions ~ N(0, 1), keys taken as already rotated;
* given hidden inputs ~ N(0, 1).

Each tensor (and each expert) is its own counter stream, so any subset can be
regenerated without the rest.
"""
from __future__ import annotations

import numpy as np

from . import normal_bf16, tensor_id
from .configs import ModelShape


def _mat(seed, kind, layer, rows, cols, std, expert=0):
    return normal_bf16(seed, tensor_id(kind, layer, expert), (rows, cols), 0.0, std)


def _gain(seed, kind, layer, n):
    return normal_bf16(seed, tensor_id(kind, layer), (n,), 1.0, 0.02)


def layer_weights(s: ModelShape, seed: int, layer: int) -> dict:
    """Dense/attention weights of one layer (routed and shared experts are separate)."""
    H, d = s.hidden, s.head_dim
    w = {}
    if s.attn:
        w["attn_norm"] = _gain(seed, "attn_norm", layer, H)
        w["w_qkv"] = _mat(seed, "w_qkv", layer, s.qkv_rows, H, s.w_std)   # rows: q heads, k heads, v heads
        w["w_o"] = _mat(seed, "w_o", layer, H, s.n_q * d, s.w_std)
    if s.ffn or s.moe:
        w["ffn_norm"] = _gain(seed, "ffn_norm", layer, H)
    if s.ffn:
        w["w_gate"] = _mat(seed, "w_gate", layer, s.ffn, H, s.w_std)
        w["w_up"] = _mat(seed, "w_up", layer, s.ffn, H, s.w_std)
        w["w_down"] = _mat(seed, "w_down", layer, H, s.ffn, s.w_std)
    if s.moe:
        w["w_router"] = _mat(seed, "w_router", layer, s.n_experts, H, s.w_std)
    return w


def expert_weights(s: ModelShape, seed: int, layer: int, expert: int):
    """(gate [I,H], up [I,H], down [H,I]) of one expert; expert ids >= n_experts are the shared ones."""
    H, I = s.hidden, s.moe_inter
    return (_mat(seed, "e_gate", layer, I, H, s.w_std, expert),
            _mat(seed, "e_up", layer, I, H, s.w_std, expert),
            _mat(seed, "e_down", layer, H, I, s.w_std, expert))


def head_weights(s: ModelShape, seed: int) -> dict:
    w = {}
    if s.embedding:
        w["embed"] = _mat(seed, "embed", 0, s.vocab, s.hidden, s.w_std)
    if s.vocab:
        if s.final_norm:
            w["final_norm"] = _gain(seed, "final_norm", 0, s.hidden)
        w["w_lm"] = _mat(seed, "w_lm", 0, s.vocab, s.hidden, s.w_std)
    return w


def kv_prefill(s: ModelShape, seed: int, layer: int, n_pos: int | None = None):
    """Cached (K, V) of one layer for positions [0, n_pos), each [n_kv, n_pos, head_dim] bf16 ~ N(0,1)."""
    n = s.kv_prefill if n_pos is None else n_pos
    shape = (s.n_kv, n, s.head_dim)
    # Position p of head g is draw (g * kv_prefill + p) * d + i, independent of any capacity.
    k = np.empty(shape, np.uint16)
    v = np.empty(shape, np.uint16)
    for g in range(s.n_kv):
        st = g * s.kv_prefill * s.head_dim
        k[g] = normal_bf16(seed, tensor_id("k_cache", layer), (n, s.head_dim), start=st)
        v[g] = normal_bf16(seed, tensor_id("v_cache", layer), (n, s.head_dim), start=st)
    return k, v


def hidden_inputs(s: ModelShape, seed: int, m: int) -> np.ndarray:
    """[m, hidden] bf16 ~ N(0,1): the given hidden states of the single-block workloads."""
    return normal_bf16(seed, tensor_id("x_in"), (m, s.hidden))

