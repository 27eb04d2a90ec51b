"""Seeded workloads built directly in device memory, for models whose weights take too long to
draw and pack on the host (the 42-layer MoE stack holds 127 G expert weights, 67 GB in MXFP4).

The draws are synth's device generator (the same streams and values as ``synth.model``), the
packing is the library's device packer (the same bytes as the host packer). Nothing here
computes any part of the decode step.
"""
from __future__ import annotations

import torch

import synth
from synth import tensor_id


def _stream(device):
    return torch.cuda.current_stream(device).cuda_stream


def normal(shape, seed: int, kind: str, layer: int = 0, expert: int = 0, mean: float = 0.0, std: float = 1.0,
           device="cuda:0", out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 bits (int16 tensor) of stream (kind, layer, expert): ``synth.model``'s tensor."""
    t = out if out is not None else torch.empty(shape, dtype=torch.int16, device=device)
    synth.normal_bf16_dev(t, seed, tensor_id(kind, layer, expert), mean, std, 0, _stream(t.device))
    return t


def layer_weights(s, seed: int, layer: int, device="cuda:0") -> dict:
    """Device copy of ``synth.model.layer_weights`` (same keys, int16 tensors of bf16 bits)."""
    H, d = s.hidden, s.head_dim
    w = {}
    if s.attn:
        w["attn_norm"] = normal((H,), seed, "attn_norm", layer, mean=1.0, std=0.02, device=device)
        w["w_qkv"] = normal((s.qkv_rows, H), seed, "w_qkv", layer, std=s.w_std, device=device)
        w["w_o"] = normal((H, s.n_q * d), seed, "w_o", layer, std=s.w_std, device=device)
    if s.ffn or s.moe:
        w["ffn_norm"] = normal((H,), seed, "ffn_norm", layer, mean=1.0, std=0.02, device=device)
    if s.ffn:
        w["w_gate"] = normal((s.ffn, H), seed, "w_gate", layer, std=s.w_std, device=device)
        w["w_up"] = normal((s.ffn, H), seed, "w_up", layer, std=s.w_std, device=device)
        w["w_down"] = normal((H, s.ffn), seed, "w_down", layer, std=s.w_std, device=device)
    if s.moe:
        w["w_router"] = normal((s.n_experts, H), seed, "w_router", layer, std=s.w_std, device=device)
    return w


def head_weights(s, seed: int, device="cuda:0") -> dict:
    w = {}
    if s.embedding:
        w["embed"] = normal((s.vocab, s.hidden), seed, "embed", 0, std=s.w_std, device=device)
    if s.vocab:
        if s.final_norm:
            w["final_norm"] = normal((s.hidden,), seed, "final_norm", 0, mean=1.0, std=0.02, device=device)
        w["w_lm"] = normal((s.vocab, s.hidden), seed, "w_lm", 0, std=s.w_std, device=device)
    return w


def packed_experts(s, seed: int, layer: int, device="cuda:0"):
    """MXFP4 planes of all routed + shared experts of one layer, drawn and packed on the device:
    (gate/up values [n, I*H], gate/up scales [n, 2*I*H/32], down values [n, H*I/2],
    down scales [n, H*I/32]) as uint8 tensors, expert e's planes contiguous."""
    from persistent_megakernel_gb300 import binding as B
    H, I = s.hidden, s.moe_inter
    n = s.n_experts + s.n_shared
    gu_v = torch.empty((n, I * H), dtype=torch.uint8, device=device)          # [2I][H] / 2
    gu_s = torch.empty((n, 2 * I * H // 32), dtype=torch.uint8, device=device)
    dn_v = torch.empty((n, H * I // 2), dtype=torch.uint8, device=device)
    dn_s = torch.empty((n, H * I // 32), dtype=torch.uint8, device=device)
    g = torch.empty((I, H), dtype=torch.int16, device=device)
    u = torch.empty_like(g)
    dn = torch.empty((H, I), dtype=torch.int16, device=device)
    st = _stream(device)
    for e in range(n):
        normal(None, seed, "e_gate", layer, e, std=s.w_std, out=g)
        normal(None, seed, "e_up", layer, e, std=s.w_std, out=u)
        normal(None, seed, "e_down", layer, e, std=s.w_std, out=dn)
        B.dec_pack_pair_device(B.DEC_MXFP4, g, u, I, H, gu_v[e], gu_s[e], st)
        B.dec_pack_device(B.DEC_MXFP4, dn, H, I, dn_v[e], dn_s[e], st)
    return gu_v, gu_s, dn_v, dn_s


def fill_kv_prefill(s, seed: int, k_cache: torch.Tensor, v_cache: torch.Tensor, kv_scales=None) -> None:
    """Write ``synth.model.kv_prefill`` of every layer into the library's caches
    [n_layers, n_kv, capacity, head_dim] (rows [0, kv_prefill) of each head). An FP8 cache
    (uint8) receives the e4m3 codes of the bf16 draws under kv_scales [n_layers, 2, n_kv]."""
    from persistent_megakernel_gb300 import binding as B
    n, d = s.kv_prefill, s.head_dim
    st = _stream(k_cache.device)
    fp8 = k_cache.dtype == torch.uint8
    tmp = torch.empty((n, d), dtype=torch.int16, device=k_cache.device) if fp8 else None
    for l in range(s.n_layers):
        for g in range(s.n_kv):
            for kv, (cache, kind) in enumerate(((k_cache, "k_cache"), (v_cache, "v_cache"))):
                dst = cache[l, g, :n]
                if not fp8:
                    synth.normal_bf16_dev(dst, seed, tensor_id(kind, l), 0.0, 1.0, g * n * d, st)
                    continue
                synth.normal_bf16_dev(tmp, seed, tensor_id(kind, l), 0.0, 1.0, g * n * d, st)
                scale = 1.0 if kv_scales is None else float(kv_scales[l][kv][g])
                B.dec_pack_kv_fp8_device(tmp, n * d, scale, dst, st)


def device_decoder(s, seed: int, capacity: int, device="cuda:0", **kw):
    """A Decoder of shape s with every weight and the KV prefill drawn and packed on the device."""
    from persistent_megakernel_gb300.model import Decoder
    torch.cuda.set_device(torch.device(device))
    layers = [layer_weights(s, seed, l, device) for l in range(s.n_layers)]
    head = head_weights(s, seed, device)
    experts = None
    if s.moe:
        cache = {}

        def experts(l):
            if l not in cache:
                cache.clear()
                cache[l] = packed_experts(s, seed, l, device)
            return cache[l]

    dec = Decoder(s, layers, head, kv=None, capacity=capacity, device=device, packed_experts=experts, **kw)
    if s.attn:
        fill_kv_prefill(s, seed, dec.k_cache, dec.v_cache, kw.get("kv_scales"))
    torch.cuda.synchronize(device)
    return dec
