"""The pins must catch plausible mistakes: each case plants one mistake in the
oracle (on the CPU, via monkeypatch) and checks that a pin test then fails."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import model as M
from oracle import ops
import tests.test_oracle_formats as tf
import tests.test_oracle_kv_fp8 as tk
import tests.test_oracle_model as tm
import tests.test_oracle_ops as to


def _rope_sign(u, pos, base):
    d = u.shape[-1]
    h = d // 2
    th = pos * base ** (-2.0 * np.arange(h) / d)
    u1, u2 = u[..., :h], u[..., h:]
    return np.concatenate([u1 * np.cos(th) + u2 * np.sin(th), -u1 * np.sin(th) + u2 * np.cos(th)], -1)


def _rope_interleaved(u, pos, base):
    d = u.shape[-1]
    th = pos * base ** (-2.0 * np.arange(d // 2) / d)
    a, b = u[..., 0::2], u[..., 1::2]
    out = np.empty_like(u)
    out[..., 0::2] = a * np.cos(th) - b * np.sin(th)
    out[..., 1::2] = a * np.sin(th) + b * np.cos(th)
    return out


def _attn_noscale(q, K, V):
    o = np.empty_like(q)
    for h in range(q.shape[0]):
        g = ops.kv_group(h, q.shape[0], K.shape[0])
        o[h] = ops.softmax(K[g] @ q[h]) @ V[g]
    return o


def _mx_swap(w):
    c, e = _ORIG_MX(w)
    return ((c >> 4) | (c << 4)).astype(np.uint8), e


def _fp8_127(w):
    w32 = F.bf16_to_f64(w).astype(np.float32)
    amax = np.max(np.abs(w32), axis=1)
    s = np.where(amax == 0, 1.0, amax / np.float32(127.0)).astype(np.float32)
    return F.round_e4m3_satfinite((w32 / s[:, None]).astype(np.float64)), s


_ORIG_MX = F.quantize_mxfp4


def _no_residual(self, l, x, pos):
    out = _ORIG_ATTN(self, l, x, pos)
    return out - x


_ORIG_ATTN = M.OracleModel.attention_block


def _cache_unrounded(self, l, x, pos):
    saved = F.f64_to_bf16
    try:
        F.f64_to_bf16 = lambda v: saved(np.round(np.asarray(v) * 8) / 8)   # coarse, wrong rounding
        return _ORIG_ATTN(self, l, x, pos)
    finally:
        F.f64_to_bf16 = saved


def _kv_fp64_division(x, scale):
    return F.round_e4m3_satfinite(np.asarray(x, np.float64) / np.asarray(scale, np.float64))


_ORIG_KV_SCALE = M.OracleModel._kv_scale


def _kv_read_other_scale(self, l, kv, ndim):
    # cache reads (and the prefill) take the other half's scale; the new row's write is right
    return _ORIG_KV_SCALE(self, l, 1 - kv if ndim == 3 else kv, ndim)


def _kv_heads_reversed(self, l, kv, ndim):
    return self.kv_scales[l, kv][::-1].reshape((-1,) + (1,) * (ndim - 1))


CASES = [
    ("rope sign", ops, "rope", _rope_sign, to.test_rope_pos0_identity_and_rotation_form),
    ("rope pairing", ops, "rope", _rope_interleaved, to.test_rope_pos0_identity_and_rotation_form),
    ("rmsnorm drops gain", ops, "rmsnorm", lambda x, g, eps: x / np.sqrt(np.mean(x * x) + eps),
     to.test_rmsnorm_closed_forms),
    ("rmsnorm eps outside root", ops, "rmsnorm", lambda x, g, eps: x / (np.sqrt(np.mean(x * x)) + eps) * g,
     to.test_rmsnorm_closed_forms),
    ("attention without 1/sqrt(d)", ops, "attention", _attn_noscale, to.test_attention_brute_force_gqa),
    ("gqa grouping modulo", ops, "kv_group", lambda h, nq, nkv: h % nkv, to.test_attention_brute_force_gqa),
    ("gemv transposed", ops, "gemv", lambda W, a: W.T @ a if W.shape[0] == W.shape[1] else W @ a,
     to.test_gemv_orientation),
    ("topk ascending", ops, "topk_desc", lambda r, k: np.argsort(r, kind="stable")[:k],
     to.test_topk_brute_force_and_ties),
    ("silu as sigmoid", ops, "silu", lambda z: 1.0 / (1.0 + np.exp(-z)), to.test_silu_and_swiglu),
    ("argmax last index", ops, "argmax_first", lambda lg: int(np.flatnonzero(lg == lg.max())[-1]),
     to.test_argmax_and_acceptance),
    ("mxfp4 nibble order", F, "quantize_mxfp4", _mx_swap, tf.test_mxfp4_quantiser_brute_force),
    ("fp8 scale 127", F, "quantize_fp8_rows", _fp8_127, tf.test_fp8_row_quantiser_brute_force),
    ("residual dropped", M.OracleModel, "attention_block", _no_residual, tm.test_dense_step_matches_loop_evaluation),
    ("cache rounding wrong", M.OracleModel, "attention_block", _cache_unrounded,
     tm.test_dense_step_matches_loop_evaluation),
    ("kv fp8 fp64 division", F, "quantize_kv_fp8", _kv_fp64_division, tk.test_ties_saturation_and_fp32_decision),
    ("kv fp8 read unscaled", F, "dequant_kv_fp8", lambda codes, scale: F.e4m3_to_f64(codes),
     tk.test_lossless_fp8_cache_equals_bf16_cache),
    ("kv fp8 keys read with value scales", M.OracleModel, "_kv_scale", _kv_read_other_scale,
     tk.test_rescaled_keys_leave_the_step_unchanged),
    ("kv fp8 head scales reversed", M.OracleModel, "_kv_scale", _kv_heads_reversed,
     tk.test_lossless_fp8_cache_equals_bf16_cache),
]


@pytest.mark.parametrize("name,mod,attr,bad,pin", CASES, ids=[c[0] for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, name, mod, attr, bad, pin):
    pin()                                   # the pin passes on the real oracle
    monkeypatch.setattr(mod, attr, bad)
    with pytest.raises(AssertionError):
        pin()
