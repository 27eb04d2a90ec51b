"""Shared test helpers: build the same seeded model for the CUDA path and the oracle."""
from __future__ import annotations

import numpy as np

import synth
from synth import model as sm
from oracle.model import OracleModel

TOL = 2e-2   # max |delta| <= TOL * max |ref| on bf16 hidden states and logits


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def weights(shape, seed):
    layers = [sm.layer_weights(shape, seed, l) for l in range(shape.n_layers)]
    head = sm.head_weights(shape, seed)
    kv = [sm.kv_prefill(shape, seed, l) for l in range(shape.n_layers)] if shape.attn else None
    experts = (lambda l, e: sm.expert_weights(shape, seed, l, e)) if shape.moe else None
    return layers, head, kv, experts


def oracle_for(shape, seed, capacity, w=None):
    layers, head, kv, experts = w if w is not None else weights(shape, seed)
    return OracleModel(shape, layers, head, experts=experts, kv=kv, capacity=capacity)


def decoder_for(shape, seed, capacity, w=None, **kw):
    from persistent_megakernel_gb300.model import Decoder
    layers, head, kv, experts = w if w is not None else weights(shape, seed)
    return Decoder(shape, layers, head, experts=experts, kv=kv, capacity=capacity, **kw)


def top2_margin(logits) -> float:
    s = np.sort(np.asarray(logits, np.float64))
    return float(s[-1] - s[-2])


_STORED = {}  # content hash of a bf16 matrix and its format -> its stored values in fp64


def _stored_f64(W, fp8):
    """The values a bf16 matrix holds once stored (bf16 as is, or its per-row FP8 quantisation),
    cached by content: several tests plant margins on the same generated head."""
    import hashlib
    from oracle import formats as F
    from oracle.model import bf16_to_f64_fast
    key = (hashlib.sha1(W.tobytes()).hexdigest(), W.shape, fp8)
    if key not in _STORED:
        _STORED.clear()
        _STORED[key] = F.dequant_fp8_rows(*F.quantize_fp8_rows(W)) if fp8 else bf16_to_f64_fast(W)
    return _STORED[key].copy()


def plant_margins(w_lm, xs, seed, margin=1.0, fp8=False):
    """Make argmax unique: for each input row x_m pick a target row t_m (seeded) and move
    W[t_m] along x_m so that its logit exceeds every other logit by `margin` (checked on the
    stored weights: bf16, or their FP8 quantisation). Returns (new W, targets). Both formats
    store each row on its own (FP8 scales are per row), so after moving a row only that row's
    stored values are recomputed."""
    from oracle import formats as F
    from oracle.model import bf16_to_f64_fast
    W = np.array(w_lm, dtype=np.uint16, copy=True)
    V = W.shape[0]
    draws = synth.bits(seed + 1, synth.tensor_id("token"), len(xs))
    targets = []
    for m, x in enumerate(xs):
        t = int(draws[m] % np.uint64(V))
        while t in targets:
            t = (t + 1) % V
        targets.append(t)
    Wf = _stored_f64(W, fp8)

    def restore(t):
        Wf[t] = (F.dequant_fp8_rows(*F.quantize_fp8_rows(W[t:t + 1])) if fp8 else bf16_to_f64_fast(W[t:t + 1]))[0]

    for _ in range(4):
        ok = True
        moved = []
        for m, x in enumerate(xs):
            t = targets[m]
            lg = Wf @ x
            others = np.delete(lg, t)
            gap = lg[t] - others.max()
            if gap < margin:
                ok = False
                alpha = (others.max() + 1.5 * margin - lg[t])
                row = bf16_to_f64_fast(W[t]) + alpha * x / float(x @ x)
                W[t] = F.f64_to_bf16(row)
                moved.append(t)
        if ok:
            return W, targets
        for t in moved:  # the next round checks the stored values of the moved rows
            restore(t)
    raise AssertionError("could not plant margins")
