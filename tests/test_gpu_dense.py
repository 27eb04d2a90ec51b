"""Parity of the CUDA path with the oracle on dense decoder configs (GPU)."""
import numpy as np
import pytest
import torch

import synth
from synth import model as sm
from synth.configs import ModelShape
from tests.harness import TOL, rel_err, weights, oracle_for, decoder_for, top2_margin

pytestmark = pytest.mark.gpu

TINY = ModelShape("tiny_dense", n_layers=2, hidden=256, n_q=4, n_kv=2, ffn=352, vocab=1000, kv_prefill=70,
                  embedding=True, w_std=0.05)


@pytest.fixture(scope="module")
def built():
    from persistent_megakernel_gb300 import build
    build.build()


def _greedy_compare(shape, seed, steps, **kw):
    w = weights(shape, seed)
    cap = shape.kv_prefill + steps + 4
    dec = decoder_for(shape, seed, cap, w=w, **kw)
    orc = oracle_for(shape, seed, cap, w=w)
    tok = synth.start_token(seed, shape.vocab)
    out = []
    for i in range(steps):
        pos = shape.kv_prefill + i
        am = dec.step(tok, pos)
        inf = orc.step_token(tok, pos)
        lg = dec.logits[0].cpu().numpy()
        hs = dec.hidden_stream()[:, 0].cpu().numpy()
        for b, ref in enumerate(inf["hidden"]):
            assert rel_err(hs[b + 1], ref) <= TOL, (i, b, rel_err(hs[b + 1], ref))
        assert rel_err(lg, inf["logits"]) <= TOL, (i, rel_err(lg, inf["logits"]))
        if top2_margin(inf["logits"]) > 1e-3 * np.max(np.abs(inf["logits"])):
            assert am == inf["token"], (i, am, inf["token"])
        out.append((am, lg.copy(), hs.copy()))
        tok = inf["token"]
    return dec, out


def test_tiny_dense_persistent(built):
    _greedy_compare(TINY, 11, 4)


@pytest.mark.parametrize("ctas", [1, 3, 7])
def test_tiny_dense_few_ctas(built, ctas):
    _greedy_compare(TINY, 12, 2, num_ctas=ctas)


def test_modes_bitwise_equal(built):
    res = {}
    for mode in ("persistent", "per_op", "graph"):
        _, out = _greedy_compare(TINY, 13, 3, mode=mode)
        res[mode] = out
    for mode in ("per_op", "graph"):
        for (a, la, ha), (b, lb, hb) in zip(res["persistent"], res[mode]):
            assert a == b and np.array_equal(la, lb) and np.array_equal(ha, hb), mode


def test_run_to_run_deterministic(built):
    _, a = _greedy_compare(TINY, 14, 2)
    _, b = _greedy_compare(TINY, 14, 2)
    for (x, lx, hx), (y, ly, hy) in zip(a, b):
        assert x == y and np.array_equal(lx, ly) and np.array_equal(hx, hy)


def test_empty_cache_position_zero(built):
    # pos 0: each token sees only its own key/value
    s = TINY.with_(kv_prefill=0)
    _greedy_compare(s, 15, 3)


def test_dense_layer_lmhead_config(built):
    s = synth.dense_layer_shape()
    seed = 0
    w = weights(s, seed)
    cap = s.kv_prefill + 4
    dec = decoder_for(s, seed, cap, w=w)
    orc = oracle_for(s, seed, cap, w=w)
    x = sm.hidden_inputs(s, seed, 1)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    am = dec.step(0, s.kv_prefill, hidden=xd)
    from oracle.model import bf16_to_f64_fast
    inf = orc.step(bf16_to_f64_fast(x[0]), s.kv_prefill)
    lg = dec.logits[0].cpu().numpy()
    hs = dec.hidden_stream()[:, 0].cpu().numpy()
    assert rel_err(hs[1], inf["hidden"][0]) <= TOL
    assert rel_err(hs[2], inf["hidden"][1]) <= TOL
    assert rel_err(lg, inf["logits"]) <= TOL
    assert am == inf["token"]
    # the new key/value row went into the cache at pos, rounded to bf16
    kc = dec.k_cache[0, :, s.kv_prefill].cpu().numpy().view(np.uint16)
    kref = orc.K[0][:, s.kv_prefill]
    from oracle.model import bf16_to_f64_fast as f
    assert rel_err(f(kc), f(kref)) <= 1e-2
