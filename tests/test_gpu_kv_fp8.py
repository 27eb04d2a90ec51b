"""FP8 e4m3 KV cache on the GPU against the oracle's FP8 cache (same per-head scales): the
prefill stored as codes by the packer, every new key and value quantised by the kernel.

Greedy steps of a small dense decoder and of the 2B decoder's shape shortened to 2 layers:
every block's output and the logits within tolerance, argmax where the top-2 gap is safe; the
codes the kernel appended agree with the oracle's (the few that differ sit next to a rounding
boundary the two fp32 keys fall on different sides of, one code apart). All three launch modes
give the same bits.
"""
import numpy as np
import pytest

import synth
from synth.configs import ModelShape
from tests.harness import TOL, rel_err, weights, top2_margin

pytestmark = pytest.mark.gpu

TINY8 = ModelShape("tiny_dense_kv8", n_layers=2, hidden=256, n_q=4, n_kv=2, ffn=352, vocab=1000, kv_prefill=70,
                   embedding=True, w_std=0.05, kv_dtype="fp8")


@pytest.fixture(scope="module")
def built():
    from persistent_megakernel_gb300 import build
    build.build()


def _scales(shape, seed):
    # distinct per layer, keys / values and head; powers of two and not (the quotient rounds)
    u = synth.normal_f64(seed, synth.tensor_id("x_in", 0, 99), shape.n_layers * 2 * shape.n_kv)
    return (0.75 + 0.25 * np.abs(u)).astype(np.float32).reshape(shape.n_layers, 2, shape.n_kv)


def _compare(shape, seed, steps, **kw):
    from oracle.model import OracleModel
    from persistent_megakernel_gb300.model import Decoder
    layers, head, kv, experts = weights(shape, seed)
    sc = _scales(shape, seed)
    cap = shape.kv_prefill + steps + 4
    dec = Decoder(shape, layers, head, experts=experts, kv=kv, capacity=cap, kv_scales=sc, **kw)
    orc = OracleModel(shape, layers, head, experts=experts, kv=kv, capacity=cap, kv_scales=sc, cache_weights=True)
    # the packer's prefill codes are the oracle's, bit for bit
    for l in range(shape.n_layers):
        n = shape.kv_prefill
        assert np.array_equal(dec.k_cache[l, :, :n].cpu().numpy(), orc.K[l][:, :n])
        assert np.array_equal(dec.v_cache[l, :, :n].cpu().numpy(), orc.V[l][:, :n])
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
        for l in range(shape.n_layers):
            for cache, ref in ((dec.k_cache, orc.K[l]), (dec.v_cache, orc.V[l])):
                got = cache[l, :, pos].cpu().numpy().astype(np.int32)
                want = ref[:, pos].astype(np.int32)
                diff = got != want
                # same sign, magnitude one code apart, and rare
                assert np.all(np.abs((got & 0x7F) - (want & 0x7F))[diff] <= 1), (i, l)
                assert diff.mean() <= 0.02, (i, l, diff.mean())
        out.append((am, lg.copy(), hs.copy()))
        tok = inf["token"]
    return dec, out


def test_tiny_dense_fp8_kv(built):
    _compare(TINY8, 21, 4)


def test_fp8_kv_few_ctas(built):
    _compare(TINY8, 22, 2, num_ctas=3)


def test_fp8_kv_2b_shape_two_layers(built):
    s = synth.dense_2b_shape().with_(n_layers=2, kv_dtype="fp8")
    _compare(s, 0, 2)


def test_fp8_kv_modes_bitwise_equal(built):
    res = {m: _compare(TINY8, 23, 3, mode=m)[1] for m in ("persistent", "per_op", "graph")}
    for mode in ("per_op", "graph"):
        for (a, la, ha), (b, lb, hb) in zip(res["persistent"], res[mode]):
            assert a == b and np.array_equal(la, lb) and np.array_equal(ha, hb), mode
