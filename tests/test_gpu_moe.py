"""Parity of the MoE FFN block with the oracle (GPU): router top-k over 512 experts, the shared
expert and the 8 routed experts' SwiGLU on MXFP4 weights, the weighted combine and the
residual, for one token and for a 4-token verify window.

The router's top-k must match the oracle exactly. Its fp32 logits are computed in a different
order than the oracle's, so the seed is chosen (by the oracle alone) so that the k-th and the
(k+1)-th logit of every token are well apart; the hidden states after the block are compared
within the usual tolerance.
"""
import numpy as np
import pytest

import synth
from synth import model as sm
from oracle import ops
from oracle.model import bf16_to_f64_fast
from tests.harness import TOL, rel_err, weights, oracle_for, decoder_for

pytestmark = pytest.mark.gpu

SHAPE = synth.moe_layer_shape(verify=4)
MARGIN = 1e-3  # relative gap the seed must leave between the k-th and (k+1)-th router logit


def _router_margin(shape, layers, xs) -> float:
    """Smallest relative gap between the k-th and (k+1)-th router logit over the tokens."""
    w = layers[0]
    gain = bf16_to_f64_fast(w["ffn_norm"])
    W = bf16_to_f64_fast(w["w_router"])
    worst = np.inf
    for x in bf16_to_f64_fast(xs):
        r = (W @ ops.rmsnorm(x, gain, shape.rms_eps)).astype(np.float32).astype(np.float64)
        srt = np.sort(r)[::-1]
        worst = min(worst, (srt[shape.top_k - 1] - srt[shape.top_k]) / np.max(np.abs(r)))
    return worst


@pytest.fixture(scope="module")
def moe():
    from persistent_megakernel_gb300 import build
    build.build()
    for seed in range(16):
        w = weights(SHAPE, seed)
        xs = sm.hidden_inputs(SHAPE, seed, 4)
        if _router_margin(SHAPE, w[0], xs) > MARGIN:
            break
    else:
        pytest.fail("no seed with well-separated router logits")
    dec = decoder_for(SHAPE, seed, 8, w=w, max_verify=4)
    orc = oracle_for(SHAPE, seed, 8, w=w)
    orc.cache_weights = True  # the stored weights, decoded once
    yield seed, xs, dec, orc
    dec.close()


def _check(dec, orc, xs, m_count):
    hs = dec.hidden_stream()[2]  # the residual stream after layer 0's FFN
    route = dec.routing(0)
    for m in range(m_count):
        inf = orc.step(bf16_to_f64_fast(xs[m]), 0)
        assert rel_err(hs[m].cpu().numpy(), inf["x_out"]) <= TOL, (m, rel_err(hs[m].cpu().numpy(), inf["x_out"]))
        got = route["topk"][m][: SHAPE.top_k].tolist()
        assert got == [int(e) for e in inf["topk"][0]], (m, got, inf["topk"][0])
        np.testing.assert_allclose(route["topk_w"][m][: SHAPE.top_k], inf["topk_w"][0], rtol=1e-4, atol=1e-6)
    # slots: the shared expert first, then the window's distinct routed experts
    assert route["expert"][0] == SHAPE.n_experts
    want = []
    for m in range(m_count):
        for e in route["topk"][m][: SHAPE.top_k]:
            if int(e) not in want:
                want.append(int(e))
    assert route["expert"][1:] == want


def test_moe_layer_one_token(moe):
    import torch
    seed, xs, dec, orc = moe
    xd = torch.from_numpy(xs[:1].view(np.int16)).cuda()
    dec.step(0, 0, hidden=xd)
    _check(dec, orc, xs, 1)


def test_moe_layer_verify_window(moe):
    import torch
    seed, xs, dec, orc = moe
    xd = torch.from_numpy(xs.view(np.int16)).cuda()
    dec.verify(None, 0, hidden=xd, k=4)
    _check(dec, orc, xs, 4)


def test_expert_prefetch_modes_agree(moe):
    """The expert prefetch (DEC_EXPERT_PREFETCH: 0 off, 1 adaptive, 2 always) is an L2 hint and
    leaves every result bit for bit unchanged. A repeated input gives the adaptive mode's
    locality rule routed experts to prefetch on the steps after the first."""
    import os
    import torch
    seed, xs, _, orc = moe
    w = weights(SHAPE, seed)
    seq = [0, 0, 1, 0, 0]  # hidden inputs of consecutive one-token steps, positions 0..4
    runs = {}
    old = os.environ.get("DEC_EXPERT_PREFETCH")
    try:
        for mode in ("0", "1", "2"):
            os.environ["DEC_EXPERT_PREFETCH"] = mode
            dec = decoder_for(SHAPE, seed, 8, w=w, max_verify=4)
            out = []
            for pos, i in enumerate(seq):
                dec.step(0, pos, hidden=torch.from_numpy(xs[i:i + 1].view(np.int16)).cuda())
                out.append(dec.hidden_stream()[2][0].cpu().numpy().copy())
            dec.close()
            runs[mode] = np.stack(out)
    finally:
        if old is None:
            os.environ.pop("DEC_EXPERT_PREFETCH", None)
        else:
            os.environ["DEC_EXPERT_PREFETCH"] = old
    assert np.array_equal(runs["0"], runs["1"]) and np.array_equal(runs["0"], runs["2"])
    inf = orc.step(bf16_to_f64_fast(xs[0]), 0)
    assert rel_err(runs["2"][0], inf["x_out"]) <= TOL
