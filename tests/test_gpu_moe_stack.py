"""The MoE decode stack (GQA attention over a 32768-position cache, MoE FFN of 512 MXFP4 experts
top-8 + 1 shared, FP8 LM head of 157184 rows, embedding) on the GPU against the oracle, with
the stack shortened to 2 layers: the full 42-layer stack repeats the same layer with 67 GB of
experts to generate. Two greedy steps, teacher-forced with the oracle's tokens."""
import numpy as np
import pytest

import synth
from oracle import ops
from oracle.model import bf16_to_f64_fast
from tests.harness import TOL, rel_err, weights, oracle_for, decoder_for, top2_margin

pytestmark = pytest.mark.gpu

STEPS = 2
ROUTER_MARGIN = 1e-3  # below this relative 8th/9th gap both selections count as correct


def _router_gap(orc, l, x):
    w = orc.layers[l]
    b = ops.rmsnorm(x, bf16_to_f64_fast(w["ffn_norm"]), orc.s.rms_eps)
    r = (orc.w(l, "w_router") @ b).astype(np.float32).astype(np.float64)
    srt = np.sort(r)[::-1]
    return (srt[orc.s.top_k - 1] - srt[orc.s.top_k]) / np.max(np.abs(r))


def test_moe_stack_two_layers():
    from persistent_megakernel_gb300 import build
    build.build()
    s = synth.moe_stack_shape().with_(n_layers=2)
    seed = 0
    w = weights(s, seed)
    cap = s.kv_prefill + STEPS + 4
    dec = decoder_for(s, seed, cap, w=w)
    orc = oracle_for(s, seed, cap, w=w)
    orc.cache_weights = True
    tok = synth.start_token(seed, s.vocab)
    checked, ambiguous = 0, 0
    for i in range(STEPS):
        pos = s.kv_prefill + i
        am = dec.step(tok, pos)
        inf = orc.step_token(tok, pos)
        hs = dec.hidden_stream()[:, 0].cpu().numpy()
        for b, ref in enumerate(inf["hidden"]):
            assert rel_err(hs[b + 1], ref) <= TOL, (i, b, rel_err(hs[b + 1], ref))
        lg = dec.logits[0].cpu().numpy()
        assert rel_err(lg, inf["logits"]) <= TOL, (i, rel_err(lg, inf["logits"]))
        for l in range(s.n_layers):
            got = dec.routing(l)["topk"][0][: s.top_k].tolist()
            if _router_gap(orc, l, inf["hidden"][2 * l]) > ROUTER_MARGIN:
                assert got == [int(e) for e in inf["topk"][l]], (i, l, got, inf["topk"][l])
                checked += 1
            else:
                ambiguous += 1
        if top2_margin(inf["logits"]) > 1e-3 * np.max(np.abs(inf["logits"])):
            assert am == inf["token"], (i, am, inf["token"])
        tok = inf["token"]
    # seed 0: the oracle leaves 3 of the 4 layer-steps unambiguous (step 1, layer 0 has a relative
    # 8th/9th gap of 3.6e-4); every one of them must match exactly
    print(f"top-k checked exactly on {checked} of {checked + ambiguous} layer-steps, {ambiguous} ambiguous")
    assert checked >= 3, (checked, ambiguous)
    dec.close()
