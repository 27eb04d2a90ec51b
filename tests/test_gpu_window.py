"""Sliding-window attention on the GPU against the oracle: every token attends to its last W
positions only (the Muse Spark Open megakernel article, section "where the kernel boundary
sits": most of that model's layers attend over the last 2,048 tokens). Tiny dense decoder with
70 cached positions and W = 24: greedy steps and a 4-token verify window (each token of the
window has its own window start), bf16 cache on the tensor-core tiles and the CUDA-core tiles
(FP8 cache)."""
import numpy as np
import pytest
import torch

import synth
from synth.configs import ModelShape
from tests.harness import TOL, rel_err, weights, oracle_for, decoder_for, top2_margin

pytestmark = pytest.mark.gpu

TINYW = ModelShape("tiny_dense_window", n_layers=2, hidden=256, n_q=4, n_kv=2, ffn=352, vocab=1000, kv_prefill=70,
                   embedding=True, w_std=0.05, attn_window=24)


@pytest.fixture(scope="module", autouse=True)
def built():
    from persistent_megakernel_gb300 import build
    build.build()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_window_steps_and_verify(kv):
    s = TINYW.with_(kv_dtype=kv)
    seed = 11
    w = weights(s, seed)
    cap = s.kv_prefill + 12
    dec = decoder_for(s, seed, cap, w=w, max_verify=4)
    orc = oracle_for(s, seed, cap, w=w)
    tok = synth.start_token(seed, s.vocab)
    for i in range(4):
        pos = s.kv_prefill + i
        am = dec.step(tok, pos)
        inf = orc.step_token(tok, pos)
        hs = dec.hidden_stream()[:, 0].cpu().numpy()
        for b, ref in enumerate(inf["hidden"]):
            assert rel_err(hs[b + 1], ref) <= TOL, (i, b, rel_err(hs[b + 1], ref))
        lg = dec.logits[0].cpu().numpy()
        assert rel_err(lg, inf["logits"]) <= TOL, (i, rel_err(lg, inf["logits"]))
        if top2_margin(inf["logits"]) > 1e-3 * np.max(np.abs(inf["logits"])):
            assert am == inf["token"], (i, am, inf["token"])
        tok = inf["token"]
    # a 4-token window at the next positions: token m sees positions pos + m - W + 1 .. pos + m
    pos = s.kv_prefill + 4
    toks = [tok, 5, 17, 401]
    infos, n_acc = orc.verify(toks, pos)
    am, acc = dec.verify(toks, pos)
    lg = dec.logits[:4].cpu().numpy()
    for m in range(4):
        assert rel_err(lg[m], infos[m]["logits"]) <= TOL, (m, rel_err(lg[m], infos[m]["logits"]))
    assert acc == n_acc
    dec.close()
