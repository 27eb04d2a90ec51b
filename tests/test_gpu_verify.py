"""Verify windows on a dense model with attention (GPU): k tokens at pos..pos+k-1 in one pass,
each attending causally to the cache and to the window's earlier tokens; logits per position
against the oracle's sequential steps, the argmax per position, and the accepted prefix."""
import numpy as np
import pytest

import synth
from tests.harness import TOL, rel_err, weights, oracle_for, decoder_for, top2_margin
from tests.test_gpu_dense import TINY

pytestmark = pytest.mark.gpu


def test_dense_verify_windows():
    from persistent_megakernel_gb300 import build
    build.build()
    seed = 31
    w = weights(TINY, seed)
    cap = TINY.kv_prefill + 8
    dec = decoder_for(TINY, seed, cap, w=w, max_verify=4)
    pos = TINY.kv_prefill
    t0 = synth.start_token(seed, TINY.vocab)
    # drafts: the oracle's own greedy continuation, the last one deliberately wrong
    greedy = [inf["token"] for inf in oracle_for(TINY, seed, cap, w=w).greedy(t0, pos, 3)]
    window = [t0, greedy[0], greedy[1], (greedy[2] + 1) % TINY.vocab]
    orc = oracle_for(TINY, seed, cap, w=w)
    for k in (4, 2, 3, 1):
        toks = window[:k]
        am, n_acc = dec.verify(toks, pos)
        infos, ref_acc = orc.verify(toks, pos)
        lg = dec.logits[:k].cpu().numpy()
        safe = True
        for i in range(k):
            assert rel_err(lg[i], infos[i]["logits"]) <= TOL, (k, i, rel_err(lg[i], infos[i]["logits"]))
            if top2_margin(infos[i]["logits"]) > 1e-3 * np.max(np.abs(infos[i]["logits"])):
                assert am[i] == infos[i]["token"], (k, i, am[i], infos[i]["token"])
            else:
                safe = False
        if safe:
            assert n_acc == ref_acc, (k, n_acc, ref_acc)
    dec.close()
