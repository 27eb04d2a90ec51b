"""The test harness's margin planting (host only): after plant_margins every input row's target
wins its logit by at least the margin on the values the head stores (bf16, or the per-row FP8
quantisation), and only the target rows move."""
import numpy as np
import pytest

import synth
from synth import model as sm
from oracle import formats as F
from oracle.model import bf16_to_f64_fast
from tests.harness import plant_margins


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("m,seed", [(1, 5), (4, 0)])
def test_planted_margins_hold_on_stored_values(fp8, m, seed):
    s = synth.lm_head_shape("bf16")
    w = sm.head_weights(s, 0)["w_lm"][:3000]
    xs = list(bf16_to_f64_fast(sm.hidden_inputs(s, seed, m)))
    W, targets = plant_margins(w, xs, seed, margin=1.0, fp8=fp8)
    Wf = F.dequant_fp8_rows(*F.quantize_fp8_rows(W)) if fp8 else bf16_to_f64_fast(W)
    for t, x in zip(targets, xs):
        lg = Wf @ x
        assert int(np.argmax(lg)) == t
        assert lg[t] - np.max(np.delete(lg, t)) >= 1.0
    moved = set(np.nonzero((W != w).any(axis=1))[0].tolist())
    assert moved <= set(targets) and len(set(targets)) == m
