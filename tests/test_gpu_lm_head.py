"""Parity of the LM-head GEMV + argmax (bf16 and dynamic FP8), batch 1 and 4 (GPU)."""
import numpy as np
import pytest
import torch

import synth
from synth import model as sm
from oracle.model import OracleModel, bf16_to_f64_fast
from tests.harness import TOL, rel_err, plant_margins

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    from persistent_megakernel_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def head_w():
    s = synth.lm_head_shape()
    return sm.head_weights(s, 0)["w_lm"]


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("m", [1, 4])
def test_lm_head(built, head_w, dtype, m):
    from persistent_megakernel_gb300.model import Decoder
    s = synth.lm_head_shape(dtype, verify=m)
    x = sm.hidden_inputs(s, 0, m)
    xf = bf16_to_f64_fast(x)
    W, targets = plant_margins(head_w, list(xf), 0, margin=1.0, fp8=(dtype == "fp8"))
    head = {"w_lm": W}
    dec = Decoder(s, [], head, max_verify=m)
    orc = OracleModel(s, [], head, cache_weights=True)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    if m == 1:
        am = [dec.step(0, 0, hidden=xd)]
    else:
        am, _ = dec.verify(None, 0, hidden=xd, k=m)
    lg = dec.logits[:m].cpu().numpy()
    for i in range(m):
        ref = orc.step(xf[i], 0)
        assert rel_err(lg[i], ref["logits"]) <= TOL, rel_err(lg[i], ref["logits"])
        assert am[i] == ref["token"] == targets[i]
