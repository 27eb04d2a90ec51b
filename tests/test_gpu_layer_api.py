"""The layer-level entry points against the oracle (GPU, through the C ABI).

dec_run_layer runs one decoder layer from and to bf16 hidden vectors; dec_lm_head runs the final
norm and the LM head alone. Both run the same kernel as a whole step on an op list of their own.

- dense layer + LM head (one layer, hidden 1024, GQA 8/2, FFN 2816, vocab 32000, 256 cached
  positions): the layer's output for one token and for a causal 3-token window, the rows it
  appends to the KV cache, then the LM head on that output;
- MoE layer (512 MXFP4 experts top-8 + 1 shared): the top-k experts and weights the router
  returns through topk_idx_dev / topk_w_dev, exact on indices, for one token and 4 tokens;
- LM head alone (157184 x 2560, bf16 and FP8 row-scaled, planted margins): logits and argmax.
"""
import numpy as np
import pytest
import torch

import synth
from synth import model as sm
from oracle.model import OracleModel, bf16_to_f64_fast
from tests.harness import TOL, rel_err, weights, oracle_for, decoder_for, plant_margins
from tests.test_gpu_moe import _router_margin, MARGIN

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from persistent_megakernel_gb300 import build
    build.build()


def _dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


@pytest.mark.parametrize("mode", ["persistent", "per_op"])
def test_run_layer_dense_window_and_head(mode):
    s = synth.dense_layer_shape()
    seed = 0
    w = weights(s, seed)
    cap = s.kv_prefill + 8
    dec = decoder_for(s, seed, cap, w=w, max_verify=4, mode=mode)
    pos = s.kv_prefill
    for m in (1, 3):
        xs = sm.hidden_inputs(s, seed + m, m)
        orc = oracle_for(s, seed, cap, w=w)  # fresh cache: rows pos.. are the window's own
        orc.cache_weights = True
        h_out = dec.run_layer(0, _dev(xs), pos)
        got = bf16_to_f64_fast(h_out.cpu().numpy().view(np.uint16))
        refs = []
        for i in range(m):  # the window, causally: token i sees positions 0 .. pos + i
            y = orc.attention_block(0, bf16_to_f64_fast(xs[i]), pos + i)
            refs.append(orc.ffn_block(0, y, {}))
        for i in range(m):
            assert rel_err(got[i], refs[i]) <= TOL, (m, i, rel_err(got[i], refs[i]))
        # the rows the layer appended to the cache are the oracle's bf16 rows
        kc = dec.k_cache[0, :, pos:pos + m].cpu().numpy().view(np.uint16)
        vc = dec.v_cache[0, :, pos:pos + m].cpu().numpy().view(np.uint16)
        assert rel_err(bf16_to_f64_fast(kc), bf16_to_f64_fast(orc.K[0][:, pos:pos + m])) <= TOL
        assert rel_err(bf16_to_f64_fast(vc), bf16_to_f64_fast(orc.V[0][:, pos:pos + m])) <= TOL
        # the LM head on the layer's bf16 output (the oracle takes the same bf16 values)
        am = dec.lm_head(h_out)
        lg = dec.logits[:m].cpu().numpy()
        for i in range(m):
            ref = orc.logits(got[i])
            assert rel_err(lg[i], ref) <= TOL, (m, i, rel_err(lg[i], ref))
            srt = np.sort(ref)
            if srt[-1] - srt[-2] > 1e-2 * np.max(np.abs(ref)):
                assert am[i] == int(np.argmax(ref)), (m, i, am[i], int(np.argmax(ref)))
    dec.close()


@pytest.mark.parametrize("m", [1, 4])
def test_run_layer_moe_topk(m):
    s = synth.moe_layer_shape(verify=4)
    for seed in range(16):
        w = weights(s, seed)
        xs = sm.hidden_inputs(s, seed, 4)
        if _router_margin(s, w[0], xs) > MARGIN:
            break
    else:
        pytest.fail("no seed with well-separated router logits")
    dec = decoder_for(s, seed, 8, w=w, max_verify=4)
    orc = oracle_for(s, seed, 8, w=w)
    orc.cache_weights = True
    h_out, idx, wts = dec.run_layer(0, _dev(xs[:m]), 0, topk=True)
    got = bf16_to_f64_fast(h_out.cpu().numpy().view(np.uint16))
    idx = idx.cpu().numpy()
    wts = wts.cpu().numpy()
    for i in range(m):
        info = {}
        ref = orc.ffn_block(0, bf16_to_f64_fast(xs[i]), info)
        assert rel_err(got[i], ref) <= TOL, (i, rel_err(got[i], ref))
        assert idx[i].tolist() == [int(e) for e in info["topk"][0]], (i, idx[i], info["topk"][0])
        np.testing.assert_allclose(wts[i], info["topk_w"][0], rtol=1e-4, atol=1e-6)
    dec.close()


@pytest.mark.parametrize("dtype,m", [("bf16", 1), ("fp8", 1), ("fp8", 4)])
def test_lm_head_entry(dtype, m):
    from persistent_megakernel_gb300.model import Decoder
    s = synth.lm_head_shape(dtype, verify=m)
    x = sm.hidden_inputs(s, 5, m)
    xf = bf16_to_f64_fast(x)
    W, targets = plant_margins(sm.head_weights(s, 0)["w_lm"], list(xf), 5, margin=1.0, fp8=(dtype == "fp8"))
    head = {"w_lm": W}
    dec = Decoder(s, [], head, max_verify=m)
    orc = OracleModel(s, [], head, cache_weights=True)
    am = dec.lm_head(_dev(x))
    lg = dec.logits[:m].cpu().numpy()
    for i in range(m):
        ref = orc.logits(xf[i])
        assert rel_err(lg[i], ref) <= TOL, rel_err(lg[i], ref)
        assert am[i] == targets[i] == int(np.argmax(ref))
    dec.close()
