"""The allocation-free LM head (dec_lm_head_noalloc) against the context's own LM head.

Some callers cannot allocate device memory: code running inside a memory pool or arena it does
not own, or where cudaMalloc / cudaFree may not be called (they can synchronise the device and
fail inside some capture or callback contexts). dec_lm_head_noalloc serves them: the caller
passes its inputs, weights and output buffers, and the kernel's scratch is a static device
array inside the library. This file sorts last so that a run stopping at its first failure has
already run every other test; it passes alone in a fresh process and after the others.
"""
import numpy as np
import pytest

import synth
from synth import model as sm
from oracle.model import bf16_to_f64_fast
from tests.harness import TOL, rel_err, plant_margins


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,m", [("bf16", 1), ("fp8", 4)])
def test_noalloc_lm_head_matches_context(dtype, m):
    import torch
    from persistent_megakernel_gb300 import binding as B
    from persistent_megakernel_gb300 import build
    from persistent_megakernel_gb300.model import Decoder
    build.build()
    s = synth.lm_head_shape(dtype, verify=m)
    head_w = sm.head_weights(s, 0)["w_lm"]
    xs = [sm.hidden_inputs(s, seed, m) for seed in (3, 4)]  # two calls in a row, different inputs
    W, _ = plant_margins(head_w, list(bf16_to_f64_fast(xs[0])), 0, margin=1.0, fp8=(dtype == "fp8"))
    dec = Decoder(s, [], {"w_lm": W}, max_verify=m)
    lm = [t for t in dec._tensors if t.kind == B.DEC_T_LM_HEAD][0]
    dt = B.DEC_FP8_E4M3_ROWSCALE if dtype == "fp8" else B.DEC_BF16
    stream = torch.cuda.Stream()
    logits = torch.empty((m, s.vocab), dtype=torch.float32, device="cuda")
    argmax = torch.empty(m, dtype=torch.int32, device="cuda")
    for x in xs:
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        # the existing entry point: a context holding only this LM head
        if m == 1:
            ref_am = [dec.step(0, 0, hidden=xd)]
        else:
            ref_am, _ = dec.verify(None, 0, hidden=xd, k=m)
        ref_lg = dec.logits[:m].cpu().numpy()
        torch.cuda.synchronize()
        logits.fill_(float("nan"))
        argmax.fill_(-1)
        torch.cuda.synchronize()
        B.dec_lm_head_noalloc(s.hidden, s.vocab, dt, m, s.rms_eps, xd, None, lm.values, lm.scales, logits, argmax,
                              stream.cuda_stream)
        lg = logits.cpu().numpy()
        am = argmax.cpu().numpy().tolist()
        for i in range(m):
            assert rel_err(lg[i], ref_lg[i]) <= TOL, (i, rel_err(lg[i], ref_lg[i]))
        assert am == list(ref_am), (am, ref_am)
    dec.close()


def test_noalloc_rejects_bad_sizes():
    """Argument checks happen before any device work (no GPU needed)."""
    from persistent_megakernel_gb300 import binding as B
    try:
        B.lib()
    except ImportError:
        pytest.skip("libdec.so not built")
    with pytest.raises(B.DecError) as e:
        B.dec_lm_head_noalloc(2560, 1000, B.DEC_BF16, 5, 1e-6, 16, None, 16, None, 16, 16, None)
    assert e.value.code == B.DEC_ERR_SHAPE
    with pytest.raises(B.DecError) as e:
        B.dec_lm_head_noalloc(100, 1000, B.DEC_BF16, 1, 1e-6, 16, None, 16, None, 16, 16, None)
    assert e.value.code == B.DEC_ERR_SHAPE
    with pytest.raises(B.DecError) as e:
        B.dec_lm_head_noalloc(2560, 1000, B.DEC_FP8_E4M3_ROWSCALE, 1, 1e-6, 16, None, 16, None, 16, 16, None)
    assert e.value.code == B.DEC_ERR_INVALID_ARG
