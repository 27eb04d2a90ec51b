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
@pytest.mark.parametrize("dtype,m,norm", [("bf16", 1, False), ("fp8", 4, False), ("bf16", 2, True), ("fp8", 1, True)])
def test_noalloc_lm_head_matches_context(dtype, m, norm):
    """Two calls in a row with different inputs: logits and argmax equal the context's LM head
    within the tolerance, the oracle's logits within the tolerance, and the planted winners."""
    import torch
    from persistent_megakernel_gb300 import binding as B
    from persistent_megakernel_gb300 import build
    from persistent_megakernel_gb300.model import Decoder
    from oracle import ops
    from oracle.model import OracleModel
    build.build()
    s = synth.lm_head_shape(dtype, verify=m).with_(final_norm=norm)
    hw = sm.head_weights(s, 0)
    xs = [sm.hidden_inputs(s, seed, m) for seed in (3, 4)]  # two calls in a row, different inputs
    gain = bf16_to_f64_fast(hw["final_norm"]) if norm else None
    feats = [bf16_to_f64_fast(x) if gain is None else
             np.stack([ops.rmsnorm(r, gain, s.rms_eps) for r in bf16_to_f64_fast(x)]) for x in xs]
    # plant a winner for every row of both calls (the LM head sees RMSNorm(x) * g when norm is on)
    W, targets = plant_margins(hw["w_lm"], [f for fs in feats for f in fs], 0, margin=1.0, fp8=(dtype == "fp8"))
    head = {"w_lm": W, **({"final_norm": hw["final_norm"]} if norm else {})}
    dec = Decoder(s, [], head, max_verify=m)
    orc = OracleModel(s, [], head, cache_weights=True)
    lm = [t for t in dec._tensors if t.kind == B.DEC_T_LM_HEAD][0]
    fn = [t for t in dec._tensors if t.kind == B.DEC_T_FINAL_NORM]
    fn_dev = fn[0].values if norm else None
    dt = B.DEC_FP8_E4M3_ROWSCALE if dtype == "fp8" else B.DEC_BF16
    stream = torch.cuda.Stream()
    logits = torch.empty((m, s.vocab), dtype=torch.float32, device="cuda")
    argmax = torch.empty(m, dtype=torch.int32, device="cuda")
    for call, x in enumerate(xs):
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
        B.dec_lm_head_noalloc(s.hidden, s.vocab, dt, m, s.rms_eps, xd, fn_dev, lm.values, lm.scales, logits, argmax,
                              stream.cuda_stream)
        lg = logits.cpu().numpy()
        am = argmax.cpu().numpy().tolist()
        for i in range(m):
            assert rel_err(lg[i], ref_lg[i]) <= TOL, (i, rel_err(lg[i], ref_lg[i]))
            ref = orc.logits(bf16_to_f64_fast(x[i]))
            assert rel_err(lg[i], ref) <= TOL, (i, rel_err(lg[i], ref))
        assert am == list(ref_am), (am, ref_am)
        assert am == targets[call * m:(call + 1) * m], (am, targets)
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
