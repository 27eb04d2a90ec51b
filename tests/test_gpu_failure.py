"""Failure detection without a GPU fault: a step whose producer op is dropped on the host makes
the consumer's bounded wait run out; the call reports DEC_ERR_TIMEOUT, stays sticky until
dec_reset, and the same context then decodes correctly (GPU)."""
import numpy as np
import pytest

import synth
from tests.harness import TOL, rel_err, weights, oracle_for, decoder_for
from tests.test_gpu_dense import TINY

pytestmark = pytest.mark.gpu


def test_dropped_op_times_out_and_recovers():
    from persistent_megakernel_gb300 import binding as B
    from persistent_megakernel_gb300 import build
    build.build()
    seed = 21
    w = weights(TINY, seed)
    cap = TINY.kv_prefill + 4
    dec = decoder_for(TINY, seed, cap, w=w, mode="per_op", timeout_ns=200_000_000)
    orc = oracle_for(TINY, seed, cap, w=w)
    tok = synth.start_token(seed, TINY.vocab)
    pos = TINY.kv_prefill
    B.dec_debug_drop_op(dec.ctx, 1)  # layer 0's attention: the o-projection waits for its output
    with pytest.raises(B.DecError) as e:
        dec.step(tok, pos)
    assert e.value.code == B.DEC_ERR_TIMEOUT, e.value
    with pytest.raises(B.DecError) as e:
        dec.step(tok, pos)  # sticky until reset
    assert e.value.code == B.DEC_ERR_STATE
    dec.reset()
    am = dec.step(tok, pos)
    ref = orc.step_token(tok, pos)
    assert rel_err(dec.logits[0].cpu().numpy(), ref["logits"]) <= TOL
    assert am == ref["token"]
    dec.close()
