"""Greedy generation chained inside one persistent launch (the monokernel): n steps, each
feeding its argmax to the next at the next position, against the same steps launched one by
one (which the other tests hold to the oracle). The tokens agree, the chain takes one launch,
and the last step's residual stream and the appended cache rows agree bit for bit. A one-layer
MoE model routes the same layer in every step, so a stale routing from the previous step would
show."""
import numpy as np
import pytest

import synth
from synth.configs import ModelShape
from tests.harness import weights, decoder_for

pytestmark = pytest.mark.gpu

TINY = ModelShape("tiny_dense", n_layers=2, hidden=256, n_q=4, n_kv=2, ffn=352, vocab=1000, kv_prefill=70,
                  embedding=True, w_std=0.05)
TINY_MOE = ModelShape("tiny_moe", n_layers=1, hidden=256, n_q=4, n_kv=2, n_experts=16, top_k=2, moe_inter=64,
                      n_shared=1, vocab=1000, kv_prefill=40, embedding=True, w_std=0.05)


@pytest.fixture(scope="module")
def built():
    from persistent_megakernel_gb300 import build
    build.build()


def _chained_vs_stepwise(shape, seed, n, **kw):
    w = weights(shape, seed)
    cap = shape.kv_prefill + n + 4
    tok0 = synth.start_token(seed, shape.vocab)
    a = decoder_for(shape, seed, cap, w=w, **kw)
    toks = a.generate(tok0, shape.kv_prefill, n)
    a.sync()
    assert a.launches() == 1
    hs_chain = a.hidden_stream().cpu().numpy().copy()
    b = decoder_for(shape, seed, cap, w=w, **kw)
    ref, tok = [], tok0
    for i in range(n):
        tok = b.step(tok, shape.kv_prefill + i)
        ref.append(tok)
    assert toks.cpu().tolist() == ref
    # the chain's last step left the residual stream (every block's output) the stepwise run's
    # last step left, bit for bit; so are the cache rows both appended
    assert np.array_equal(hs_chain, b.hidden_stream().cpu().numpy())
    if shape.attn:
        rows = slice(shape.kv_prefill, shape.kv_prefill + n)
        assert np.array_equal(a.k_cache[:, :, rows].cpu().numpy(), b.k_cache[:, :, rows].cpu().numpy())
        assert np.array_equal(a.v_cache[:, :, rows].cpu().numpy(), b.v_cache[:, :, rows].cpu().numpy())
    a.close()
    b.close()


def test_dense_chain(built):
    _chained_vs_stepwise(TINY, 31, 8)


def test_dense_chain_few_ctas(built):
    _chained_vs_stepwise(TINY, 32, 5, num_ctas=3)


def test_moe_one_layer_chain(built):
    _chained_vs_stepwise(TINY_MOE, 33, 6)


def test_chain_of_one(built):
    _chained_vs_stepwise(TINY, 34, 1)
