"""The full 42-layer MoE stack on the GPU, its 67 GB of experts drawn and packed on the device.

1. The device generator gives the host generator's values (sampled tensors of every kind).
2. The device packer gives the host packer's bytes (bf16 pair, FP8 rows, MXFP4, edge values).
3. Greedy steps of the full stack, teacher-forced per layer, at steps 0, 1 and 2 and at the
   workload's last step (511, reached by a device-chained generation): for sampled layers the
   oracle recomputes the attention block and the MoE block from the GPU's own input to that
   block, over a cache holding the prefill plus the GPU's own rows of the earlier steps; every
   block output within tolerance, top-k exact wherever the oracle's 8th/9th router gap is safe
   (at least 3 of every 4 layer-steps must be checked; the others are reported as ambiguous);
   the logits of every checked step against the oracle's FP8 head applied to the GPU's final
   hidden state, and the argmax where the top-2 gap is safe.
4. A 4-token verify window of the full stack, teacher-forced per sampled layer and position.
"""
import numpy as np
import pytest
import torch

import synth
from synth import model as sm
from oracle import formats as F
from oracle import ops
from oracle.model import OracleModel, bf16_to_f64_fast
from tests.harness import TOL, rel_err, top2_margin

pytestmark = pytest.mark.gpu

SEED = 0
STEPS = 3          # steps 0 .. STEPS-1 are checked, then the workload's last step
LAST = 511         # the 512-step workload's last step
LAYERS = (0, 1, 21, 41)
ROUTER_MARGIN = 1e-3


@pytest.fixture(scope="module")
def built():
    from persistent_megakernel_gb300 import build
    build.build()
    synth.build_device()


def _dev_bits(shape, kind, layer=0, expert=0, mean=0.0, std=1.0, start=0):
    t = torch.empty(shape, dtype=torch.int16, device="cuda:0")
    synth.normal_bf16_dev(t, SEED, synth.tensor_id(kind, layer, expert), mean, std, start,
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return t.cpu().numpy().view(np.uint16)


def test_device_generator_equals_host(built):
    s = synth.moe_stack_shape()
    cases = [((s.qkv_rows, s.hidden), "w_qkv", 7, 0, 0.0, 0.02, 0),
             ((s.hidden,), "attn_norm", 3, 0, 1.0, 0.02, 0),
             ((s.moe_inter, s.hidden), "e_gate", 5, 311, 0.0, 0.02, 0),
             ((s.hidden, s.moe_inter), "e_down", 41, 512, 0.0, 0.02, 0),
             ((1001, s.head_dim), "k_cache", 9, 0, 0.0, 1.0, 3 * s.kv_prefill * s.head_dim + 1),
             ((4096, s.hidden), "w_lm", 0, 0, 0.0, 0.02, 0),
             ((7,), "x_in", 0, 0, 0.0, 1.0, 5)]
    for shape, kind, layer, expert, mean, std, start in cases:
        want = synth.normal_bf16(SEED, synth.tensor_id(kind, layer, expert), shape, mean, std, start=start)
        got = _dev_bits(shape, kind, layer, expert, mean, std, start)
        assert np.array_equal(got, want), (kind, int(np.sum(got != want)))


def test_device_packer_equals_host(built):
    from persistent_megakernel_gb300 import binding as B
    from persistent_megakernel_gb300.model import pack_host, pack_device
    a = synth.normal_bf16(SEED, 901, (96, 1024), 0.0, 0.02)
    b = synth.normal_bf16(SEED, 902, (96, 1024), 0.0, 0.02)
    a[0, :32] = 0                                   # zero block / row edge cases
    a[1, :] = 0x8000                                # negative zeros
    a[2, 5] = 0x0001                                # bf16 subnormal
    a[3, 7] = 0x4480                                # a large outlier
    a[4, 64:96] = synth.normal_bf16(SEED, 903, 32, 0.0, 1e-30)
    da = torch.from_numpy(a.view(np.int16)).cuda()
    db = torch.from_numpy(b.view(np.int16)).cuda()
    for dtype in (B.DEC_BF16, B.DEC_FP8_E4M3_ROWSCALE, B.DEC_MXFP4):
        for pair in (False, True):
            hv, hs = pack_host(dtype, a, b if pair else None)
            dv, ds = pack_device(dtype, da, db if pair else None)
            torch.cuda.synchronize()
            assert np.array_equal(dv.cpu().numpy(), hv), (dtype, pair)
            if hs is not None:
                assert np.array_equal(ds.cpu().numpy()[:hs.size], hs), (dtype, pair)


def _layer_oracle(s, l):
    """A one-layer oracle holding layer l's weights, cache prefill and experts."""
    return OracleModel(s.with_(n_layers=1), [sm.layer_weights(s, SEED, l)], {}, 
                       experts=lambda _, e: sm.expert_weights(s, SEED, l, e),
                       kv=[sm.kv_prefill(s, SEED, l)], capacity=s.kv_prefill + LAST + 1, cache_weights=True)


def _router_gap(orc, x):
    w = orc.layers[0]
    b = ops.rmsnorm(x, bf16_to_f64_fast(w["ffn_norm"]), orc.s.rms_eps)
    r = (orc.w(0, "w_router") @ b).astype(np.float32).astype(np.float64)
    srt = np.sort(r)[::-1]
    return (srt[orc.s.top_k - 1] - srt[orc.s.top_k]) / np.max(np.abs(r))


class _Head:
    """The oracle's FP8 head, quantised once (codes + scales kept), applied in row chunks."""

    def __init__(self, s):
        self.s = s
        w = sm.head_weights(s, SEED)
        self.embed = w["embed"]
        self.gain = bf16_to_f64_fast(w["final_norm"])
        self.codes, self.scales = [], []
        for r0 in range(0, s.vocab, 16384):
            c, sc = F.quantize_fp8_rows(w["w_lm"][r0:r0 + 16384])
            self.codes.append(c)
            self.scales.append(sc)

    def logits(self, x):
        f = ops.rmsnorm(x, self.gain, self.s.rms_eps)
        return np.concatenate([F.dequant_fp8_rows(c, sc) @ f for c, sc in zip(self.codes, self.scales)])


def _check_step(dec, s, head, orcs, tok, pos, i, counts):
    """One GPU step at pos, teacher-forced per sampled layer against the oracle."""
    am = dec.step(tok, pos)
    hs = dec.hidden_stream()[:, 0].cpu().numpy().astype(np.float64)
    for l in LAYERS:
        orc = orcs[l]
        if pos > s.kv_prefill:  # the cache rows of earlier steps: the GPU's own
            orc.K[0][:, s.kv_prefill:pos] = dec.k_cache[l, :, s.kv_prefill:pos].cpu().numpy().view(np.uint16)
            orc.V[0][:, s.kv_prefill:pos] = dec.v_cache[l, :, s.kv_prefill:pos].cpu().numpy().view(np.uint16)
        x_in = bf16_to_f64_fast(head.embed[tok]) if l == 0 else hs[2 * l]
        y = orc.attention_block(0, x_in, pos)
        assert rel_err(hs[2 * l + 1], y) <= TOL, (i, l, "attention", rel_err(hs[2 * l + 1], y))
        info = {}
        z = orc.ffn_block(0, hs[2 * l + 1], info)
        assert rel_err(hs[2 * l + 2], z) <= TOL, (i, l, "moe", rel_err(hs[2 * l + 2], z))
        got = dec.routing(l)["topk"][0][: s.top_k].tolist()
        if _router_gap(orc, hs[2 * l + 1]) > ROUTER_MARGIN:
            assert got == [int(e) for e in info["topk"][0]], (i, l, got, info["topk"][0])
            counts["checked"] += 1
        else:
            counts["ambiguous"] += 1
    lg_ref = head.logits(hs[2 * s.n_layers])
    lg = dec.logits[0].cpu().numpy()
    assert rel_err(lg, lg_ref) <= TOL, (i, rel_err(lg, lg_ref))
    if top2_margin(lg_ref) > 1e-3 * np.max(np.abs(lg_ref)):
        assert am == ops.argmax_first(lg_ref), (i, am, ops.argmax_first(lg_ref))
    return am


def test_moe_stack_full_teacher_forced(built):
    from tests.device_inputs import device_decoder
    s = synth.moe_stack_shape()
    dec = device_decoder(s, SEED, s.kv_prefill + LAST + 8)
    head = _Head(s)
    orcs = {l: _layer_oracle(s, l) for l in LAYERS}
    tok = synth.start_token(SEED, s.vocab)
    counts = {"checked": 0, "ambiguous": 0}
    for i in range(STEPS):
        tok = _check_step(dec, s, head, orcs, tok, s.kv_prefill + i, i, counts)
    # steps STEPS .. LAST-1 chained on the device, then the last step checked the same way
    out = dec.generate(tok, s.kv_prefill + STEPS, LAST - STEPS)
    dec.sync()
    tok = int(out[-1].item())
    _check_step(dec, s, head, orcs, tok, s.kv_prefill + LAST, LAST, counts)
    n = (STEPS + 1) * len(LAYERS)
    print(f"top-k checked exactly on {counts['checked']} of {n} layer-steps, {counts['ambiguous']} ambiguous")
    assert counts["checked"] >= 3 * n // 4, counts
    dec.close()


def test_moe_stack_full_verify_window(built):
    """A 4-token verify window of the full stack at positions 32768..32771 (a context with
    max_verify 4), teacher-forced per sampled layer: the oracle takes each position in turn,
    causally, over the prefill plus the window's earlier rows as the GPU wrote them; every block
    output within tolerance, top-k exact wherever the oracle's gap is safe (3 of 4 at least),
    and every position's logits against the oracle's FP8 head."""
    from tests.device_inputs import device_decoder
    s = synth.moe_stack_shape()
    dec = device_decoder(s, SEED, s.kv_prefill + 8, max_verify=4)
    head = _Head(s)
    orcs = {l: _layer_oracle(s, l) for l in LAYERS}
    tok0 = synth.start_token(SEED, s.vocab)
    toks = [tok0] + [int(x) for x in synth.bits(SEED, synth.tensor_id("token", 0, 1), 3) % np.uint64(s.vocab)]
    pos = s.kv_prefill
    am, _ = dec.verify(toks, pos)
    hs = dec.hidden_stream().cpu().numpy().astype(np.float64)  # [2L + 1][4][H]
    kc = {l: dec.k_cache[l, :, pos:pos + 4].cpu().numpy().view(np.uint16) for l in LAYERS}
    vc = {l: dec.v_cache[l, :, pos:pos + 4].cpu().numpy().view(np.uint16) for l in LAYERS}
    counts = {"checked": 0, "ambiguous": 0}
    for m in range(4):
        for l in LAYERS:
            orc = orcs[l]
            if m > 0:  # the window's earlier rows, as the GPU appended them
                orc.K[0][:, pos:pos + m] = kc[l][:, :m]
                orc.V[0][:, pos:pos + m] = vc[l][:, :m]
            x_in = bf16_to_f64_fast(head.embed[toks[m]]) if l == 0 else hs[2 * l, m]
            y = orc.attention_block(0, x_in, pos + m)
            assert rel_err(hs[2 * l + 1, m], y) <= TOL, (m, l, "attention", rel_err(hs[2 * l + 1, m], y))
            info = {}
            z = orc.ffn_block(0, hs[2 * l + 1, m], info)
            assert rel_err(hs[2 * l + 2, m], z) <= TOL, (m, l, "moe", rel_err(hs[2 * l + 2, m], z))
            got = dec.routing(l)["topk"][m][: s.top_k].tolist()
            if _router_gap(orc, hs[2 * l + 1, m]) > ROUTER_MARGIN:
                assert got == [int(e) for e in info["topk"][0]], (m, l, got, info["topk"][0])
                counts["checked"] += 1
            else:
                counts["ambiguous"] += 1
        lg_ref = head.logits(hs[2 * s.n_layers, m])
        lg = dec.logits[m].cpu().numpy()
        assert rel_err(lg, lg_ref) <= TOL, (m, rel_err(lg, lg_ref))
        if top2_margin(lg_ref) > 1e-3 * np.max(np.abs(lg_ref)):
            assert am[m] == ops.argmax_first(lg_ref), (m, am[m], ops.argmax_first(lg_ref))
    n = 4 * len(LAYERS)
    print(f"verify window: top-k checked exactly on {counts['checked']} of {n} layer-positions, "
          f"{counts['ambiguous']} ambiguous")
    assert counts["checked"] >= 3 * n // 4, counts
    dec.close()
