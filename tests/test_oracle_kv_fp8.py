"""Pins of the oracle's FP8 KV cache (e4m3 codes with one fp32 scale per layer, K/V and kv head;
the engines in the Kimi-K3 8xB300 benchmark run fp8_e4m3 caches and fall back to scale 1.0).

- every finite e4m3 code survives a round trip under power-of-two scales;
- rounding ties go to the even code, values beyond 448 s saturate, and the decision is taken on
  the fp32 quotient x / s;
- a cache whose contents are exactly representable is lossless: the FP8 cache then gives the
  bf16 cache's step bit for bit, with different scales on keys and values and on every head, so
  a scale dropped, swapped or taken from the wrong head changes the result.
"""
import numpy as np
import pytest

from oracle import formats as F
from oracle.model import OracleModel
from synth.configs import ModelShape

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)


@pytest.mark.parametrize("scale", [1.0, 0.125, 4.0, 2.0 ** -7])
def test_every_code_round_trips(scale):
    v = F.e4m3_to_f64(FINITE) * scale
    q = F.quantize_kv_fp8(v, scale)
    assert np.array_equal(q, FINITE)
    assert np.array_equal(F.dequant_kv_fp8(q, scale), v)


def test_ties_saturation_and_fp32_decision():
    pos = np.arange(0x7E, dtype=np.uint8)           # positive codes 0 .. 0x7D and their successors
    lo, hi = F.e4m3_to_f64(pos), F.e4m3_to_f64(pos + 1)
    mid = (lo + hi) / 2                               # exact in fp32 (4 significant bits + 1)
    for s in (1.0, 2.0 ** -5):
        q = F.quantize_kv_fp8(mid * s, s)
        even = np.where(pos % 2 == 0, pos, pos + 1)
        assert np.array_equal(q, even)
        up = np.nextafter(np.float32(mid * s), np.float32(np.inf)).astype(np.float64)
        dn = np.nextafter(np.float32(mid * s), np.float32(0)).astype(np.float64)
        assert np.array_equal(F.quantize_kv_fp8(up, s), pos + 1)
        assert np.array_equal(F.quantize_kv_fp8(dn, s), pos)
        assert F.quantize_kv_fp8(np.array([449.0 * s, 1e30]), s).tolist() == [0x7E, 0x7E]
        assert F.quantize_kv_fp8(np.array([-449.0 * s]), s).tolist() == [0xFE]
    # quotients that are off a midpoint exactly but land on it in fp32 take the fp32 tie (even
    # code), not the side the exact quotient lies on
    found = 0
    for s in np.float32([3.3, 0.3, 1.7, 5.9, 0.77, 11.1]):
        for c in (0x30, 0x38, 0x3B, 0x45):                          # lower codes of four midpoints
            m = (F.e4m3_to_f64(c) + F.e4m3_to_f64(c + 1)) / 2
            x = np.float32(m * float(s))
            for step in range(-8, 9):
                xi = x
                for _ in range(abs(step)):
                    xi = np.nextafter(xi, np.float32(np.inf if step > 0 else 0))
                if np.float32(xi / s) == np.float32(m) and float(xi) / float(s) != m:
                    want = c if c % 2 == 0 else c + 1
                    assert F.quantize_kv_fp8(np.array([float(xi)]), float(s)).tolist() == [want]
                    found += 1
    assert found >= 4, found


def _lossless_model(kv_dtype, scales, prefill=None):
    """One attention-only layer whose keys and values are small integers: x is +-1 (RMS 1,
    eps 0, unit gains), W_qkv rows for keys and values have three +-1 entries, RoPE is the
    identity at position 0."""
    H, d = 128, 128
    s = ModelShape("kvtest", n_layers=1, hidden=H, n_q=4, n_kv=2, kv_prefill=0 if prefill is None else
                   prefill[0][0].shape[1], rms_eps=0.0, kv_dtype=kv_dtype)
    rng = np.random.default_rng(5)
    wq = rng.normal(0, 0.05, (s.n_q * d, H))
    wkv = np.zeros((2 * s.n_kv * d, H))
    for r in range(wkv.shape[0]):
        cols = rng.choice(H, 3, replace=False)
        wkv[r, cols] = rng.choice([-1.0, 1.0], 3)
    w_qkv = F.f64_to_bf16(np.vstack([wq, wkv]))
    layer = {"attn_norm": np.full(H, 0x3F80, np.uint16),
             "w_qkv": w_qkv,
             "w_o": F.f64_to_bf16(rng.normal(0, 0.05, (H, s.n_q * d)))}
    x0 = np.where(rng.random(H) < 0.5, -1.0, 1.0)
    cap = s.kv_prefill + 2
    return s, OracleModel(s, [layer], {}, kv=prefill, capacity=cap, kv_scales=scales), x0


def test_lossless_fp8_cache_equals_bf16_cache():
    # keys 0.5 and 2 per head, values 4 and 0.25: every k / s and v / s stays exact in e4m3
    scales = np.array([[[0.5, 2.0], [4.0, 0.25]]], np.float32)
    _, fp8, x0 = _lossless_model("fp8", scales)
    _, ref, _ = _lossless_model("bf16", None)
    got = fp8.step(x0, 0)["hidden"][0]
    want = ref.step(x0, 0)["hidden"][0]
    assert np.array_equal(got, want)
    # the stored codes are the values divided by their own head's scale
    k = F.dequant_kv_fp8(fp8.K[0][:, 0], scales[0, 0][:, None])
    v = F.dequant_kv_fp8(fp8.V[0][:, 0], scales[0, 1][:, None])
    assert np.array_equal(k, F.bf16_to_f64(ref.K[0][:, 0]))
    assert np.array_equal(v, F.bf16_to_f64(ref.V[0][:, 0]))
    assert np.abs(k).max() >= 2 and np.abs(v).max() >= 2


def test_prefill_is_quantised_with_its_heads_scales():
    scales = np.array([[[0.5, 2.0], [4.0, 0.25]]], np.float32)
    rng = np.random.default_rng(6)
    codes = rng.choice(FINITE, size=(2, 2, 7, 128))                 # [K/V][head][pos][d]
    vals = F.e4m3_to_f64(codes) * scales[0][:, :, None, None]        # exact in bf16 too
    pre = (F.f64_to_bf16(vals[0]), F.f64_to_bf16(vals[1]))
    assert np.array_equal(F.bf16_to_f64(pre[0]), vals[0])
    _, orc, _ = _lossless_model("fp8", scales, prefill=[pre])
    # -0 and +0 are both exact zeros; compare values, then codes away from zero
    assert np.array_equal(F.dequant_kv_fp8(orc.K[0][:, :7], scales[0, 0][:, None, None]), vals[0])
    assert np.array_equal(F.dequant_kv_fp8(orc.V[0][:, :7], scales[0, 1][:, None, None]), vals[1])
    nz = (codes[0] & 0x7F) != 0
    assert np.array_equal(orc.K[0][:, :7][nz], codes[0][nz])


def test_rescaled_keys_leave_the_step_unchanged():
    # 16 cached positions and the new token at 16: doubling every key scale moves each stored key
    # code by one binade, which is exact in e4m3's normal range, so the step changes only through
    # the few keys near zero (subnormal codes). Reading keys with any other scale than the one
    # they were written with scales the scores, and the step moves by far more.
    import synth
    from synth import model as sm
    s = ModelShape("kvtest2", n_layers=1, hidden=256, n_q=4, n_kv=2, kv_prefill=16, kv_dtype="fp8")
    layer = sm.layer_weights(s, 3, 0)
    kv = [sm.kv_prefill(s, 3, 0)]
    x0 = synth.normal_f64(3, synth.tensor_id("x_in"), s.hidden)
    base = np.array([[[0.5, 2.0], [4.0, 0.25]]], np.float32)
    twice = base.copy()
    twice[0, 0] *= 2
    outs = []
    for sc in (base, twice):
        orc = OracleModel(s, [layer], {}, kv=kv, capacity=s.kv_prefill + 2, kv_scales=sc)
        outs.append(orc.step(x0, s.kv_prefill)["hidden"][0] - x0)      # the attention block's update
    a, b = outs
    assert np.max(np.abs(a - b)) <= 1e-3 * np.max(np.abs(a)), np.max(np.abs(a - b)) / np.max(np.abs(a))
    ref = OracleModel(s.with_(kv_dtype="bf16"), [layer], {}, kv=kv, capacity=s.kv_prefill + 2)
    r = ref.step(x0, s.kv_prefill)["hidden"][0] - x0
    # e4m3 keeps 3 mantissa bits: the update stays within a few percent of the bf16 cache's
    assert np.max(np.abs(a - r)) <= 0.1 * np.max(np.abs(r))
