"""Pins of the oracle's number formats and quantisers (CPU only).

Each check compares the oracle with something other than itself: the hardware
fp32 interpretation of bf16 bits, torch's float8_e4m3fn conversion, the OCP
spec tables under tests/golden/, the input generator's independent bf16
rounding, or brute force over every code.
"""
import os

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.model import bf16_to_f64_fast
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _all_bf16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_bf16_decode_matches_fp32_upper_half():
    codes = _all_bf16()
    ours = F.bf16_to_f64(codes)
    hw = (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(hw)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], hw[~nan])
    # signed zeros kept
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])


def test_bf16_fast_decode_equals_definition():
    codes = _all_bf16()
    a, b = F.bf16_to_f64(codes), bf16_to_f64_fast(codes)
    nan = np.isnan(a)
    assert np.array_equal(nan, np.isnan(b))
    assert np.array_equal(a[~nan], b[~nan])


def test_bf16_rounding_idempotent_and_ties_even():
    codes = np.arange(0x7F80, dtype=np.uint16)           # every positive finite code
    vals = F.bf16_to_f64(codes)
    assert np.array_equal(F.f64_to_bf16(vals), codes)
    assert np.array_equal(F.f64_to_bf16(-vals[1:]), codes[1:] | 0x8000)
    mid = (vals[:-1] + vals[1:]) / 2                      # exact midpoints in fp64
    got = F.f64_to_bf16(mid)
    want = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(got, want)


def test_bf16_rounding_matches_generator_and_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))
    ours = F.f64_to_bf16(x)
    gen = np.array([synth.f64_to_bf16(v) for v in x], dtype=np.uint16)
    assert np.array_equal(ours, gen)
    # fp32-representable inputs: torch's fp32 -> bf16 is round-to-nearest-even
    x32 = x.astype(np.float32)
    t = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.f64_to_bf16(x32.astype(np.float64)), t)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = F.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ours[~nan], ref[~nan])


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_e2m1_decode_matches_ocp_table():
    for code, val in _golden_lines("e2m1_values.txt"):
        got = F.e2m1_to_f64(np.array([int(code)], np.uint8))[0]
        assert got == float(val) and np.signbit(got) == val.startswith("-")


def test_e4m3_e8m0_landmarks():
    for fmt, code, val in _golden_lines("fp8_e4m3_landmarks.txt"):
        c = np.array([int(code, 16)], np.uint8)
        got = (F.e4m3_to_f64 if fmt == "e4m3" else F.e8m0_to_f64)(c)[0]
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val)


def test_e4m3_rounding_matches_torch_in_range():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(50000) * np.exp(rng.uniform(-12, 6, 50000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    grid = F.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)  # midpoints are exact in fp32
    x = np.concatenate([x, mids, -mids])
    ours = F.round_e4m3_satfinite(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates():
    assert F.round_e4m3_satfinite(np.array([1e6, -500.0, 464.0]))[0] == 0x7E
    assert F.round_e4m3_satfinite(np.array([-500.0]))[0] == 0xFE


def test_e2m1_tie_table():
    # ties between neighbours go to the even code (OCP round-to-nearest-even)
    cases = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0, 7.0: 6.0, 100.0: 6.0}
    for x, want in cases.items():
        c = F.round_e2m1_satfinite(np.array([x, -x]))
        assert F.e2m1_to_f64(c)[0] == want and F.e2m1_to_f64(c)[1] == -want


def _brute_nearest(y, grid_vals):
    """index of the nearest value in an arbitrary list, ties -> even index (pure Python)."""
    best, bi = None, None
    for i, g in enumerate(grid_vals):
        d = abs(y - g)
        if best is None or d < best or (d == best and i % 2 == 0):
            best, bi = d, i
    return bi


def test_fp8_row_quantiser_brute_force():
    w = synth.normal_bf16(7, 99, (6, 40), 0.0, 0.02)
    w[2] = 0                                            # a zero row takes scale 1
    codes, s = F.quantize_fp8_rows(w)
    assert s.dtype == np.float32 and s[2] == 1.0 and np.all(codes[2] == 0)
    grid = list(F.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8)))
    w32 = F.bf16_to_f64(w).astype(np.float32)
    for r in range(w.shape[0]):
        amax = float(np.max(np.abs(w32[r])))
        if amax:
            assert s[r] == np.float32(amax) / np.float32(448.0)
        for c in range(w.shape[1]):
            y = float(np.float32(w32[r, c]) / s[r])
            idx = _brute_nearest(min(abs(y), 448.0), grid)
            assert codes[r, c] & 0x7F == idx
            assert (codes[r, c] >> 7) == (1 if np.signbit(w32[r, c]) else 0)
    # the largest element of each non-zero row maps to +-448
    deq = F.dequant_fp8_rows(codes, s)
    for r in (0, 1, 3):
        assert np.max(np.abs(F.e4m3_to_f64(codes[r]))) == 448.0
    assert np.max(np.abs(deq - F.bf16_to_f64(w))) <= np.max(np.abs(F.bf16_to_f64(w))) / 16 + 1e-12


def test_mxfp4_quantiser_brute_force():
    w = synth.normal_bf16(5, 77, (5, 96), 0.0, 0.02)
    w[1, 32:64] = 0                                     # an all-zero block
    codes, e = F.quantize_mxfp4(w)
    assert codes.shape == (5, 48) and e.shape == (5, 3)
    v = F.bf16_to_f64(w)
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for r in range(5):
        for b in range(3):
            blk = v[r, 32 * b:32 * b + 32]
            amax = np.max(np.abs(blk))
            if amax == 0:
                assert e[r, b] == 0
            else:
                X = 2.0 ** (int(e[r, b]) - 127)
                assert 4.0 <= amax / X < 8.0             # X = 2^(floor(log2 amax) - 2)
            X = 2.0 ** (int(e[r, b]) - 127)
            for i in range(32):
                col = 32 * b + i
                byte = codes[r, col // 2]
                c = (byte & 0xF) if col % 2 == 0 else (byte >> 4)
                y = blk[i] / X
                assert (c & 7) == _brute_nearest(min(abs(y), 6.0), grid)
                assert (c >> 3) == (1 if np.signbit(blk[i]) else 0)


def test_mxfp4_scale_on_powers_of_two_and_saturation():
    # a block whose max is exactly 2^k takes X = 2^(k-2); values in (6, 8) * X saturate to 6
    for k in (-10, -3, 0, 2):
        row = np.zeros((1, 32))
        row[0, 0] = 2.0 ** k
        row[0, 1] = 2.0 ** k * 0.99
        codes, e = F.quantize_mxfp4(F.f64_to_bf16(row))
        assert int(e[0, 0]) - 127 == k - 2
        # 2^k / 2^(k-2) = 4 -> code 6 (value 4); 0.99 * 4 = 3.96 -> 4
        assert codes[0, 0] & 0xF == 6 and codes[0, 0] >> 4 == 6
    row = np.zeros((1, 32))
    row[0, 0] = 7.5                                     # amax/X = 7.5 -> saturates to 6
    codes, e = F.quantize_mxfp4(F.f64_to_bf16(row))
    assert int(e[0, 0]) - 127 == 0 and codes[0, 0] & 0xF == 7


def test_mxfp4_idempotent():
    w = synth.normal_bf16(9, 11, (4, 128), 0.0, 0.02)
    codes, e = F.quantize_mxfp4(w)
    deq = F.dequant_mxfp4(codes, e)
    codes2, e2 = F.quantize_mxfp4(F.f64_to_bf16(deq))
    assert np.array_equal(codes, codes2) and np.array_equal(e, e2)


@pytest.mark.parametrize("std", [0.02, 1.0])
def test_generator_moments_and_reproducible(std):
    a = synth.normal_bf16(0, 1234, 200000, 0.0, std)
    b = synth.normal_bf16(0, 1234, 1000, 0.0, std, start=199000)
    assert np.array_equal(a[199000:], b)               # counter-based: any slice regenerates
    v = F.bf16_to_f64(a)
    assert abs(v.mean()) < 0.01 * std and abs(v.std() / std - 1) < 0.01


def test_generator_draws_match_splitmix64_reference():
    # published SplitMix64 outputs for state 0 (tests/golden/splitmix64_seed0.txt)
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_seed0.txt")
    want = [int(ln, 16) for ln in open(path) if ln.strip() and not ln.startswith("#")]
    lib = synth._get()
    assert [lib.synth_draw(0, i) for i in range(len(want))] == want


def test_generator_normals_restate_box_muller():
    # the normals are Box-Muller on consecutive draw pairs (restated here in Python from the
    # definition: u1 in (0, 1], u2 in [0, 1), cos for even and sin for odd indices), rounded to
    # bf16 by the oracle's own rounding
    import math
    M64 = (1 << 64) - 1
    G = 0x9E3779B97F4A7C15

    def mix(z):
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        return z ^ (z >> 31)

    seed, tid, start, n = 7, synth.tensor_id("w_qkv", 3), 1001, 64
    key = mix(mix((seed + G) & M64) ^ tid)
    draw = lambda i: mix((key + (i + 1) * G) & M64)
    z = []
    for idx in range(start, start + n):
        p = idx >> 1
        u1 = ((draw(2 * p) >> 11) + 1) * 2.0 ** -53
        u2 = (draw(2 * p + 1) >> 11) * 2.0 ** -53
        r = math.sqrt(-2.0 * math.log(u1))
        a = 6.283185307179586476925286766559 * u2
        z.append(r * (math.sin(a) if idx & 1 else math.cos(a)))
    z = np.array(z)
    assert np.array_equal(synth.normal_f64(seed, tid, n, 0.0, 1.0, start=start), z)
    got = synth.normal_bf16(seed, tid, n, 0.25, 0.02, start=start)
    assert np.array_equal(got, F.f64_to_bf16(0.25 + 0.02 * z))
