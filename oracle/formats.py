"""Number formats of the oracle: bfloat16, FP8 e4m3 (fn), FP4 e2m1, E8M0, and the quantisers.

Test infrastructure only (see the package docstring).

Each decoder is written from the format's definition (sign, exponent field,
bias, mantissa, subnormals, special codes); each quantiser follows the rule
stated in its docstring. Formats: bfloat16 (8-bit exponent, bias 127, 7-bit
mantissa); OCP 8-bit floating point e4m3 "fn" variant (bias 7, no infinities,
S.1111.111 is NaN, max 448); OCP Microscaling (MX) v1.0 element type FP4 e2m1
(bias 1, max 6) and scale type E8M0 (2^(e-127), 0xFF is NaN). MXFP4 and the
per-row FP8 LM head are the weight encodings named by the Ling-3.0-flash DGX
Spark article ("optimisation 1: Humming MXFP4 MoE", "optimisation 2: online FP8
LM head").
"""
from __future__ import annotations

import numpy as np

# ------------------------------------------------------------------ decoders


def bf16_to_f64(bits) -> np.ndarray:
    """Value of bfloat16 codes: (-1)^s * 2^(e-127) * 1.m  (e>0), (-1)^s * 2^-126 * 0.m (e=0)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = np.where(b >> 15, -1.0, 1.0)
    e = (b >> 7) & 0xFF
    m = (b & 0x7F).astype(np.float64)
    normal = s * np.ldexp(1.0 + m / 128.0, (e - 127).astype(np.int32))
    sub = s * np.ldexp(m / 128.0, -126)
    out = np.where(e == 0, sub, normal)
    special = e == 0xFF
    if np.any(special):
        out = np.where(special & (m == 0), s * np.inf, out)
        out = np.where(special & (m != 0), np.nan, out)
    return out


def e4m3_to_f64(codes) -> np.ndarray:
    """Value of e4m3fn codes: bias 7, 3 mantissa bits, subnormals 2^-6 * 0.m, 0x7F/0xFF NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = s * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int32))
    sub = s * np.ldexp(m / 8.0, -6)
    out = np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def e2m1_to_f64(codes) -> np.ndarray:
    """Value of 4-bit e2m1 codes (low 4 bits used): bias 1, 1 mantissa bit, subnormal 0.5 * m."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64) & 0xF
    s = np.where(c >> 3, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    normal = s * np.ldexp(1.0 + m / 2.0, (e - 1).astype(np.int32))
    sub = s * (m / 2.0)
    return np.where(e == 0, sub, normal)


def e8m0_to_f64(codes) -> np.ndarray:
    """Value of E8M0 scale codes: 2^(e-127), 0xFF NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int32)
    return np.where(c == 0xFF, np.nan, np.ldexp(1.0, c - 127))


# ------------------------------------------------------------------ rounding helpers


def _grid_round(vals: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid point to each |value| (grid ascending, index = code);
    an exact tie goes to the even index (round half to even on codes). Values beyond the
    last grid point take the last index (saturation)."""
    a = np.abs(vals)
    hi = np.searchsorted(grid, a, side="left")          # first grid >= a
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    dlo = a - grid[lo]
    dhi = grid[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(a >= grid[-1], len(grid) - 1, idx)
    idx = np.where(a <= grid[0], 0, idx)
    return idx


def f64_to_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 (ties to even code), as stored in the KV cache."""
    x = np.asarray(x, dtype=np.float64)
    # every positive finite bf16 code in ascending order equals its own index
    pos_codes = np.arange(0x7F80, dtype=np.uint16)
    grid = bf16_to_f64(pos_codes)
    idx = _grid_round(x, grid)
    # beyond the largest finite value by at least half an ulp the result is infinity
    big = np.abs(x) >= grid[-1] + (grid[-1] - grid[-2]) / 2
    idx = np.where(big, 0x7F80, idx)
    sign = (np.signbit(x)).astype(np.uint16) << 15
    return (idx.astype(np.uint16) | sign).astype(np.uint16)


_E4M3_POS = e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))   # codes 0..126, ascending, max 448
_E2M1_POS = e2m1_to_f64(np.arange(8, dtype=np.uint8))      # 0, .5, 1, 1.5, 2, 3, 4, 6


def round_e4m3_satfinite(x) -> np.ndarray:
    """e4m3fn code nearest to x (ties to even code), saturated to +-448; sign bit = sign of x."""
    x = np.asarray(x, dtype=np.float64)
    idx = _grid_round(x, _E4M3_POS)
    return (idx.astype(np.uint8) | (np.signbit(x).astype(np.uint8) << 7)).astype(np.uint8)


def round_e2m1_satfinite(x) -> np.ndarray:
    """e2m1 code nearest to x (ties to even code), saturated to +-6; sign bit = sign of x."""
    x = np.asarray(x, dtype=np.float64)
    idx = _grid_round(x, _E2M1_POS)
    return (idx.astype(np.uint8) | (np.signbit(x).astype(np.uint8) << 3)).astype(np.uint8)


# ------------------------------------------------------------------ quantisers

FP8_MAX = 448.0


def quantize_fp8_rows(w_bf16) -> tuple[np.ndarray, np.ndarray]:
    """Dynamic per-row FP8 of a bf16 matrix [R, C] (Ling-3.0-flash DGX Spark article,
    "optimisation 2: online FP8 LM head": the bf16 head is quantised to FP8 at load time).

    Per row r, in IEEE fp32 (the precision the packer computes in):
      s_r = amax_r / 448  (a zero row takes s_r = 1);
      q   = e4m3_satfinite_RNE(w / s_r)   with the fp32 division correctly rounded.
    Returns (codes uint8 [R, C], scales float32 [R]); the dequantised weight is s_r * e4m3(q).
    """
    w32 = bf16_to_f64(w_bf16).astype(np.float32)         # exact: bf16 is a subset of fp32
    amax = np.max(np.abs(w32), axis=1)
    s = (amax / np.float32(FP8_MAX)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    y = (w32 / s[:, None]).astype(np.float32)            # fp32 correctly-rounded division
    return round_e4m3_satfinite(y.astype(np.float64)), s


def dequant_fp8_rows(codes, scales) -> np.ndarray:
    return e4m3_to_f64(codes) * np.asarray(scales, np.float64)[:, None]


MX_BLOCK = 32
E2M1_EMAX = 2      # exponent of e2m1's largest normal (6 = 1.5 * 2^2)


def quantize_mxfp4(w_bf16) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4 of a bf16 matrix [R, C] along C in blocks of 32 (OCP MX v1.0 conversion rule).

    Per block: X = 2^(floor(log2 amax) - 2) stored as E8M0 e = floor(log2 amax) - 2 + 127
    clamped to [0, 254]; each element code = e2m1_satfinite_RNE(v / X) (exact division by a
    power of two), sign bit = sign of v. A block of zeros takes e = 0 and +0 codes.
    Two codes per byte, the even element in the low nibble.
    Returns (codes uint8 [R, C/2], scales uint8 [R, C/32]).
    """
    v = bf16_to_f64(w_bf16)
    R, C = v.shape
    assert C % MX_BLOCK == 0
    blk = v.reshape(R, C // MX_BLOCK, MX_BLOCK)
    amax = np.max(np.abs(blk), axis=2)
    _, ex = np.frexp(amax)                     # amax = f * 2^ex, f in [0.5, 1) -> floor(log2) = ex - 1
    e = np.where(amax > 0, ex - 1 - E2M1_EMAX + 127, 0)
    e = np.clip(e, 0, 254).astype(np.int64)
    X = np.ldexp(1.0, (e - 127).astype(np.int32))
    q = round_e2m1_satfinite(blk / X[:, :, None]).reshape(R, C)
    packed = (q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)
    return packed.astype(np.uint8), e.astype(np.uint8)


def dequant_mxfp4(codes, scales) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    R, half = codes.shape
    q = np.empty((R, half * 2), np.uint8)
    q[:, 0::2] = codes & 0xF
    q[:, 1::2] = codes >> 4
    vals = e2m1_to_f64(q).reshape(R, -1, MX_BLOCK)
    return (vals * e8m0_to_f64(scales)[:, :, None]).reshape(R, half * 2)


# ------------------------------------------------------------------ FP8 KV cache


def quantize_kv_fp8(x, scale) -> np.ndarray:
    """e4m3fn codes of KV-cache entries ``x`` under ``scale`` s (Kimi-K3 on 8xB300, section on
    the log warnings: both engines keep the KV cache as fp8_e4m3, and without a calibrated
    scaling factor they fall back to a scale of 1.0). The stored value is s * e4m3(q) with
    q = e4m3_satfinite_RNE(x / s); x is taken in fp32 and the division is IEEE fp32 (the
    precision the kernel computes a new key or value in). ``scale`` (fp32, > 0) broadcasts
    against x, e.g. one scale per kv head."""
    x32 = np.asarray(x, np.float64).astype(np.float32)
    s32 = np.asarray(scale, np.float32)
    y = (x32 / s32).astype(np.float32)
    return round_e4m3_satfinite(y.astype(np.float64))


def dequant_kv_fp8(codes, scale) -> np.ndarray:
    """Value of FP8 KV-cache codes: s * e4m3(q), ``scale`` broadcasting against the codes."""
    return e4m3_to_f64(codes) * np.asarray(scale, np.float32).astype(np.float64)
