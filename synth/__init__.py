"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle.

Holds input generation only (counter-based draws, tensor naming, model
shapes); none of the decode step's arithmetic lives here. The C source
``gen.c`` states the generator's definition; this wrapper compiles it on first
use and returns numpy arrays of bfloat16 bits (``uint16``) or fp64 values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .configs import (  # noqa: F401
    ModelShape,
    CONFIGS,
    dense_layer_shape,
    dense_2b_shape,
    moe_layer_shape,
    lm_head_shape,
    moe_stack_shape,
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` into ``libsynth.so`` next to it (gcc, OpenMP)."""
    stale = force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, dbl, ptr = ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
            lib.synth_stream_key.restype = u64
            lib.synth_stream_key.argtypes = [u64, u64]
            lib.synth_draw.restype = u64
            lib.synth_draw.argtypes = [u64, u64]
            lib.synth_f64_to_bf16.restype = ctypes.c_uint16
            lib.synth_f64_to_bf16.argtypes = [dbl]
            lib.synth_normal_at.restype = dbl
            lib.synth_normal_at.argtypes = [u64, u64]
            for name in ("synth_normal_bf16", "synth_normal_f64"):
                fn = getattr(lib, name)
                fn.restype = None
                fn.argtypes = [u64, u64, u64, u64, dbl, dbl, ptr]
            lib.synth_bits.restype = None
            lib.synth_bits.argtypes = [u64, u64, u64, u64, ptr]
            _lib = lib
    return _lib


def normal_bf16(seed: int, tid: int, shape, mean: float = 0.0, std: float = 1.0, start: int = 0) -> np.ndarray:
    """bf16 bits of ``mean + std * N(0,1)`` draws ``start..start+n-1`` of stream ``tid``."""
    n = int(np.prod(shape)) if not isinstance(shape, int) else shape
    out = np.empty(n, dtype=np.uint16)
    if n:
        _get().synth_normal_bf16(seed, tid, start, n, mean, std, out.ctypes.data)
    return out.reshape(shape)


def normal_f64(seed: int, tid: int, shape, mean: float = 0.0, std: float = 1.0, start: int = 0) -> np.ndarray:
    n = int(np.prod(shape)) if not isinstance(shape, int) else shape
    out = np.empty(n, dtype=np.float64)
    if n:
        _get().synth_normal_f64(seed, tid, start, n, mean, std, out.ctypes.data)
    return out.reshape(shape)


def bits(seed: int, tid: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    if n:
        _get().synth_bits(seed, tid, start, n, out.ctypes.data)
    return out


def f64_to_bf16(v: float) -> int:
    return int(_get().synth_f64_to_bf16(float(v)))


# ---------------------------------------------------------------- tensor naming
# Every synthetic tensor is its own counter stream, so any tensor (or any
# expert) regenerates independently of the others.
KIND = {
    "embed": 1,
    "attn_norm": 2,
    "w_qkv": 3,
    "w_o": 4,
    "ffn_norm": 5,
    "w_gate": 6,
    "w_up": 7,
    "w_down": 8,
    "w_router": 9,
    "e_gate": 10,
    "e_up": 11,
    "e_down": 12,
    "final_norm": 13,
    "w_lm": 14,
    "k_cache": 15,
    "v_cache": 16,
    "x_in": 17,
    "token": 18,
}


def tensor_id(kind: str, layer: int = 0, expert: int = 0) -> int:
    return ((layer + 1) << 40) | (KIND[kind] << 24) | expert


def start_token(seed: int, vocab: int) -> int:
    """The seeded first token: draw 0 of the ``token`` stream, modulo the vocabulary."""
    return int(bits(seed, tensor_id("token"), 1)[0] % np.uint64(vocab))
