"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle.

Holds input generation only (counter-based draws, tensor naming, model
shapes); none of the decode step's arithmetic lives here. The header
``gen_core.h`` states the generator's definition; ``gen.c`` runs it on the host
(this wrapper compiles it on first use and returns numpy arrays of bfloat16 bits
(``uint16``) or fp64 values) and ``gen_dev.cu`` on the GPU, writing device
memory directly for weights too large to draw on the host.
"""
from __future__ import annotations

import ctypes
import os
import shutil
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
_CORE = os.path.join(_HERE, "gen_core.h")
_LIB = os.path.join(_HERE, "libsynth.so")
_DEV_SRC = os.path.join(_HERE, "gen_dev.cu")
_DEV_LIB = os.path.join(_HERE, "libsynth_dev.so")
_lock = threading.Lock()
_lib = None
_dev_lib = None


def build(force: bool = False) -> str:
    """Compile ``gen.c`` into ``libsynth.so`` next to it (gcc, OpenMP)."""
    stale = force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(_CORE))
    if stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def build_device(force: bool = False) -> str:
    """Compile ``gen_dev.cu`` into ``libsynth_dev.so`` (nvcc, sm_103a, no fused multiply-add)."""
    stale = force or not os.path.exists(_DEV_LIB) or os.path.getmtime(_DEV_LIB) < max(
        os.path.getmtime(_DEV_SRC), os.path.getmtime(_CORE))
    if stale:
        nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
        tmp = _DEV_LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false", "-std=c++17",
             "-Xcompiler", "-fPIC", "-shared", _DEV_SRC, "-o", tmp]
        )
        os.replace(tmp, _DEV_LIB)
    return _DEV_LIB


def _get_dev():
    global _dev_lib
    with _lock:
        if _dev_lib is None:
            if not os.path.exists(_DEV_LIB):
                raise ImportError(f"{_DEV_LIB} is missing: build it with synth.build_device()")
            lib = ctypes.CDLL(_DEV_LIB)
            u64, dbl, ptr = ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
            lib.synth_normal_bf16_dev.restype = ctypes.c_int
            lib.synth_normal_bf16_dev.argtypes = [u64, u64, u64, u64, dbl, dbl, ptr, ptr]
            _dev_lib = lib
    return _dev_lib


def normal_bf16_dev(out, seed: int, tid: int, mean: float = 0.0, std: float = 1.0, start: int = 0,
                    stream=None) -> None:
    """Fill the contiguous 2-byte device tensor ``out`` with the bf16 bits of draws
    ``start..start+out.numel()-1`` of stream ``tid`` (the values :func:`normal_bf16` returns),
    queued on ``stream`` (a cudaStream_t handle; None: the legacy default stream)."""
    if out.element_size() != 2 or not out.is_contiguous():
        raise ValueError("normal_bf16_dev writes a contiguous tensor of 2-byte elements")
    rc = _get_dev().synth_normal_bf16_dev(seed, tid, start, out.numel(), mean, std, out.data_ptr(), stream)
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16_dev: CUDA error {rc}")


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
