"""ctypes binding of ``include/dec.h``: the same names, argument marshalling only.

Loading fails loudly when ``libdec.so`` has not been built (``persistent_megakernel_gb300.build``);
there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# DEC_LIB_VARIANT=trace selects the self-timing build (libdec_trace.so)
_VARIANT = os.environ.get("DEC_LIB_VARIANT", "")
LIB_PATH = os.path.join(HERE, f"libdec_{_VARIANT}.so" if _VARIANT else "libdec.so")

DEC_OK = 0
DEC_ERR_INVALID_ARG = 1
DEC_ERR_SHAPE = 2
DEC_ERR_DTYPE = 3
DEC_ERR_STATE = 4
DEC_ERR_CUDA = 5
DEC_ERR_TIMEOUT = 6
DEC_ERR_CAPACITY = 7

DEC_BF16 = 0
DEC_FP8_E4M3_ROWSCALE = 1
DEC_MXFP4 = 2
DEC_FP8_E4M3 = 3

DEC_MODE_PERSISTENT = 0
DEC_MODE_PER_OP = 1
DEC_MODE_PER_OP_GRAPH = 2

(DEC_T_EMBED, DEC_T_ATTN_NORM, DEC_T_WQKV, DEC_T_WO, DEC_T_FFN_NORM, DEC_T_WGATEUP, DEC_T_WDOWN, DEC_T_WROUTER,
 DEC_T_EXPERT_GATEUP, DEC_T_EXPERT_DOWN, DEC_T_FINAL_NORM, DEC_T_LM_HEAD) = range(12)

# every symbol include/dec.h declares
EXPORTS = ("dec_workspace_bytes", "dec_init", "dec_load_weights", "dec_set_kv_cache", "dec_step", "dec_generate",
           "dec_verify", "dec_debug_buffers", "dec_reset", "dec_sync", "dec_last_launch_count", "dec_last_error",
           "dec_free", "dec_packed_bytes", "dec_pack", "dec_pack_pair", "dec_pack_device", "dec_pack_pair_device",
           "dec_set_kv_scales", "dec_pack_kv_fp8", "dec_pack_kv_fp8_device", "dec_trace_buffer", "dec_lm_head_noalloc",
           "dec_debug_drop_op", "dec_run_layer", "dec_lm_head")


class DecConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layers", "hidden", "n_q", "n_kv", "head_dim", "ffn", "n_experts", "top_k", "moe_inter", "n_shared",
        "vocab", "kv_capacity", "max_verify", "embedding", "final_norm")] + [
        ("rms_eps", ctypes.c_float), ("rope_base", ctypes.c_float),
        ("lm_head_dtype", ctypes.c_int), ("expert_dtype", ctypes.c_int), ("mode", ctypes.c_int),
        ("spin_timeout_ns", ctypes.c_uint64), ("num_ctas", ctypes.c_int), ("kv_dtype", ctypes.c_int),
        ("attn_window", ctypes.c_int)]


class DecTensor(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("layer", ctypes.c_int), ("dtype", ctypes.c_int), ("rows", ctypes.c_int),
                ("cols", ctypes.c_int), ("values", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


class DecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dec status {code}: {msg}")
        self.code = code


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with persistent_megakernel_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
        sig = {
            "dec_workspace_bytes": (SZ, [ctypes.POINTER(DecConfig)]),
            "dec_init": (I, [ctypes.POINTER(DecConfig), P, P, ctypes.POINTER(P)]),
            "dec_load_weights": (I, [P, ctypes.POINTER(DecTensor), I]),
            "dec_set_kv_cache": (I, [P, P, P]),
            "dec_set_kv_scales": (I, [P, P]),
            "dec_pack_kv_fp8": (I, [P, SZ, ctypes.c_float, P]),
            "dec_pack_kv_fp8_device": (I, [P, SZ, ctypes.c_float, P, P]),
            "dec_step": (I, [P, ctypes.c_int32, P, ctypes.c_int32, P, P]),
            "dec_generate": (I, [P, ctypes.c_int32, ctypes.c_int32, I, P]),
            "dec_run_layer": (I, [P, I, P, I, ctypes.c_int32, P, P, P]),
            "dec_lm_head": (I, [P, P, I, P, P]),
            "dec_verify": (I, [P, P, P, I, ctypes.c_int32, P, P, P]),
            "dec_debug_buffers": (I, [P, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P)]),
            "dec_trace_buffer": (I, [P, ctypes.POINTER(P), ctypes.POINTER(I), ctypes.POINTER(I)]),
            "dec_reset": (I, [P]),
            "dec_sync": (I, [P]),
            "dec_last_launch_count": (I, [P]),
            "dec_debug_drop_op": (I, [P, I]),
            "dec_last_error": (ctypes.c_char_p, []),
            "dec_free": (None, [P]),
            "dec_packed_bytes": (I, [I, I, I, ctypes.POINTER(SZ), ctypes.POINTER(SZ)]),
            "dec_pack": (I, [I, P, I, I, P, P]),
            "dec_pack_pair": (I, [I, P, P, I, I, P, P]),
            "dec_pack_device": (I, [I, P, I, I, P, P, P]),
            "dec_pack_pair_device": (I, [I, P, P, I, I, P, P, P]),
            "dec_lm_head_noalloc": (I, [I, I, I, I, ctypes.c_float, P, P, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def dec_last_error() -> str:
    return lib().dec_last_error().decode()


def check(code: int):
    if code != DEC_OK:
        raise DecError(code, dec_last_error())


def _p(x):
    """device / host pointer of a torch tensor, numpy array, int or None"""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(type(x))


def dec_workspace_bytes(cfg: DecConfig) -> int:
    return lib().dec_workspace_bytes(ctypes.byref(cfg))


def dec_init(cfg: DecConfig, stream, workspace) -> int:
    out = ctypes.c_void_p()
    check(lib().dec_init(ctypes.byref(cfg), _p(stream), _p(workspace), ctypes.byref(out)))
    return out.value


def dec_load_weights(ctx: int, tensors) -> None:
    arr = (DecTensor * len(tensors))(*tensors)
    check(lib().dec_load_weights(ctx, arr, len(tensors)))


def dec_set_kv_cache(ctx: int, k, v) -> None:
    check(lib().dec_set_kv_cache(ctx, _p(k), _p(v)))


def dec_step(ctx: int, token: int, hidden, pos: int, logits=None, want_argmax=True):
    am = ctypes.c_int32(-1)
    check(lib().dec_step(ctx, token, _p(hidden), pos, _p(logits), ctypes.byref(am) if want_argmax else None))
    return am.value if want_argmax else None


def dec_run_layer(ctx: int, layer: int, h_in, m: int, pos: int, h_out, topk_idx=None, topk_w=None) -> None:
    check(lib().dec_run_layer(ctx, layer, _p(h_in), m, pos, _p(h_out), _p(topk_idx), _p(topk_w)))


def dec_lm_head(ctx: int, h_in, m: int, logits=None, want_argmax=True):
    am = (ctypes.c_int32 * 4)()
    check(lib().dec_lm_head(ctx, _p(h_in), m, _p(logits), am if want_argmax else None))
    return list(am)[:m] if want_argmax else None


def dec_generate(ctx: int, token: int, pos: int, n: int, tokens_out=None) -> None:
    check(lib().dec_generate(ctx, token, pos, n, _p(tokens_out)))


def dec_verify(ctx: int, tokens, hidden, k: int, pos: int, logits=None, want_argmax=True):
    """Returns (argmaxes, accepted count); with want_argmax False the call does not wait and
    returns None."""
    am = (ctypes.c_int32 * 4)()
    nacc = ctypes.c_int32(0)
    toks = (ctypes.c_int32 * 4)(*(list(tokens) + [0] * (4 - len(tokens)))) if tokens is not None else None
    if not want_argmax:
        check(lib().dec_verify(ctx, toks, _p(hidden), k, pos, _p(logits), None, None))
        return None
    check(lib().dec_verify(ctx, toks, _p(hidden), k, pos, _p(logits), am, ctypes.byref(nacc)))
    return list(am)[:k], nacc.value


def dec_debug_buffers(ctx: int):
    h, q, r = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    check(lib().dec_debug_buffers(ctx, ctypes.byref(h), ctypes.byref(q), ctypes.byref(r)))
    return h.value, q.value, r.value


def dec_trace_buffer(ctx: int):
    """(device pointer or None, n_ctas, n_ops) of the self-timing records."""
    r, c, o = ctypes.c_void_p(), ctypes.c_int(), ctypes.c_int()
    check(lib().dec_trace_buffer(ctx, ctypes.byref(r), ctypes.byref(c), ctypes.byref(o)))
    return r.value, c.value, o.value


def dec_reset(ctx: int) -> None:
    check(lib().dec_reset(ctx))


def dec_sync(ctx: int) -> None:
    check(lib().dec_sync(ctx))


def dec_debug_drop_op(ctx: int, op: int) -> None:
    check(lib().dec_debug_drop_op(ctx, op))


def dec_last_launch_count(ctx: int) -> int:
    return lib().dec_last_launch_count(ctx)


def dec_free(ctx: int) -> None:
    lib().dec_free(ctx)


def dec_packed_bytes(dtype: int, rows: int, cols: int):
    v, s = ctypes.c_size_t(), ctypes.c_size_t()
    check(lib().dec_packed_bytes(dtype, rows, cols, ctypes.byref(v), ctypes.byref(s)))
    return v.value, s.value


def dec_lm_head_noalloc(hidden: int, vocab: int, dtype: int, m: int, rms_eps: float, hidden_dev, final_norm_dev,
                        w_values_dev, w_scales_dev, logits_dev, argmax_dev, stream) -> None:
    """The LM head for callers that cannot allocate device memory (all buffers are the caller's;
    the library's static scratch serves the kernel). Synchronises the stream."""
    check(lib().dec_lm_head_noalloc(hidden, vocab, dtype, m, rms_eps, _p(hidden_dev), _p(final_norm_dev),
                                    _p(w_values_dev), _p(w_scales_dev), _p(logits_dev), _p(argmax_dev), _p(stream)))


def dec_pack(dtype: int, w_bf16, rows: int, cols: int, out_values, out_scales=None) -> None:
    check(lib().dec_pack(dtype, _p(w_bf16), rows, cols, _p(out_values), _p(out_scales)))


def dec_pack_pair(dtype: int, a_bf16, b_bf16, rows: int, cols: int, out_values, out_scales=None) -> None:
    check(lib().dec_pack_pair(dtype, _p(a_bf16), _p(b_bf16), rows, cols, _p(out_values), _p(out_scales)))


def dec_pack_device(dtype: int, w_bf16_dev, rows: int, cols: int, out_values_dev, out_scales_dev=None, stream=None) -> None:
    """dec_pack on device buffers, queued on `stream` (a cudaStream_t handle or None)."""
    check(lib().dec_pack_device(dtype, _p(w_bf16_dev), rows, cols, _p(out_values_dev), _p(out_scales_dev), _p(stream)))


def dec_pack_pair_device(dtype: int, a_dev, b_dev, rows: int, cols: int, out_values_dev, out_scales_dev=None,
                         stream=None) -> None:
    check(lib().dec_pack_pair_device(dtype, _p(a_dev), _p(b_dev), rows, cols, _p(out_values_dev), _p(out_scales_dev),
                                     _p(stream)))


def dec_set_kv_scales(ctx: int, scales_dev) -> None:
    check(lib().dec_set_kv_scales(ctx, _p(scales_dev)))


def dec_pack_kv_fp8(bf16, n: int, scale: float, out) -> None:
    check(lib().dec_pack_kv_fp8(_p(bf16), n, scale, _p(out)))


def dec_pack_kv_fp8_device(bf16_dev, n: int, scale: float, out_dev, stream=None) -> None:
    check(lib().dec_pack_kv_fp8_device(_p(bf16_dev), n, scale, _p(out_dev), _p(stream)))
