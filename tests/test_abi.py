"""The C ABI library without a GPU: it loads, exports every symbol include/dec.h declares,
rejects bad configs and calls on the host, and its packer writes exactly the bytes of the
oracle's own quantisers (integer work: bit-exact)."""
import ctypes
import os
import re

import numpy as np
import pytest

import synth
from oracle import formats as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def B():
    from persistent_megakernel_gb300 import build
    build.build()
    from persistent_megakernel_gb300 import binding
    binding.lib()
    return binding


def _declared():
    text = open(os.path.join(ROOT, "include", "dec.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dec_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(B):
    names = _declared()
    assert len(names) >= 16
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.EXPORTS) == names


def test_struct_layouts_match_header(B, tmp_path):
    # the binding's structs against the header, measured by a host compile of include/dec.h
    import subprocess
    src = tmp_path / "cfg.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "dec.h"\n'
        'int main(void) { printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(dec_config), '
        'offsetof(dec_config, spin_timeout_ns), offsetof(dec_config, kv_dtype), offsetof(dec_config, attn_window), '
        'sizeof(dec_tensor), offsetof(dec_tensor, values)); return 0; }\n')
    exe = tmp_path / "cfg"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert got == [ctypes.sizeof(B.DecConfig), B.DecConfig.spin_timeout_ns.offset, B.DecConfig.kv_dtype.offset,
                   B.DecConfig.attn_window.offset, ctypes.sizeof(B.DecTensor), B.DecTensor.values.offset]


def test_routing_block_layout_matches_reader(tmp_path):
    # the Python reader's offsets (model.Decoder.routing) against the struct the kernel writes,
    # measured by a host compile of the internal header
    import subprocess
    from persistent_megakernel_gb300.model import Decoder
    src = tmp_path / "rb.cpp"
    src.write_text(
        '#include <cstddef>\n#include <cstdio>\n#include "dec_internal.h"\nusing decimpl::RouteBlock;\n'
        'int main() { std::printf("%zu %zu %zu %zu %zu\\n", sizeof(RouteBlock), offsetof(RouteBlock, expert), '
        'offsetof(RouteBlock, w), offsetof(RouteBlock, topk), offsetof(RouteBlock, topk_w)); }\n')
    exe = tmp_path / "rb"
    csrc = os.path.join(ROOT, "persistent_megakernel_gb300", "csrc")
    from persistent_megakernel_gb300 import build
    cuda_inc = os.path.join(build._cuda_home(build._nvcc()), "include")
    subprocess.check_call(["g++", "-std=c++17", "-I", csrc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                           str(src), "-o", str(exe)])
    size, expert, w, topk, topk_w = map(int, subprocess.check_output([str(exe)]).split())
    S, T, K = Decoder.ROUTE_SLOTS, Decoder.ROUTE_TOKENS, Decoder.ROUTE_K
    assert size == 4 * Decoder.ROUTE_WORDS == 920
    assert (expert, w, topk, topk_w) == (4, 4 * (1 + S), 4 * (1 + S + T * S), 4 * (1 + S + T * S + T * K))


def _cfg(B, **kw):
    c = B.DecConfig()
    base = dict(n_layers=1, hidden=256, n_q=4, n_kv=2, head_dim=128, ffn=512, vocab=100, kv_capacity=64, max_verify=1,
                embedding=1, final_norm=1, rms_eps=1e-6, rope_base=1e4, num_ctas=8)
    base.update(kw)
    for k, v in base.items():
        setattr(c, k, v)
    return c


def test_workspace_bytes_and_config_validation(B):
    assert B.dec_workspace_bytes(_cfg(B)) > 0
    bad = [dict(hidden=100), dict(head_dim=64), dict(n_kv=3), dict(max_verify=5), dict(ffn=12),
           dict(n_q=32, n_kv=2), dict(ffn=0, n_experts=8, top_k=9, moe_inter=64), dict(embedding=1, vocab=0),
           dict(ffn=0, n_experts=8, top_k=2, moe_inter=48), dict(mode=7)]
    for b in bad:
        assert B.dec_workspace_bytes(_cfg(B, **b)) == 0, b
        assert "invalid config" in B.dec_last_error()


def test_init_rejects_bad_arguments(B):
    out = ctypes.c_void_p()
    L = B.lib()
    assert L.dec_init(ctypes.byref(_cfg(B)), None, None, ctypes.byref(out)) == B.DEC_ERR_INVALID_ARG
    assert L.dec_init(ctypes.byref(_cfg(B)), None, 0x1001, ctypes.byref(out)) == B.DEC_ERR_INVALID_ARG
    assert "aligned" in B.dec_last_error()
    assert L.dec_init(ctypes.byref(_cfg(B, hidden=96)), None, 0x1000, ctypes.byref(out)) == B.DEC_ERR_INVALID_ARG
    assert L.dec_step(None, 0, None, 0, None, None) == B.DEC_ERR_INVALID_ARG
    assert L.dec_reset(None) == B.DEC_ERR_INVALID_ARG


def test_packed_bytes(B):
    assert B.dec_packed_bytes(B.DEC_BF16, 3, 16) == (96, 0)
    assert B.dec_packed_bytes(B.DEC_FP8_E4M3_ROWSCALE, 3, 32) == (96, 12)
    assert B.dec_packed_bytes(B.DEC_MXFP4, 4, 64) == (128, 8)
    with pytest.raises(B.DecError):
        B.dec_packed_bytes(B.DEC_MXFP4, 4, 48)


def test_fp8_packer_equals_oracle_quantiser(B):
    w = synth.normal_bf16(3, 501, (64, 2560), 0.0, 0.02)
    w[5] = 0
    w[6, :] = 0x8000                                   # negative zeros
    w[7, 3] = 0x4480                                   # 1024.0: a large outlier
    vals = np.empty(64 * 2560, np.uint8)
    scales = np.empty(64, np.float32)
    B.dec_pack(B.DEC_FP8_E4M3_ROWSCALE, w, 64, 2560, vals, scales)
    codes, s = F.quantize_fp8_rows(w)
    assert np.array_equal(s, scales)
    assert np.array_equal(codes.reshape(-1), vals)


def test_mxfp4_packer_equals_oracle_quantiser(B):
    w = synth.normal_bf16(4, 502, (48, 768), 0.0, 0.02)
    w[1, 32:64] = 0
    w[2, 0] = 0x0001                                   # bf16 subnormal
    w[3, 64:96] = synth.normal_bf16(4, 503, 32, 0.0, 1e-30)   # tiny block
    vals = np.empty(48 * 384, np.uint8)
    scales = np.empty(48 * 24, np.uint8)
    B.dec_pack(B.DEC_MXFP4, w, 48, 768, vals, scales)
    codes, e = F.quantize_mxfp4(w)
    assert np.array_equal(e.reshape(-1), scales)
    assert np.array_equal(codes.reshape(-1), vals)


def _finite_bf16_upto(limit_bits: int) -> np.ndarray:
    """Every finite bf16 bit pattern (both signs) whose magnitude is at most limit_bits."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mag = allb & 0x7FFF
    return allb[(mag < 0x7F80) & (mag <= limit_bits)]


def _bits(x: float) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0] >> 16)


@pytest.mark.parametrize("amax", [1.0, 448.0, 3e-5, 1e30, 0.02, 7.5, 3.3e38, 2.0 ** -130])
def test_fp8_packer_every_bf16_value(B, amax):
    # rows [amax, v ...] with every finite |v| <= amax: each e4m3 code and rounding tie is reached
    vals = _finite_bf16_upto(_bits(amax))
    cols = 512
    rows = -(-len(vals) // (cols - 1))
    w = np.zeros((rows, cols), np.uint16)
    w[:, 0] = _bits(amax)
    flat = np.zeros(rows * (cols - 1), np.uint16)
    flat[:len(vals)] = vals
    w[:, 1:] = flat.reshape(rows, cols - 1)
    out = np.empty(rows * cols, np.uint8)
    sc = np.empty(rows, np.float32)
    B.dec_pack(B.DEC_FP8_E4M3_ROWSCALE, w, rows, cols, out, sc)
    codes, s = F.quantize_fp8_rows(w)
    assert np.array_equal(s, sc)
    assert np.array_equal(codes.reshape(-1), out)


@pytest.mark.parametrize("bmax", [1.0, 6.0, 5.0, 0.75, 2.0 ** -133, 2.0 ** -126, 1e30, 3.3e38])
def test_mxfp4_packer_every_bf16_value(B, bmax):
    # blocks [bmax, 31 values with |v| <= bmax], the maximum at a seeded position of each block
    vals = _finite_bf16_upto(_bits(bmax))
    nb = -(-len(vals) // 31)
    nb += (-nb) % 32
    blocks = np.zeros((nb, 32), np.uint16)
    flat = np.zeros(nb * 31, np.uint16)
    flat[:len(vals)] = vals
    blocks[:, 1:] = flat.reshape(nb, 31)
    blocks[:, 0] = _bits(bmax)
    perm = np.argsort(synth.bits(7, 506, nb * 32).reshape(nb, 32), axis=1)
    blocks = np.take_along_axis(blocks, perm, axis=1)
    w = np.ascontiguousarray(blocks.reshape(-1, 1024))
    rows = w.shape[0]
    out = np.empty(rows * 512, np.uint8)
    sc = np.empty(rows * 32, np.uint8)
    B.dec_pack(B.DEC_MXFP4, w, rows, 1024, out, sc)
    codes, e = F.quantize_mxfp4(w)
    assert np.array_equal(e.reshape(-1), sc)
    assert np.array_equal(codes.reshape(-1), out)


@pytest.mark.parametrize("scale", [1.0, 0.3, 3.3, 2.0 ** -5])
def test_kv_fp8_packer_equals_oracle_quantiser(B, scale):
    vals = _finite_bf16_upto(0x7F7F)                     # every finite bf16 value
    out = np.empty(vals.size, np.uint8)
    B.dec_pack_kv_fp8(vals, vals.size, scale, out)
    want = F.quantize_kv_fp8(F.bf16_to_f64(vals), scale)
    assert np.array_equal(out, want)


def test_kv_fp8_entry_points_reject_bad_arguments(B):
    L = B.lib()
    assert L.dec_set_kv_scales(None, None) == B.DEC_ERR_INVALID_ARG
    v = np.zeros(4, np.uint16)
    o = np.zeros(4, np.uint8)
    assert L.dec_pack_kv_fp8(v.ctypes.data, 4, ctypes.c_float(0.0), o.ctypes.data) == B.DEC_ERR_INVALID_ARG
    assert L.dec_pack_kv_fp8(None, 4, ctypes.c_float(1.0), o.ctypes.data) == B.DEC_ERR_INVALID_ARG
    assert L.dec_pack_kv_fp8_device(None, 4, ctypes.c_float(1.0), 0x10000, None) == B.DEC_ERR_INVALID_ARG
    assert B.dec_workspace_bytes(_cfg(B, kv_dtype=7)) == 0


def test_device_packer_rejects_bad_arguments(B):
    # checked on the host before any launch, so no GPU is needed
    L = B.lib()
    ok = 0x10000
    assert L.dec_pack_device(B.DEC_MXFP4, None, 4, 64, ok, ok, None) == B.DEC_ERR_INVALID_ARG
    assert L.dec_pack_device(B.DEC_MXFP4, ok, 4, 64, ok, None, None) == B.DEC_ERR_INVALID_ARG
    assert L.dec_pack_device(B.DEC_MXFP4, ok + 8, 4, 64, ok, ok, None) == B.DEC_ERR_INVALID_ARG
    assert L.dec_pack_device(B.DEC_MXFP4, ok, 4, 48, ok, ok, None) == B.DEC_ERR_SHAPE
    assert L.dec_pack_device(B.DEC_FP8_E4M3_ROWSCALE, ok, 4, 64, ok, ok + 2, None) == B.DEC_ERR_INVALID_ARG
    assert L.dec_pack_device(7, ok, 4, 64, ok, ok, None) == B.DEC_ERR_DTYPE
    assert L.dec_pack_pair_device(B.DEC_BF16, ok, None, 4, 64, ok, None, None) == B.DEC_ERR_INVALID_ARG
    assert "aligned" in B.dec_last_error() or "null" in B.dec_last_error()


def test_pair_packer_interleaves_rows(B):
    a = synth.normal_bf16(5, 504, (6, 64), 0.0, 0.02)
    b = synth.normal_bf16(5, 505, (6, 64), 0.0, 0.02)
    vals = np.empty(12 * 32, np.uint8)
    sc = np.empty(12 * 2, np.uint8)
    B.dec_pack_pair(B.DEC_MXFP4, a, b, 6, 64, vals, sc)
    inter = np.empty((12, 64), np.uint16)
    inter[0::2], inter[1::2] = a, b
    codes, e = F.quantize_mxfp4(inter)
    assert np.array_equal(codes.reshape(-1), vals) and np.array_equal(e.reshape(-1), sc)
    out = np.empty(12 * 64, np.uint16)
    B.dec_pack_pair(B.DEC_BF16, a, b, 6, 64, out, None)
    assert np.array_equal(out.reshape(12, 64), inter)


def test_drop_op_only_in_per_op_mode():
    """The failure-injection hook refuses persistent contexts and ops outside the step (no GPU
    work: the checks come before any launch)."""
    from persistent_megakernel_gb300 import binding as B
    from persistent_megakernel_gb300.model import make_config
    from synth.configs import ModelShape
    import torch
    s = ModelShape("t", n_layers=1, hidden=256, n_q=4, n_kv=2, ffn=352, vocab=1000, kv_prefill=8)
    for mode, op, code in (("persistent", 0, B.DEC_ERR_STATE), ("per_op", 99, B.DEC_ERR_INVALID_ARG)):
        cfg = make_config(s, 16, 1, mode, num_ctas=3)
        n = B.dec_workspace_bytes(cfg)
        ws = torch.zeros(n + 256, dtype=torch.uint8)
        off = (-ws.data_ptr()) % 256
        try:
            ctx = B.dec_init(cfg, None, ws[off:off + n])
        except B.DecError:
            pytest.skip("dec_init needs a CUDA runtime")
        try:
            with pytest.raises(B.DecError) as e:
                B.dec_debug_drop_op(ctx, op)
            assert e.value.code == code
        finally:
            B.dec_free(ctx)


@pytest.mark.parametrize("hidden,n_q,n_kv,ffn,experts", [(1024, 8, 2, 2816, 0), (2560, 20, 4, 6912, 0),
                                                          (2560, 20, 4, 0, 512), (4096, 32, 8, 11008, 0),
                                                          (256, 4, 2, 352, 0)])
@pytest.mark.parametrize("m", [1, 2, 4])
@pytest.mark.parametrize("ctas", [1, 3, 152, 304])
def test_workspace_sizing_sweep(hidden, n_q, n_kv, ffn, experts, m, ctas):
    """Host-side layout for a sweep of shapes, windows and grid sizes: either a workspace size
    or a clear shape error (no device needed when the grid size is given)."""
    from persistent_megakernel_gb300 import binding as B
    from persistent_megakernel_gb300.model import make_config
    from synth.configs import ModelShape
    s = ModelShape("sweep", n_layers=2, hidden=hidden, n_q=n_q, n_kv=n_kv, ffn=ffn, n_experts=experts,
                   top_k=8 if experts else 0, moe_inter=768 if experts else 0, n_shared=1 if experts else 0,
                   vocab=32000, kv_prefill=128, embedding=True)
    cfg = make_config(s, 256, m, "persistent", num_ctas=ctas)
    n = B.dec_workspace_bytes(cfg)
    if n == 0:
        assert "shared memory" in B.dec_last_error(), B.dec_last_error()
    else:
        # at least the tagged hidden stream and the logits
        assert n >= (2 * s.n_layers + 1) * m * hidden * 8 + m * s.vocab * 4
