"""The roofline helper reproduces the worked arithmetic the pages print
(tests/golden/roofline_pages.txt) and the per-token byte counts of the workloads."""
import os

import pytest

from persistent_megakernel_gb300 import roofline as R
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "roofline_pages.txt")


def _rows():
    for ln in open(GOLDEN):
        if ln.strip() and not ln.startswith("#"):
            kind, args, result, _cite = [t.strip() for t in ln.split("|")]
            kv = dict(a.split("=") for a in args.split())
            yield kind, {k: float(v) for k, v in kv.items()}, [float(x) for x in result.split()]


@pytest.mark.parametrize("kind,a,want", list(_rows()))
def test_pages_arithmetic(kind, a, want):
    close = lambda x, y: abs(x - y) <= 0.01 * y            # the pages round their results
    if kind == "bound":
        got = R.bound_tokens_per_s(a["bw_tbs"] * 1e12, a["weight_gb"] * 1e9, a["kv_gb"] * 1e9, a["beta"])
        assert close(got, want[0])
    elif kind == "launch":
        ov = R.launch_overhead_us(a["launch_us"], a["kernels"], int(a["layers"]))
        assert close(ov, want[0]) and close(R.ceiling_tokens_per_s(ov), want[1])
    elif kind == "budget":
        assert close(R.budget_us(a["tok_s"]), want[0])
    elif kind == "spec":
        assert close(a["accepted"] / (a["step_ms"] * 1e-3), want[0])


def test_workload_bytes():
    c2 = synth.dense_2b_shape()
    b = R.algorithmic_bytes(c2, 4096)
    # 28 layers x (qkv 3584x2560 + o 2560^2 + 3 x 6912x2560) bf16 + head 32768x2560 + KV 4097 rows
    w = 28 * 2 * (3584 * 2560 + 2560 * 2560 + 3 * 6912 * 2560) + 2 * 32768 * 2560
    kv = 28 * 2 * 4 * 128 * 2 * 4097
    assert abs(b - (w + kv)) < 28 * 3 * 2 * 2560 + 10       # norm gains and the embedding row
    assert 4.25e9 < b < 4.26e9
    c4 = synth.lm_head_shape("fp8")
    assert R.algorithmic_bytes(c4, 0) == 157184 * 2560 + 4 * 157184
    c3 = synth.moe_layer_shape()
    per_expert = 1536 * (1280 + 80) + 2560 * (384 + 24)
    assert R.algorithmic_bytes(c3, 0) == 2 * 512 * 2560 + 2 * 2560 + 9 * per_expert


def test_traffic_figures_follow_their_sources(monkeypatch):
    """bench.py reports a committed DRAM figure only for the kernel sources it was captured on
    (their sha256 is stored beside it): same sources, the figure; changed sources, null."""
    import json
    import os
    import bench
    recs = json.load(open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")))
    assert {"dense_2b", "moe_stack", "dense_2b_verify4", "moe_stack_verify4"} <= set(recs)
    for key, rec in recs.items():
        assert rec["dram_bytes_per_step"] > 0 and len(rec["source_sha256"]) == 64 and rec["capture"]
        monkeypatch.setattr(bench, "sources_sha256", lambda files, s=rec["source_sha256"]: s)
        assert bench.ncu_traffic(key, bench.kernel_sources()) == rec["dram_bytes_per_step"]
        monkeypatch.setattr(bench, "sources_sha256", lambda files: "0" * 64)
        assert bench.ncu_traffic(key, bench.kernel_sources()) is None
    assert bench.ncu_traffic("no_such_workload", bench.kernel_sources()) is None
