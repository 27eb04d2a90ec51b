"""Benchmark: batch-1 greedy decode of the 2B-class dense decoder on one GB300 per rank.

Workload (the 2B dense config): 28 layers, hidden 2560, GQA 20 q / 4 kv heads of dim 128,
SwiGLU 6912, vocabulary 32768, bf16 weights ~N(0, 0.02) (random init, seeded), bf16 KV cache
prefilled to 4096 positions ~N(0, 1), greedy steps from a seeded token. A step is one whole
decode step (embedding row, 28 layers of RMSNorm / QKV / RoPE + KV append / attention /
o-proj / SwiGLU FFN, final norm, LM head, argmax). Steps run in greedy chains of 256
(positions 4096..4351, the workload's 256 steps), each chain one launch of the persistent
megakernel (dec_generate), repeated until K steps are timed.

``--workload moe_stack`` times the 42-layer MoE stack instead (GQA 20/4 over a 32768-position
cache, MoE of 512 MXFP4 experts top-8 + 1 shared, FP8 LM head 157184 x 2560, 512 greedy steps
per chain, positions 32768..33279); its 67 GB of experts are drawn and packed on the device.
``--token-stream repeat`` feeds the start token at every step instead (one launch per step),
a stream whose expert routing repeats; the expert prefetch mode comes from the library's
DEC_EXPERT_PREFETCH (0 off, the default; 1 adaptive; 2 always). ``--verify k`` times k-token verify
windows. ``--workload dense_layer | moe_layer | lm_head`` times the small configurations cold
(L2 flushed before every step) and hot.

Prints ONE JSON line (rank 0). Multi-GPU runs are replicas: every rank decodes its own
request on its own GPU with no communication on the data path; value = all ranks' tokens /
the slowest rank's time (weak scaling). ``--impl reference`` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "batch-1 decode tokens/s and achieved HBM GB/s (fraction of GB300 peak)"
CHAIN = 256          # greedy steps of the workload, positions 4096 .. 4351
NOMINAL_HBM_GBS = 8000.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def dist_setup(n_gpus, backend: str = "nccl"):
    """Rank, world size and local rank; one replica per GPU (torchrun env). The timing
    reductions below are the only collectives: the decode path itself has none."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return dist.get_rank(), ws, local
    return 0, 1, 0


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, secs: float, ws: int) -> float:
    """Units all ranks processed over the slowest rank's time (weak scaling: every replica
    runs the same per-GPU work)."""
    return ws * units_per_rank / max_over_ranks(secs, ws)


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join(ROOT, f".bench_clocks_{os.getpid()}.csv")

    def start(self):
        self.f = open(self.path, "w")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}", "--format=csv",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            self.f.close()
            os.remove(self.path)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        text = open(self.path).read()
        try:
            os.remove(self.path)
        except OSError:
            pass
        for ln in text.splitlines()[1:]:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1].split()[0]), float(f[2].split()[0]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def sources_sha256(source_files) -> str:
    sha = hashlib.sha256()
    for f in source_files:
        sha.update(open(f, "rb").read())
    return sha.hexdigest()


def ncu_traffic(key: str, source_files):
    """DRAM bytes (read + write) per decode step, or per verify window, of workload `key` from
    the committed ncu figures (profiles/dram_traffic.json), if the sources they were taken on are
    unchanged; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(key)
    if not rec:
        return None
    return float(rec["dram_bytes_per_step"]) if sources_sha256(source_files) == rec["source_sha256"] else None


def routing_overlap(dec, s, tok, pos, n, fixed=False):
    """Mean share of a MoE layer's routed experts that the step before had also chosen, over n
    one-token steps from (tok, pos), greedy or (fixed) all feeding tok, and every layer
    (untimed; read from the routing blocks)."""
    from persistent_megakernel_gb300 import binding as B
    prev, shares = None, []
    for i in range(n):
        nxt = B.dec_step(dec.ctx, tok, None, pos + i, None, True)
        tok = tok if fixed else nxt
        cur = [set(dec.routing(l)["expert"][s.n_shared:]) for l in range(s.n_layers)]
        if prev is not None:
            shares += [len(a & b) / max(1, len(a)) for a, b in zip(cur, prev)]
        prev = cur
    return float(np.mean(shares)) if shares else None


def kernel_sources():
    """Every source that shapes the kernel's launches: the device code and the host runtime
    that sets tile geometry, the op list and the workspace layout."""
    c = os.path.join(ROOT, "persistent_megakernel_gb300", "csrc")
    return [os.path.join(c, f) for f in ("megakernel.cu", "gemv.cuh", "ptx.cuh", "dec_internal.h", "api.cpp")]


def build_workload(seed: int, layers: int = 0):
    import synth
    from synth import model as sm
    s = synth.dense_2b_shape()
    if layers:
        s = s.with_(n_layers=layers)
    layers = [sm.layer_weights(s, seed, l) for l in range(s.n_layers)]
    head = sm.head_weights(s, seed)
    kv = [sm.kv_prefill(s, seed, l) for l in range(s.n_layers)]
    return s, layers, head, kv


WORKLOADS = {
    "dense_2b": "dense_2b: {L} layers, hidden 2560, GQA 20/4 x 128, SwiGLU 6912, vocab 32768, KV prefill 4096, "
                "batch 1, greedy, chains of 256 steps (pos 4096-4351)",
    "moe_stack": "moe_stack: {L} layers, hidden 2560, GQA 20/4 x 128, MoE 512 experts top-8 + 1 shared "
                 "(intermediate 768, MXFP4), FP8 LM head 157184 x 2560, KV prefill 32768, batch 1, greedy, "
                 "chains of 512 steps (pos 32768-33279)",
}


def workload_shape(name: str, layers: int = 0):
    import synth
    s = synth.dense_2b_shape() if name == "dense_2b" else synth.moe_stack_shape()
    return s.with_(n_layers=layers) if layers else s


def cpu_baseline_layer(s, seed):
    """The oracle on one decoder layer of one token of a large workload (attention over the
    cache + FFN of layer 0, its weights decoded as the oracle does in every step), repeated until
    about 10 s of CPU work; tokens/s scaled by the layer's share of the token's bytes."""
    import synth
    from synth import model as sm
    from oracle.model import OracleModel
    from persistent_megakernel_gb300 import roofline as R
    s1 = s.with_(n_layers=1)
    experts = (lambda l, e: sm.expert_weights(s, seed, 0, e)) if s.moe else None
    orc = OracleModel(s1, [sm.layer_weights(s, seed, 0)], sm.head_weights(s, seed), experts=experts,
                      kv=[sm.kv_prefill(s, seed, 0)], capacity=s.kv_prefill + 8)
    x = orc.embed(synth.start_token(seed, s.vocab))
    n, t0 = 0, time.perf_counter()
    while n < 6 and (n == 0 or time.perf_counter() - t0 < 10.0):
        y = orc.attention_block(0, x, s.kv_prefill)
        orc.ffn_block(0, y, {})
        n += 1
    dt = (time.perf_counter() - t0) / n
    share = (R.layer_weight_bytes(s) + R.kv_bytes(s, s.kv_prefill) / s.n_layers) / R.algorithmic_bytes(s, s.kv_prefill)
    cores = len(os.sched_getaffinity(0))
    return {"value": share / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} x one decoder layer (attention over {s.kv_prefill + 1} positions + FFN, weights and "
                      f"experts decoded per step) of one token, fp64 numpy: {dt:.2f} s per layer, scaled by the "
                      f"layer's share {share:.4f} of the token's bytes"}


def cpu_baseline(s, layers, head, kv, seed):
    """The oracle as it stands: full decode steps (28 layers + LM head, weights decoded to fp64
    in every step) at positions 4096, 4097, ... until about 10 s of CPU work (at most 6 steps)."""
    import synth
    from oracle.model import OracleModel
    orc = OracleModel(s, layers, head, kv=kv, capacity=s.kv_prefill + 8)
    tok = synth.start_token(seed, s.vocab)
    n, t0 = 0, time.perf_counter()
    while n < 6 and (n == 0 or time.perf_counter() - t0 < 10.0):
        tok = orc.step_token(tok, s.kv_prefill + n)["token"]
        n += 1
    dt = (time.perf_counter() - t0) / n
    cores = len(os.sched_getaffinity(0))
    return {"value": 1.0 / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} full greedy decode steps (28 layers + LM head, pos 4096..) of the fp64 numpy oracle: "
                      f"{dt:.2f} s per step"}


def cpu_baseline_one_core(workload: str, seed: int):
    """The oracle's layer sample (cpu_baseline_layer) on one host core: a child process pinned to
    one core with every BLAS / OpenMP pool at one thread (set before numpy loads)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", NUMEXPR_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-one-core", "--workload", workload,
                            "--seed", str(seed)], env=env, capture_output=True, text=True, timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, never fatal to the bench line
        return {"error": f"one-core sample failed: {type(e).__name__}"}


def run_reference(args):
    """Reference arm: the CPU oracle on the same workload; each step = one decoder layer of one
    token (dense 2B: attention + FFN of layer i mod 4 at position 4096 + i mod 256, the 28 layers
    having the same shape; MoE stack: layer 0 at position 32768 + i mod 512), throughput scaled
    by that layer's share of the token's algorithmic bytes. The sampled layers' weights are
    decoded to fp64 before the warm-up (MoE experts as the oracle selects them, then kept), so a
    run of K steps stays within minutes and a few GB of host memory."""
    if int(os.environ.get("RANK", "0")) != 0:
        return  # the oracle runs once, on rank 0; other ranks exit without work
    import synth
    from synth import model as sm
    from oracle.model import OracleModel
    from persistent_megakernel_gb300 import roofline as R
    if args.workload == "dense_2b":
        s, layers, head, kv = build_workload(args.seed)
        chain, ref_layers = CHAIN, 4
        orc = OracleModel(s, layers, head, kv=kv, capacity=s.kv_prefill + chain + 1, cache_weights=True)
    else:
        s = workload_shape(args.workload)
        chain, ref_layers = s.steps, 1
        orc = OracleModel(s.with_(n_layers=1), [sm.layer_weights(s, args.seed, 0)], sm.head_weights(s, args.seed),
                          experts=lambda l, e: sm.expert_weights(s, args.seed, 0, e),
                          kv=[sm.kv_prefill(s, args.seed, 0)], capacity=s.kv_prefill + chain + 1, cache_weights=True)
    x = orc.embed(synth.start_token(args.seed, s.vocab))
    per_token = R.algorithmic_bytes(s, s.kv_prefill)
    layer_bytes = R.layer_weight_bytes(s) + R.kv_bytes(s, s.kv_prefill) / s.n_layers

    def one(i):
        l, pos = i % ref_layers, s.kv_prefill + (i % chain)
        y = orc.attention_block(l, x, pos)
        orc.ffn_block(l, y, {})

    for i in range(ref_layers):  # decode the sampled layers' weights (setup, like loading)
        one(i)
    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(args.warmup + i)
    dt = time.perf_counter() - t0
    value = args.steps * (layer_bytes / per_token) / dt
    cores = len(os.sched_getaffinity(0))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload].format(L=s.n_layers), "step": "one decoder layer of one token"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"one decoder layer (attention + FFN, layers 0-{ref_layers - 1} in turn) per step, "
                                   "fp64 numpy, weights decoded once before timing"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def timed_generate(dec, ctx_handle, tok0, pos0, K, launches_per_step, chain=CHAIN):
    """K greedy steps in chains of `chain` on the device; returns (seconds by CUDA events, launches)."""
    import torch
    from persistent_megakernel_gb300 import binding as B
    out = torch.empty(chain, dtype=torch.int32, device=dec.device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(dec.stream)
    done, launches = 0, 0
    while done < K:
        n = min(chain, K - done)
        B.dec_generate(ctx_handle, tok0, pos0, n, out)
        launches += B.dec_last_launch_count(ctx_handle)
        done += n
    e1.record(dec.stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3, launches


def timed_fixed(dec, tok, pos0, K, chain=CHAIN):
    """K one-token steps that all feed token `tok` (teacher-forced, no readback), one launch
    each, at positions pos0 + (i % chain); returns (seconds by CUDA events, launches)."""
    import torch
    from persistent_megakernel_gb300 import binding as B
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(dec.stream)
    launches = 0
    for i in range(K):
        B.dec_step(dec.ctx, tok, None, pos0 + (i % chain), None, False)
        launches += B.dec_last_launch_count(dec.ctx)
    e1.record(dec.stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3, launches


SMALL = {
    "dense_layer": "dense_layer: one dense decoder layer + LM head, hidden 1024, GQA 8/2 x 128, SwiGLU 2816, "
                   "vocab 32000, 256 cached positions, hidden inputs ~N(0,1)",
    "moe_layer": "moe_layer: one MoE FFN block, hidden 2560, 512 MXFP4 experts top-8 + 1 shared (intermediate "
                 "768), bf16 router, hidden inputs ~N(0,1)",
    "lm_head": "lm_head: final LM head alone, 157184 x 2560 ({dt}), hidden inputs ~N(0,1)",
}


def run_small(args, rank, ws, local):
    """The small configurations (one dense layer + head, one MoE block, the LM head alone), which
    fit in L2 or nearly: each step runs on one of 16 seeded inputs in turn (different routings
    for the MoE block), timed cold, a 256 MB write flushing L2 before every step outside its
    CUDA events, and hot (steps back to back, weights left in L2 where they fit). e2e: the
    call a user makes on host buffers: the input copied in from pinned memory, the argmax (or,
    for the MoE block, dec_run_layer's bf16 output) copied out, every step."""
    import torch
    import synth
    from synth import model as sm
    from persistent_megakernel_gb300 import build as pbuild
    pbuild.build()
    from persistent_megakernel_gb300 import binding as B
    from persistent_megakernel_gb300 import roofline as R
    from persistent_megakernel_gb300.model import Decoder
    from oracle.model import OracleModel, bf16_to_f64_fast
    from tests.harness import weights
    k = args.verify
    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    if args.workload == "dense_layer":
        s = synth.dense_layer_shape()
    elif args.workload == "moe_layer":
        s = synth.moe_layer_shape(verify=k)
    else:
        s = synth.lm_head_shape(args.lm_head, verify=k)
    layers, head, kv, experts = weights(s, args.seed)
    cap = s.kv_prefill + 8
    dec = Decoder(s, layers, head, experts=experts, kv=kv, capacity=cap, device=dev, max_verify=k)
    pos = s.kv_prefill
    R_IN = 16
    xs_host = [sm.hidden_inputs(s, args.seed + 100 + i, k) for i in range(R_IN)]
    xs = [torch.from_numpy(x.view(np.int16)).to(dev) for x in xs_host]

    def one(i):
        if k == 1:
            B.dec_step(dec.ctx, 0, xs[i % R_IN], pos, None, False)
        else:
            B.dec_verify(dec.ctx, None, xs[i % R_IN], k, pos, None, want_argmax=False)

    routed = None
    if s.moe:  # distinct routed experts per step, averaged over the inputs
        n = []
        for i in range(R_IN):
            one(i)
            n.append(dec.routing(0)["n_slots"] - s.n_shared)
        routed = float(np.mean(n))
    bytes_step = R.algorithmic_bytes(s, pos, m=k, n_routed_active=None if routed is None else routed)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    K = args.steps
    for i in range(args.warmup):
        one(i)
    clocks = Clocks(local)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(dec.stream):
        for i in range(K):
            flush.fill_(i & 255)
            ev[i][0].record(dec.stream)
            one(i)
            ev[i][1].record(dec.stream)
    torch.cuda.synchronize()
    cold = sum(a.elapsed_time(b) for a, b in ev) * 1e-3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(dec.stream)
    for i in range(K):
        one(i)
    e1.record(dec.stream)
    torch.cuda.synchronize()
    hot = e0.elapsed_time(e1) * 1e-3
    barrier(ws)
    clk = clocks.stop()
    cold_max = max_over_ranks(cold, ws)
    # end to end through the C ABI on host buffers
    pin = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs_host]
    xin = torch.empty_like(xs[0])
    hout = torch.empty((k, s.hidden), dtype=torch.int16, device=dev)
    hout_host = torch.empty((k, s.hidden), dtype=torch.int16).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        with torch.cuda.stream(dec.stream):
            xin.copy_(pin[i % R_IN], non_blocking=True)
        if s.moe:
            B.dec_run_layer(dec.ctx, 0, xin, k, pos, hout)
            with torch.cuda.stream(dec.stream):
                hout_host.copy_(hout, non_blocking=True)
            dec.stream.synchronize()
        elif k == 1:
            B.dec_step(dec.ctx, 0, xin, pos, None, True)
        else:
            B.dec_verify(dec.ctx, None, xin, k, pos, None)
    e2e_secs = time.perf_counter() - t0
    d2h = 2 * k * s.hidden if s.moe else 4 * k + 32
    # the oracle on one token of the same configuration, as it stands, on the host cores
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        orc = OracleModel(s, layers, head, experts=experts, kv=kv, capacity=cap)
        xf = bf16_to_f64_fast(xs_host[0][0])
        orc.step(xf, pos)
        n_done, t0 = 0, time.perf_counter()
        while n_done < 3 or time.perf_counter() - t0 < 5.0:
            orc.step(bf16_to_f64_fast(xs_host[n_done % R_IN][0]), pos)
            n_done += 1
        per = (time.perf_counter() - t0) / n_done
        cpu = {"value": 1.0 / per, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{n_done} one-token steps of the fp64 numpy oracle on this configuration: {per:.3f} s each"}
    if rank == 0:
        peak, peak_kind = peaks()
        per_cold = cold_max / K
        achieved = bytes_step / per_cold / 1e9
        unit = "tokens/s" if k == 1 else "window tokens/s"
        print(json.dumps({
            "metric": METRIC, "value": whole_job_rate(K * k, cold, ws), "unit": unit, "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": 1e3 * per_cold, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": SMALL[args.workload].format(dt=args.lm_head), "verify": k, "mode": "persistent",
                       "routed_experts_per_step": routed,
                       "l2": "cold: a 256 MB write flushes L2 before every step, outside the step's CUDA events; "
                             "16 seeded inputs in turn",
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "traffic": None, "algorithmic_bytes_per_launch": bytes_step,
                         "launch_us": 1e6 * per_cold, "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                         "kernel": "dec_megakernel (one launch per step)"},
            "hot_l2": {"value": whole_job_rate(K * k, hot, ws), "unit": unit, "ms_per_step": 1e3 * hot / K,
                       "achieved_gbs": bytes_step / (hot / K) / 1e9,
                       "note": "steps back to back: weights that fit stay in L2 (not a bandwidth figure)"},
            "cpu_baseline": cpu,
            "e2e": {"value": whole_job_rate(K * k, e2e_secs, ws), "unit": unit,
                    "h2d_bytes_per_step": 2 * k * s.hidden + 60, "d2h_bytes_per_step": d2h, "steps": K,
                    "note": ("dec_run_layer" if s.moe else ("dec_step" if k == 1 else "dec_verify")) +
                            " per step: the input copied in from pinned host memory, the result copied out"},
            "gpu_launches": K,
            "clocks": clk,
        }))


def run_verify(args, rank, ws, local):
    """Verify windows of k tokens (the MTP verify step of the Ling-3.0-flash DGX Spark article,
    "optimisation 3"): each call feeds k tokens at the next k positions (positions advance by k,
    as if every draft were accepted). value: windows launched back to back with no readback,
    CUDA events on the library's stream; e2e: the same windows through dec_verify with the
    model's last prediction fed back as each window's first token and the k argmaxes and the
    accepted count read back every window. roofline = the window's algorithmic bytes (weights
    once, the union of the window's experts, the KV rows read) over its device time."""
    import torch
    import synth
    from persistent_megakernel_gb300 import build as pbuild
    pbuild.build()
    from persistent_megakernel_gb300 import binding as B
    from persistent_megakernel_gb300 import roofline as R
    from persistent_megakernel_gb300.model import Decoder
    k = args.verify
    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    n_win = args.warmup + args.steps
    if args.workload == "dense_2b":
        s, layers, head, kv = build_workload(args.seed, args.layers)
        cap = s.kv_prefill + k * n_win + 8
        dec = Decoder(s, layers, head, kv=kv, capacity=cap, mode=args.mode, device=dev, max_verify=k)
    else:
        from tests.device_inputs import device_decoder
        s = workload_shape(args.workload, args.layers)
        cap = s.kv_prefill + k * n_win + 8
        dec = device_decoder(s, args.seed, cap, dev, mode=args.mode, max_verify=k)
    drafts = synth.bits(args.seed, synth.tensor_id("token", 0, 1), n_win * k) % np.uint64(s.vocab)
    tok0 = synth.start_token(args.seed, s.vocab)

    def toks_of(i, first):
        return [int(first)] + [int(x) for x in drafts[i * k + 1:(i + 1) * k]]

    # device-timed: back-to-back windows, no host readback between them
    for i in range(args.warmup):
        B.dec_verify(dec.ctx, toks_of(i, tok0), None, k, s.kv_prefill + i * k, None, want_argmax=False)
    barrier(ws)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(dec.stream)
    for i in range(args.warmup, n_win):
        B.dec_verify(dec.ctx, toks_of(i, tok0), None, k, s.kv_prefill + i * k, None, want_argmax=False)
    e1.record(dec.stream)
    torch.cuda.synchronize()
    secs = e0.elapsed_time(e1) * 1e-3
    barrier(ws)
    B.dec_sync(dec.ctx)
    # end to end: the model's prediction fed back, argmaxes and status read back every window
    tok = tok0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.warmup, n_win):
        am, _ = B.dec_verify(dec.ctx, toks_of(i, tok), None, k, s.kv_prefill + i * k, None)
        tok = am[-1]
    e2e_secs = time.perf_counter() - t0
    routed = None
    if s.moe:  # distinct routed experts of the last window, averaged over the layers
        routed = float(np.mean([dec.routing(l)["n_slots"] - s.n_shared for l in range(s.n_layers)]))
    pos_mid = s.kv_prefill + k * (args.warmup + args.steps // 2)
    bytes_win = R.algorithmic_bytes(s, pos_mid, m=k, n_routed_active=None if routed is None else round(routed))
    per_win = max_over_ranks(secs, ws) / args.steps
    peak, peak_kind = peaks()
    achieved = bytes_win / per_win / 1e9
    traffic = ncu_traffic(f"{args.workload}_verify{k}", kernel_sources()) if not args.layers else None  # per window
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        # the oracle's window is k causal steps: its window tokens/s are its tokens/s
        cpu = cpu_baseline_layer(s, args.seed)
        cpu["one_core"] = cpu_baseline_one_core(args.workload, args.seed)
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": whole_job_rate(args.steps * k, secs, ws), "unit": "window tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * per_win,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOADS[args.workload].format(L=s.n_layers), "verify": k,
                       "step": f"one verify window of {k} tokens (one launch)", "mode": args.mode,
                       "routed_experts_per_layer": routed,
                       "l2": "no flush: each window streams %.2f GB > 129 MB L2" % (bytes_win / 1e9)},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "traffic": traffic, "algorithmic_bytes_per_launch": bytes_win,
                         "launch_us": 1e6 * per_win,
                         "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                         "kernel": "dec_megakernel (one launch per window)"},
            "cpu_baseline": cpu,
            "e2e": {"value": whole_job_rate(args.steps * k, e2e_secs, ws), "unit": "window tokens/s",
                    "h2d_bytes_per_step": 60 + 4 * k, "d2h_bytes_per_step": 4 * k + 32, "steps": args.steps,
                    "note": "dec_verify per window: tokens and position copied in, argmaxes and status copied out"},
            "gpu_launches": args.steps,
        }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="persistent", choices=["persistent", "per_op", "graph"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-compare", action="store_true", help="skip the launch-per-op comparison")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="dense_2b", choices=sorted(WORKLOADS) + sorted(SMALL))
    ap.add_argument("--lm-head", default="bf16", choices=["bf16", "fp8"], help="--workload lm_head: its format")
    ap.add_argument("--verify", type=int, default=1, choices=[1, 2, 3, 4],
                    help="> 1: time verify windows of this many tokens")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"], help="KV cache format (fp8: e4m3, scales 1.0)")
    ap.add_argument("--token-stream", default="greedy", choices=["greedy", "repeat"],
                    help="repeat: every step feeds the start token (teacher-forced, one launch per step), "
                         "a stream whose MoE routing repeats from step to step")
    ap.add_argument("--cpu-one-core", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling captures only: fewer decoder layers (the line is then not the workload's)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.cpu_one_core:  # child of cpu_baseline_one_core: the oracle's layer sample on one core
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
        print(json.dumps(cpu_baseline_layer(workload_shape(args.workload), args.seed)))
        return
    if args.impl == "reference":
        if args.workload in SMALL:
            ap.error("--impl reference times dense_2b or moe_stack (a small workload's line carries its oracle's time)")
        return run_reference(args)

    rank, ws, local = dist_setup(args.gpus)
    if args.workload in SMALL:
        return run_small(args, rank, ws, local)
    if args.verify > 1:
        return run_verify(args, rank, ws, local)
    import torch
    import synth
    from persistent_megakernel_gb300 import build as pbuild
    pbuild.build()
    from persistent_megakernel_gb300 import binding as B
    from persistent_megakernel_gb300 import roofline as R
    from persistent_megakernel_gb300.model import Decoder

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    chain = CHAIN
    layers = head = kv = None
    if args.workload == "dense_2b":
        s, layers, head, kv = build_workload(args.seed, args.layers)
        s = s.with_(kv_dtype=args.kv)
        cap = s.kv_prefill + chain + 8
        dec = Decoder(s, layers, head, kv=kv, capacity=cap, mode=args.mode, device=dev)
    else:
        from tests.device_inputs import device_decoder
        s = workload_shape(args.workload, args.layers).with_(kv_dtype=args.kv)
        chain = s.steps
        dec = device_decoder(s, args.seed, s.kv_prefill + chain + 8, dev, mode=args.mode)
    tok0 = synth.start_token(args.seed, s.vocab)
    pos0 = s.kv_prefill

    # warm-up, then exactly K timed steps bracketed by barrier + synchronize
    fixed = args.token_stream == "repeat"

    def run_steps(K):
        return timed_fixed(dec, tok0, pos0, K, chain) if fixed else timed_generate(dec, dec.ctx, tok0, pos0, K, 1, chain)

    run_steps(args.warmup)
    clocks = Clocks(local)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    secs, launches = run_steps(args.steps)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    secs_max = max_over_ranks(secs, ws)
    value = whole_job_rate(args.steps, secs, ws)
    # five more timed runs after the one the line reports (the median shows the run-to-run spread)
    Kr = min(args.steps, chain)
    rep = [run_steps(Kr)[0] / Kr * 1e3 for _ in range(5)]
    repeat = {"runs": 5, "steps_each": Kr, "median_ms_per_step": statistics.median(rep),
              "ms_per_step": [round(x, 4) for x in rep]}

    # algorithmic bytes per step averaged over the positions the timed steps used; one launch runs
    # a chain of steps, so per launch: bytes per step x steps per launch over the launch's time
    poss = [pos0 + (i % chain) for i in range(args.steps)]
    bytes_step = float(np.mean([R.algorithmic_bytes(s, p) for p in poss]))
    steps_per_launch = args.steps / launches
    launch_s = secs / launches
    peak, peak_kind = peaks()
    achieved = bytes_step * steps_per_launch / launch_s / 1e9
    traffic_key = args.workload + ("_kv8" if args.kv == "fp8" else "")
    traffic_step = ncu_traffic(traffic_key, kernel_sources()) if args.mode == "persistent" and not args.layers else None
    traffic = traffic_step * steps_per_launch if traffic_step is not None else None
    overlap = None
    if s.moe and rank == 0:
        overlap = routing_overlap(dec, s, tok0, pos0, 9, fixed)

    # end to end through the C ABI with host buffers: token in, argmax out, every step
    K2 = min(args.steps, chain)
    tok = tok0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K2):
        nxt = B.dec_step(dec.ctx, tok, None, pos0 + i, None, True)
        tok = tok if fixed else nxt
    e2e_secs = time.perf_counter() - t0
    e2e = {"value": whole_job_rate(K2, e2e_secs, ws), "unit": "tokens/s", "h2d_bytes_per_step": 60, "d2h_bytes_per_step": 36,
           "steps": K2, "note": "dec_step per token: token and position copied in, argmax and status copied out"}

    compare = None
    if not args.no_compare and args.mode == "persistent":
        compare = {}
        Kc = min(args.steps, chain)
        for mode in ("per_op", "graph"):
            ctx, wsb = dec.context(mode)
            timed_generate(dec, ctx, tok0, pos0, 4, 1, chain)
            t, L = timed_generate(dec, ctx, tok0, pos0, Kc, 1, chain)
            compare[mode] = {"tokens_s": Kc / t, "launches_per_step": L / Kc, "steps": Kc}
            B.dec_free(ctx)
            del wsb
        compare["persistent"] = {"tokens_s": args.steps / secs, "launches_per_step": launches / args.steps}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(s, layers, head, kv, args.seed) if layers is not None else cpu_baseline_layer(s, args.seed)
        cpu["one_core"] = cpu_baseline_one_core(args.workload, args.seed)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * secs_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOADS[args.workload].format(L=s.n_layers) +
                                   (", FP8 e4m3 KV cache (scales 1.0)" if args.kv == "fp8" else ""),
                       "weights": ("bf16 ~N(0,0.02) seeded, accumulate fp32" if args.workload == "dense_2b" else
                                   "bf16 attention / router / embedding, MXFP4 experts and FP8 head quantised from "
                                   "seeded bf16 ~N(0,0.02), drawn and packed on the device; accumulate fp32"),
                       "mode": args.mode,
                       "l2": "no flush: each step streams %.2f GB > 129 MB L2" % (bytes_step / 1e9),
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                         "traffic_per_step": traffic_step,
                         "algorithmic_bytes_per_launch": bytes_step * steps_per_launch,
                         "algorithmic_bytes_per_step": bytes_step, "steps_per_launch": steps_per_launch,
                         "launch_us": launch_s * 1e6, "step_us": 1e6 * secs / args.steps,
                         "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                         "kernel": "dec_megakernel (one launch per chain of greedy steps)"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
            "compare_launch_modes": compare,
            "repeat": repeat,
        }
        if fixed:
            line["config"]["token_stream"] = ("repeat: every step feeds the start token at the next position "
                                              "(teacher-forced, one launch per step)")
        if s.moe:
            line["config"]["expert_prefetch"] = {
                "mode": int(os.environ.get("DEC_EXPERT_PREFETCH", "0")),
                "routed_overlap_with_previous_step": overlap}
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
