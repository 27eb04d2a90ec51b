"""Self-timing of the megakernel: read the per-(CTA, op) %globaltimer records of a build made
with DEC_TRACE (``build.build(variant="trace")``, loaded with DEC_LIB_VARIANT=trace), summarise
where a step's time goes, and export a Chrome trace.

Each CTA stamps, per op: consumer start, input ready (dependency wait over), prologue done
(activations in shared memory), all warps' tiles done, op end (signalled); its producer
stamps its first and last tile issue of the op and counts the tiles. The kernel times itself
because an external profiler sees one long bar per launch (Muse Spark Open megakernel
article, section "where else the 5.9 ms goes": lane 0 of every block writes globaltimer
stamps to a global array; a build flag compiles it out; outputs stay bit-identical).

    DEC_LIB_VARIANT=trace python -m persistent_megakernel_gb300.trace [--layers N] [--steps S]
        [--workload moe_stack]
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

OP_NAMES = ["qkv", "attn", "oproj", "gateup", "down", "router", "shared_gateup", "routed_gateup", "exp_down",
            "lm_head"]
FIELDS = ["start", "ready", "prologue", "tiles", "end", "p_first", "p_last", "p_count", "loaded", "late",
          "merge", "merge_ready"]
NF = len(FIELDS)


def op_types(shape) -> list[str]:
    """Op order of a step, as the runtime builds it."""
    out = []
    for _ in range(shape.n_layers):
        if shape.n_q:
            out += ["qkv", "attn", "oproj"]
        if shape.ffn:
            out += ["gateup", "down"]
        if shape.n_experts:
            out += ["router", "routed_gateup", "exp_down"]
    if shape.vocab:
        out.append("lm_head")
    return out


TILE_LOG = 1024   # tiles logged per consumer warp of CTA 0
TILE_STAMPS = 6   # clock64: issued, wait start, landed, computed, released, pad
CONSUMER_WARPS = 7


def region(dec, with_tiles=False):
    """uint8 view of the trace records inside the decoder's workspace (None without DEC_TRACE)."""
    from . import binding as B
    ptr, n_ctas, n_ops = B.dec_trace_buffer(dec.ctx)
    if not ptr:
        return None, n_ctas, n_ops
    off = ptr - dec.ws.data_ptr()
    n = n_ctas * n_ops * NF * 8 + (CONSUMER_WARPS * TILE_LOG * TILE_STAMPS * 8 if with_tiles else 0)
    return dec.ws[off:off + n], n_ctas, n_ops


def clear(dec):
    r, _, _ = region(dec, with_tiles=True)
    if r is not None:
        r.zero_()


def read(dec) -> np.ndarray:
    import torch
    r, n_ctas, n_ops = region(dec)
    if r is None:
        raise RuntimeError("the loaded library was built without DEC_TRACE")
    torch.cuda.synchronize()
    return r.cpu().numpy().view(np.uint64).reshape(n_ctas, n_ops, NF).astype(np.int64)


def read_tiles(dec) -> np.ndarray:
    """[consumer warps, TILE_LOG, 6] clock64 stamps of CTA 0's tiles: issued (producer), consumer
    starts waiting, data landed, compute done, released."""
    import torch
    r, n_ctas, n_ops = region(dec, with_tiles=True)
    torch.cuda.synchronize()
    a = r.cpu().numpy().view(np.uint64).astype(np.int64)
    return a[n_ctas * n_ops * NF:].reshape(CONSUMER_WARPS, TILE_LOG, TILE_STAMPS)


def tile_summary(t: np.ndarray, ghz: float = 2.07) -> dict:
    """Median cycles -> microseconds per tile phase over CTA 0's warps."""
    x = t.reshape(-1, TILE_STAMPS)
    x = x[(x[:, 0] > 0) & (x[:, 4] > 0)]
    us = lambda d: float(np.median(d) / ghz / 1e3)
    return {"tiles": int(len(x)),
            "issue_to_landed_us": us(x[:, 2] - x[:, 0]),
            "issue_before_wait_us": us(x[:, 1] - x[:, 0]),
            "wait_us": us(x[:, 2] - x[:, 1]),
            "compute_us": us(x[:, 3] - x[:, 2]),
            "release_us": us(x[:, 4] - x[:, 3])}


def summarize(rec: np.ndarray, names: list[str]) -> dict:
    """Mean microseconds per phase and op kind over CTAs and layers, plus the step span."""
    t0 = rec[:, :, 0][rec[:, :, 0] > 0].min()
    res = {"step_us": float((rec[:, :, 4].max() - t0) / 1e3), "ops": {}}
    for kind in dict.fromkeys(names):
        idx = [i for i, n in enumerate(names) if n == kind]
        r = rec[:, idx, :]
        live = r[:, :, 0] > 0
        d = lambda a, b: float(np.mean((r[:, :, b] - r[:, :, a])[live]) / 1e3)
        has_p = r[:, :, 7] > 0
        lead = float(np.mean((r[:, :, 0] - r[:, :, 5])[live & has_p]) / 1e3) if np.any(live & has_p) else 0.0
        # latest completion across CTAs of each op instance, relative to the earliest start
        span = [float((r[:, k, 4].max() - r[:, k, 0][r[:, k, 0] > 0].min()) / 1e3) for k in range(len(idx))]
        has_l = r[:, :, 8] > 0
        load = float(np.mean((r[:, :, 8] - r[:, :, 1])[live & has_l]) / 1e3) if np.any(live & has_l) else 0.0
        has_m = r[:, :, 11] > 0
        merge = float(np.mean((r[:, :, 11] - r[:, :, 10])[live & has_m]) / 1e3) if np.any(live & has_m) else 0.0
        res["ops"][kind] = {
            "count": len(idx), "wait": d(0, 1), "prologue": d(1, 2), "tiles": d(2, 3), "end": d(3, 4),
            "load": load, "late_words": float(np.mean(r[:, :, 9])), "merge_wait": merge,
            "producer_lead": lead, "tiles_issued": float(np.mean(r[:, :, 7])), "span_all_ctas": float(np.mean(span))}
    return res


def chrome(rec: np.ndarray, names: list[str], path: str) -> None:
    t0 = rec[:, :, 0][rec[:, :, 0] > 0].min()
    ev = []
    for c in range(rec.shape[0]):
        for i, n in enumerate(names):
            r = rec[c, i]
            if r[0] == 0:
                continue
            for a, b, what in ((0, 1, "wait"), (1, 2, "prologue"), (2, 3, "tiles"), (3, 4, "end")):
                ev.append({"name": f"{n}:{what}", "ph": "X", "pid": 0, "tid": c, "ts": (r[a] - t0) / 1e3,
                           "dur": max(0, r[b] - r[a]) / 1e3})
            if r[7]:
                ev.append({"name": f"{n}:issue", "ph": "X", "pid": 1, "tid": c, "ts": (r[5] - t0) / 1e3,
                           "dur": max(0, r[6] - r[5]) / 1e3})
    json.dump({"traceEvents": ev}, open(path, "w"))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=28)
    ap.add_argument("--steps", type=int, default=4)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--chrome", default="")
    ap.add_argument("--dump", default="", help="save the raw records (.npz)")
    ap.add_argument("--workload", default="dense_2b", choices=["dense_2b", "moe_stack"],
                    help="moe_stack: weights drawn and packed on the device")
    args = ap.parse_args(argv)
    variant = os.environ.get("DEC_LIB_VARIANT", "")
    if "trace" not in variant:
        sys.exit("set DEC_LIB_VARIANT to a build with DEC_TRACE (trace)")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch
    import synth
    from synth import model as sm
    from . import build
    from .model import Decoder
    if variant == "trace":
        build.build(variant="trace")
    if args.workload == "dense_2b":
        s = synth.dense_2b_shape().with_(n_layers=args.layers)
        layers = [sm.layer_weights(s, args.seed, l) for l in range(s.n_layers)]
        head = sm.head_weights(s, args.seed)
        kv = [sm.kv_prefill(s, args.seed, l) for l in range(s.n_layers)]
        dec = Decoder(s, layers, head, kv=kv, capacity=s.kv_prefill + 64)
    else:
        from tests.device_inputs import device_decoder
        s = synth.moe_stack_shape().with_(n_layers=args.layers)
        dec = device_decoder(s, args.seed, s.kv_prefill + 64)
    tok = synth.start_token(args.seed, s.vocab)
    for i in range(args.steps):
        clear(dec)
        tok = dec.step(tok, s.kv_prefill + i)
    rec = read(dec)
    names = op_types(s)
    summ = summarize(rec, names)
    tiles = read_tiles(dec)
    summ["tile_log"] = tile_summary(tiles)
    if args.dump:
        np.savez(args.dump, rec=rec, tiles=tiles, names=np.array(names))
    print(json.dumps(summ, indent=1))
    if args.chrome:
        chrome(rec, names, args.chrome)


if __name__ == "__main__":
    main()
