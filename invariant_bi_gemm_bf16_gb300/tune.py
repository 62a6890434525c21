"""Command line of the offline pin tuner (see tuner.py).

    python -m invariant_bi_gemm_bf16_gb300.tune --workload llama31-70b-decode --out table.json

Workloads (synthetic inputs, random-init weights of the named shapes):
  llama31-70b-decode  the 4-layer Llama-3.1-70B-shaped decode step (stack.py)
                      at batch sizes 1, 8, 32, 64, 128, 256 with weights
                      1, 2, 4, 2, 1, 1 (recorded by running the stack);
  llama31-8b-prefill  the Llama-3.1-8B qkv, gate_up and down_proj projections at
                      M = 1, 8, 32, 128, 1024, 4096, 8192, one call each.
  llama31-8b-decode   the same projections at decode batch sizes 1, 8, 16, 32,
                      64 with weights 1, 2, 2, 4, 1.
  decode-attention-70b  decode attention with Llama-3.1-70B heads (64 query, 8
                      key/value, pages of 16) over three decode steps, one each:
                      64 requests with lengths uniform on [512, 8192], 256 on
                      [64, 2048], and one request of 32768; the split size is
                      the tuned pin.
The tuned table is one pin tuple per (N, K), for every batch size.  For the
decode workload, the additivity error delta is measured on the whole step
(default tuple against tuned tuple) and reported with its bound.
"""
from __future__ import annotations

import argparse
import json
import sys

import torch

from . import binding as bd
from . import tuner

DECODE_MIX = {1: 1, 8: 2, 32: 4, 64: 2, 128: 1, 256: 1}
PREFILL_MS = (1, 8, 32, 128, 1024, 4096, 8192)
DECODE8B_MIX = {1: 1, 8: 2, 16: 2, 32: 4, 64: 1}


def stack_time_us(stack, xs, reps=5):
    """Device time of the decode mix (each batch size its weight's number of
    steps), captured in a CUDA graph and replayed, like the families' timing."""
    for x in xs.values():
        stack.forward(x)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for M, x in xs.items():
            for _ in range(DECODE_MIX[M]):
                stack.forward(x)
    g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1e3 / reps


def run_decode(args):
    from . import inputs
    from .stack import LLAMA31_70B, DecodeStack, random_layers
    shape = LLAMA31_70B
    layers = random_layers(shape, seed=0)
    stack = DecodeStack(shape, layers)
    xs = {M: inputs.device_normal((M, shape.hidden), seed=0, stream=0) for M in DECODE_MIX}
    rec = tuner.Recorder()
    with rec:
        for M, x in xs.items():
            for _ in range(DECODE_MIX[M]):
                stack.forward(x)
    torch.cuda.synchronize()
    flags = bd.BI_FLAG_SCHEDULE_AUTO | bd.BI_FLAG_PREFETCH_W   # weights are never written while serving
    entries = []
    for (N, K), calls in sorted(rec.families().items()):
        e = tuner.tune_family(N, K, calls, mode=args.mode, reps=args.reps, base_flags=flags)
        print(json.dumps({k: e[k] for k in ("N", "K", "T_us", "T_default_us", "measured", "legal")}),
              file=sys.stderr, flush=True)
        entries.append(e)
    # additivity check on the whole step, C = T(default) - sum_f T_f(default);
    # the two tuples are timed alternately and the medians taken
    import statistics
    table = {(e["N"], e["K"]): bd.Pins(**e["pins"]) for e in entries}
    tuned = DecodeStack(shape, layers, pin_table=table)
    td, tt = [], []
    for _ in range(3):
        td.append(stack_time_us(stack, xs))
        tt.append(stack_time_us(tuned, xs))
    t_default, t_tuned = statistics.median(td), statistics.median(tt)
    c_other = t_default - sum(e["T_default_us"] for e in entries)
    delta = tuner.measured_delta(t_tuned, c_other, [e["T_us"] for e in entries])
    meta = {"workload": "llama31-70b-decode: 4-layer Llama-3.1-70B-shaped decode step, batch mix %s"
                        % json.dumps(DECODE_MIX),
            "device": torch.cuda.get_device_name(), "sm_count": torch.cuda.get_device_properties(0).multi_processor_count,
            "mode": args.mode, "T_workload_default_us": round(t_default, 1), "T_workload_tuned_us": round(t_tuned, 1),
            "C_other_us": round(c_other, 1), "delta": round(delta, 4), "delta_bound": round(tuner.delta_bound(delta), 4)}
    return entries, meta


def run_projections(args, calls_of_m, name):
    flags = bd.BI_FLAG_SCHEDULE_AUTO | bd.BI_FLAG_PREFETCH_W
    entries = []
    for N, K in ((6144, 4096), (28672, 4096), (4096, 14336)):
        calls = list(calls_of_m)
        e = tuner.tune_family(N, K, calls, mode=args.mode, reps=args.reps, base_flags=flags)
        print(json.dumps({k: e[k] for k in ("N", "K", "T_us", "T_default_us", "measured", "legal")}),
              file=sys.stderr, flush=True)
        entries.append(e)
    meta = {"workload": name, "device": torch.cuda.get_device_name(),
            "sm_count": torch.cuda.get_device_properties(0).multi_processor_count, "mode": args.mode}
    return entries, meta


def run_prefill(args):
    return run_projections(args, [(M, 1) for M in PREFILL_MS],
                           "llama31-8b-prefill: qkv, gate_up, down_proj at M = %s, one call each" % (PREFILL_MS,))


def run_decode8b(args):
    return run_projections(args, sorted(DECODE8B_MIX.items()),
                           "llama31-8b-decode: qkv, gate_up, down_proj at the decode batch mix %s"
                           % json.dumps(DECODE8B_MIX))


ATTN_STEPS = ((64, 512, 8192), (256, 64, 2048), (1, 32768, 32768))


def run_attention(args):
    import numpy as np
    rng = np.random.default_rng(70)
    calls = [([int(x) for x in rng.integers(lo, hi + 1, size=B)], 1) for B, lo, hi in ATTN_STEPS]
    e = tuner.tune_attention(64, 8, 16, calls)
    print(json.dumps(e["attention"]["measured"]), file=sys.stderr, flush=True)
    meta = {"workload": "decode-attention-70b: 64 query / 8 key-value heads, pages of 16; steps (B, lo, hi) = %s"
                        % (ATTN_STEPS,),
            "device": torch.cuda.get_device_name(), "sm_count": torch.cuda.get_device_properties(0).multi_processor_count}
    return [e], meta


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=["llama31-70b-decode", "llama31-8b-prefill", "llama31-8b-decode",
                                           "decode-attention-70b"], required=True)
    ap.add_argument("--mode", choices=["search", "exhaustive"], default="search")
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--out", required=True)
    args = ap.parse_args(argv)
    bd.load()
    if args.workload == "llama31-70b-decode":
        entries, meta = run_decode(args)
    elif args.workload == "llama31-8b-prefill":
        entries, meta = run_prefill(args)
    elif args.workload == "llama31-8b-decode":
        entries, meta = run_decode8b(args)
    else:
        entries, meta = run_attention(args)
    tuner.dump(entries, args.out, **meta)
    tuner.load(args.out)   # the written table must validate
    print(json.dumps({k: v for k, v in meta.items()}), flush=True)


if __name__ == "__main__":
    main()
