"""Benchmark of the batch-invariant linear layer on GB300.

Default workload (one GPU): the Llama-3.1-8B down_proj GEMM, W [4096, 14336],
swept over M = 1, 2, 4, ..., 8192 tokens.  One step = one bi_gemm_bf16_ws call at
every M of the sweep.  `value` = the sweep's FLOPs / its device time (TFLOPS).
Per-M times, TFLOPS, GB/s, roofline fractions and the torch.mm (cuBLAS) time on
the same tensors are in "sweep".

The same JSON line also carries, unless switched off: "stack" (the 4-layer
Llama-3.1-70B-shaped decode step at 32 tokens, us/step), "fused" (RMSNorm +
the Llama-3.1-8B qkv and gate_up projections in one call, per M), "rmsnorm"
(the RMSNorm token sweep at H = 4096 and 8192, GB/s) and "lm_head" (the
Llama-3.1-8B lm_head with per-token log-probabilities) and "fp8" (the
down_proj shape in E4M3 with per-token scales), each against torch on the
same tensors.

L2 handling: every launch reads a weight copy that was not read by the
previous launches (enough copies that they exceed the 129 MB L2), and
activations rotate likewise; no flush writes are issued.

--impl reference times the CPU oracle (the reference arm of this build) on a
bounded sample of the same workload.  Under torchrun each rank runs the same
per-GPU workload on its own replica (weak scaling: rows are independent and
the reduction tree never depends on M, so no collective is needed).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
DOWN_N, DOWN_K = 4096, 14336
SWEEP_M = [1 << i for i in range(14)]  # 1 .. 8192
EPS = 1e-5


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of single
# launches, from ncu captures of `python bench.py --single-m M --launches 2`
# (summaries in profiles/), keyed by build_fingerprint() of the GEMM kernel's
# sources: valid only for the kernel build they were taken on.
NCU_TRAFFIC = {
    "b490e113673c64e71c7e774aaa74af97c0ded5e15ed16ffca2afebf67b418fdf": {8192: 962324224 + 65573888,
                                                                        1: 117515520 + 2776320},
}


def build_fingerprint(kernel_files=("gemm_kernel.cuh", "gemm.cu", "ptx.cuh", "internal.h", "rowmath.cuh", "bounds.cuh")):
    """SHA-256 of the sources one kernel is compiled from (default: the GEMM
    kernel's) and the compiler flags: DRAM counters taken by ncu stay valid
    while this is unchanged.  The public header is left out: the kernel uses
    only its ABI constants (tile sizes, flag bits, status codes), which do not
    change."""
    import hashlib
    from invariant_bi_gemm_bf16_gb300 import build as B
    h = hashlib.sha256()
    try:
        for name in kernel_files:
            with open(os.path.join(B.CSRC, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    except OSError:
        return None
    h.update(" ".join(B.NVCC_FLAGS).encode())
    return h.hexdigest()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def gemm_work(M, N, K):
    """Algorithmic FLOPs and bytes of one GEMM (W counted once)."""
    return 2.0 * M * N * K, 2.0 * (N * K + M * K + M * N)


def roof_time_us(flops, bytes_, peaks):
    return max(flops / (peaks["bf16_tflops"] * 1e6), bytes_ / (peaks["hbm_gbs"] * 1e3))


# ---------------------------------------------------------------------------
# distributed helpers (torchrun: one rank per GPU)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            if torch.cuda.is_available():
                self.pg.barrier(device_ids=[self.local_rank])
            else:
                self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, v: float) -> float:
        if not self.pg:
            return v
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def shard_rows(total: int, world: int, rank: int):
    """Contiguous row range [lo, hi) of `rank` when `total` independent rows are
    split over `world` ranks (a replica of W on every rank, no exchange)."""
    return (total * rank // world, total * (rank + 1) // world)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock / throttle samples every 20 ms; only the samples that
    arrive while the timed region runs (mark_start .. mark_end) are kept."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0 = self.t0 if self.t0 is not None else -1e30
        t1 = self.t1 if self.t1 is not None else 1e30
        for ts, line in self.lines:
            if ts < t0 or ts > t1 + 0.025:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "window_s": round((t1 - t0), 3) if self.t0 is not None and self.t1 is not None else None}


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------

_ORACLE_INPUTS = {}


def oracle_inputs(max_rows: int):
    """Host bf16 bit patterns of the down_proj workload (seed 0), cached."""
    from invariant_bi_gemm_bf16_gb300 import inputs
    if max_rows not in _ORACLE_INPUTS:
        W = inputs.bits(inputs.normal((DOWN_N, DOWN_K), std=0.02, seed=0, stream=inputs.STREAM_W))
        X = inputs.bits(inputs.normal((max_rows, DOWN_K), seed=0, stream=inputs.STREAM_X))
        _ORACLE_INPUTS[max_rows] = (X, W)
    return _ORACLE_INPUTS[max_rows]


def oracle_gemm_throughput(target_s: float = 12.0, max_rows: int = 2048):
    """Times the oracle's down_proj GEMM on a sample of rows (all 4096 output
    features each), grown until it takes about target_s seconds.  Returns
    (TFLOPS, seconds, rows, threads)."""
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    X, W = oracle_inputs(max_rows)
    rows = 2
    while True:
        t0 = time.perf_counter()
        oracle.gemm(X[:rows], W, nthreads=threads)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or rows >= max_rows:
            break
        rows = min(max_rows, max(rows * 2, int(rows * target_s / max(dt, 1e-3))))
    flops = 2.0 * rows * DOWN_N * DOWN_K
    return flops / dt / 1e12, dt, rows, threads


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_gemm_1thread(rows: int = 16):
    """The oracle's down_proj GEMM on `rows` rows with one thread: (TFLOPS, seconds)."""
    import oracle
    X, W = oracle_inputs(max(rows, 2))
    t0 = time.perf_counter()
    oracle.gemm(X[:rows], W, nthreads=1)
    dt = time.perf_counter() - t0
    return 2.0 * rows * DOWN_N * DOWN_K / dt / 1e12, dt


def smi_gpu_id(local_rank: int) -> str:
    """The nvidia-smi -i argument for this process's GPU."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

class DownProjSweep:
    """configs: Llama-3.1-8B down_proj, X [M,14336] ~N(0,1), W [4096,14336] ~N(0,0.02)."""
    name = "down_proj_m_sweep"

    def __init__(self, bd, dev, seed, sweep=SWEEP_M):
        from invariant_bi_gemm_bf16_gb300 import inputs
        self.bd = bd
        self.dev = dev
        self.N, self.K = DOWN_N, DOWN_K
        self.ms = list(sweep)
        wbytes = self.N * self.K * 2
        self.nw = max(2, math.ceil(2 * L2_BYTES / wbytes) + 1)
        self.W = [inputs.device_normal((self.N, self.K), std=0.02, seed=seed, stream=inputs.STREAM_W + 16 * i,
                                       device=dev) for i in range(self.nw)]
        self.X = {}
        for M in self.ms:
            nx = min(self.nw, max(1, math.ceil(2 * L2_BYTES / (M * self.K * 2))))
            self.X[M] = [inputs.device_normal((M, self.K), seed=seed, stream=inputs.STREAM_X + 16 * i, device=dev)
                         for i in range(nx)]
        self.Y = {M: torch.empty((M, self.N), dtype=torch.bfloat16, device=dev) for M in self.ms}
        # the weight copies are never written while the sweep runs
        self.pins = bd.bi_pins_default(self.N, self.K)
        self.pins = self.pins.replace(flags=self.pins.flags | bd.BI_FLAG_PREFETCH_W)
        # one fold workspace for every M (bi_gemm_bf16_ws): its counters are
        # zeroed once and every call leaves them zero
        fold = max(bd.bi_gemm_bf16_workspace_bytes(M, self.N, self.K, self.pins) for M in self.ms)
        self.ws = torch.zeros(max(fold, 256), dtype=torch.uint8, device=dev)
        self.it = 0

    def launches_per_step(self):
        return len(self.ms)

    def step(self, events=None, use_torch=False):
        for j, M in enumerate(self.ms):
            xs = self.X[M]
            x = xs[self.it % len(xs)]
            w = self.W[self.it % self.nw]
            if events is not None:
                events[j][0].record()
            if use_torch:
                torch.mm(x, w.t(), out=self.Y[M])
            else:
                self.bd.bi_gemm_bf16(x, w, out=self.Y[M], pins=self.pins, workspace=self.ws)
            if events is not None:
                events[j][1].record()
            self.it += 1

    def time_m(self, j, reps=20, use_torch=False):
        """Average device time of one launch at the j-th M, from `reps`
        back-to-back launches (rotating weight copies) between two events."""
        M = self.ms[j]
        xs = self.X[M]
        for i in range(3):
            self._launch(M, xs[i % len(xs)], self.W[i % self.nw], use_torch)
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        for i in range(reps):
            self._launch(M, xs[i % len(xs)], self.W[i % self.nw], use_torch)
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) * 1e3 / reps

    def median_m(self, j, reps=50, use_torch=False):
        """Median device time of one launch at the j-th M over `reps` launches,
        each between its own pair of events (rotating weight copies), after
        10 untimed launches."""
        M = self.ms[j]
        xs = self.X[M]
        for i in range(10):
            self._launch(M, xs[i % len(xs)], self.W[i % self.nw], use_torch)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for i in range(reps):
            ev[i][0].record()
            self._launch(M, xs[i % len(xs)], self.W[i % self.nw], use_torch)
            ev[i][1].record()
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) * 1e3 for a, b in ev]))

    def _launch(self, M, x, w, use_torch):
        if use_torch:
            torch.mm(x, w.t(), out=self.Y[M])
        else:
            self.bd.bi_gemm_bf16(x, w, out=self.Y[M], pins=self.pins, workspace=self.ws)

    def work(self):
        f = sum(gemm_work(M, self.N, self.K)[0] for M in self.ms)
        b = sum(gemm_work(M, self.N, self.K)[1] for M in self.ms)
        return f, b

    def e2e_step(self, host_x, host_y, batched=True, depth=2, chunk_rows=0):
        """Through the public API with host buffers: the rows of every M are
        copied in from pinned memory in chunks, multiplied and copied back into
        pinned memory, the copies of one chunk overlapping the GEMMs of the
        others.  batched: one bi_gemm_bf16_host_batch call over the sweep (one
        pipeline across the M boundaries); else bi_gemm_bf16_host once per M.
        depth: ring slots in the workspace; chunk_rows: rows per chunk of the
        batched call (0: the library's default)."""
        need = depth * self.bd.bi_gemm_bf16_host_slot_bytes(list(self.ms), self.N, self.K,
                                                            chunk_rows if batched else 0)
        if getattr(self, "host_ws", None) is None or self.host_ws.numel() != need:
            self.host_ws = torch.empty(need, dtype=torch.uint8, device=self.dev)
        h2d = sum(M * self.K * 2 for M in self.ms)
        d2h = sum(M * self.N * 2 for M in self.ms)
        if batched:
            ws = [self.W[(self.it + j) % self.nw] for j in range(len(self.ms))]
            self.bd.bi_gemm_bf16_host_batch([host_x[M] for M in self.ms], ws, outs=[host_y[M] for M in self.ms],
                                            pins=self.pins, workspace=self.host_ws, chunk_rows=chunk_rows)
            self.it += len(self.ms)
            return h2d, d2h
        for M in self.ms:
            self.bd.bi_gemm_bf16_host(host_x[M], self.W[self.it % self.nw], out=host_y[M], pins=self.pins,
                                      workspace=self.host_ws)
            self.it += 1
        return h2d, d2h


def torch_stack_forward(x, layers, shape):
    """The same decode-step stack with torch.mm and F.rms_norm (cuBLAS; not
    batch-invariant): the speed reference for the stack."""
    import torch.nn.functional as F
    s = shape
    M = x.shape[0]
    for L in layers:
        xn = F.rms_norm(x, (s.hidden,), L["g_attn"], s.eps)
        qkv = torch.mm(xn, L["Wqkv"].t())
        v = qkv[:, (s.n_q + s.n_kv) * s.head_dim:].reshape(M, s.n_kv, 1, s.head_dim)
        att = v.expand(M, s.n_kv, s.n_q // s.n_kv, s.head_dim).reshape(M, s.n_q * s.head_dim)
        h = x + torch.mm(att, L["Wo"].t())
        hn = F.rms_norm(h, (s.hidden,), L["g_mlp"], s.eps)
        gu = torch.mm(hn, L["Wgu"].t())
        act = F.silu(gu[:, :s.inter]) * gu[:, s.inter:]
        x = h + torch.mm(act, L["Wd"].t())
    return x


def run_stack(args, dist, peaks):
    """Configuration 5: the 4-layer Llama-3.1-70B-shaped decode step at 32 tokens."""
    from invariant_bi_gemm_bf16_gb300.stack import LLAMA31_70B, DecodeStack, random_layers
    from invariant_bi_gemm_bf16_gb300 import inputs
    shape = LLAMA31_70B
    layers = random_layers(shape, seed=dist.rank)
    stack = DecodeStack(shape, layers)
    x = inputs.device_normal((32, shape.hidden), seed=dist.rank, stream=0)
    for _ in range(args.warmup):
        stack.forward(x)
    t = dist.max(time_steps(lambda: stack.forward(x), args.steps, dist))
    us = t / args.steps * 1e6
    for _ in range(args.warmup):
        torch_stack_forward(x, layers, shape)
    tt = dist.max(time_steps(lambda: torch_stack_forward(x, layers, shape), args.steps, dist))
    tus = tt / args.steps * 1e6
    wbytes = sum(v.numel() * 2 for L in layers for v in L.values())
    roof_us = wbytes / (peaks["hbm_gbs"] * 1e3)
    res = {"workload": "4-layer Llama-3.1-70B-shaped decode step, 32 tokens, hidden 8192, GQA 64/8 x 128, "
                       "SwiGLU 28672, RMSNorm before attention and MLP; attention at a context of one token",
           "us_per_step": round(us, 1), "torch_us_per_step": round(tus, 1), "vs_torch": round(tus / us, 3),
           "weight_bytes": wbytes, "roofline_us": round(roof_us, 1), "roofline_frac": round(roof_us / us, 3),
           "bound": "hbm", "launches_per_step": stack.launches_per_step()}
    del stack, layers
    torch.cuda.empty_cache()
    return res


def time_reps(fn, reps):
    """Average device time (us) of one call, from `reps` back-to-back calls
    (fn(i) rotates its inputs) between two events, after 3 untimed calls."""
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for i in range(reps):
        fn(i)
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1e3 / reps


GRAPH_TIMING = ("per call: --per-m-reps calls captured in one CUDA graph and replayed between two CUDA "
                "events (ours and torch's alike), so host overhead is out of the timed region")


def time_graph(fn, reps):
    """Average device time (us) of one call when `reps` calls (fn(i) rotates
    its inputs) are captured in one CUDA graph and replayed: the host's
    per-call overhead (the Python binding, argument checks, tensor-map
    encoding) is out of the timed region, so small launches are timed on the
    device alone.  Warm-up: 3 eager calls, one replay."""
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    g.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1e3 / reps


def copies_for(nbytes: int, cap: int = 64) -> int:
    """Copies of a tensor so that consecutive calls never find it in L2."""
    return max(1, min(cap, math.ceil(2 * L2_BYTES / max(nbytes, 1)) + 1))


def run_rmsnorm(args, dist, peaks):
    """Configuration 4: RMSNorm over M tokens at H = 4096 and 8192; row m of X
    ~ N(0, s_m), s_m log-uniform on [0.1, 10] (drawn on the device from a
    seeded generator), g ~ N(1, 0.1), eps = 1e-5.  HBM-bound: B = 4MH + 2H."""
    import torch.nn.functional as F
    from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
    dev = torch.device("cuda", dist.local_rank)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + dist.rank)
    out = []
    for H in (4096, 8192):
        g = inputs.device_normal((H,), std=0.1, mean=1.0, seed=dist.rank, stream=inputs.STREAM_G, device=dev)
        for M in [1 << i for i in range(15)] + [3, 37, 1001]:
            n = copies_for(M * H * 2)
            xs = []
            for i in range(n):
                x = inputs.device_normal((M, H), seed=dist.rank, stream=inputs.STREAM_X + 16 * i, device=dev)
                scale = torch.exp(torch.empty((M, 1), device=dev).uniform_(math.log(0.1), math.log(10.0),
                                                                         generator=gen))
                xs.append((x.float() * scale).to(torch.bfloat16))
            y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
            us = time_graph(lambda i: bd.bi_rmsnorm_bf16(xs[i % n], g, 1e-5, out=y), args.per_m_reps)
            tus = time_graph(lambda i: F.rms_norm(xs[i % n], (H,), g, 1e-5), args.per_m_reps)
            b = 4 * M * H + 2 * H
            out.append({"H": H, "M": M, "us": round(us, 2), "gbs": round(b / us / 1e3, 1),
                        "roofline_frac": round(b / (peaks["hbm_gbs"] * 1e3) / us, 3),
                        "torch_rms_norm_us": round(tus, 2), "vs_torch": round(tus / us, 3)})
            del xs
    big = [r for r in out if r["M"] == 16384]
    return {"timing": GRAPH_TIMING, "workload": "RMSNorm, H in {4096, 8192}, M = 1..16384 and 3, 37, 1001; rows ~N(0, s_m), "
                        "s_m log-uniform on [0.1, 10]", "bound": "hbm",
            "largest": {("H%d" % r["H"]): {"gbs": r["gbs"], "roofline_frac": r["roofline_frac"],
                                           "vs_torch": r["vs_torch"]} for r in big},
            "sweep": out}


def run_fused(args, dist, peaks):
    """Configuration 3: RMSNorm + projection in one call (bi_rmsnorm_gemm_bf16)
    for the Llama-3.1-8B qkv [6144, 4096] and gate_up [28672, 4096] weights,
    against F.rms_norm + torch.mm on the same tensors."""
    import torch.nn.functional as F
    from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
    dev = torch.device("cuda", dist.local_rank)
    K = 4096
    g = inputs.device_normal((K,), std=0.1, mean=1.0, seed=dist.rank, stream=inputs.STREAM_G, device=dev)
    res = []
    for name, N in (("qkv", 6144), ("gate_up", 28672)):
        nw = copies_for(N * K * 2, cap=8)
        W = [inputs.device_normal((N, K), std=0.02, seed=dist.rank, stream=inputs.STREAM_W + 16 * i, device=dev)
             for i in range(nw)]
        pins = bd.bi_pins_default(N, K)
        pins = pins.replace(flags=pins.flags | bd.BI_FLAG_PREFETCH_W)
        for M in (1, 8, 32, 128, 1024, 4096, 8192):
            nx = copies_for(M * K * 2, cap=8)
            xs = [inputs.device_normal((M, K), seed=dist.rank, stream=inputs.STREAM_X + 16 * i, device=dev)
                  for i in range(nx)]
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            # the RMSNorm's scratch, with the GEMM's fold workspace in front (zeroed)
            ws = torch.zeros(bd.bi_rmsnorm_gemm_workspace_bytes(M, K) + bd.bi_gemm_bf16_workspace_bytes(M, N, K, pins),
                             dtype=torch.uint8, device=dev)
            us = time_graph(lambda i: bd.bi_rmsnorm_gemm_bf16(xs[i % nx], g, W[i % nw], 1e-5, pins=pins, out=y,
                                                             workspace=ws), args.per_m_reps)
            tus = time_graph(lambda i: torch.mm(F.rms_norm(xs[i % nx], (K,), g, 1e-5), W[i % nw].t(), out=y),
                            args.per_m_reps)
            f = 2.0 * M * N * K
            b = 2.0 * (N * K + M * K + M * N) + 2 * K
            t_roof = max(f / (peaks["bf16_tflops"] * 1e6), b / (peaks["hbm_gbs"] * 1e3))
            res.append({"proj": name, "N": N, "K": K, "M": M, "us": round(us, 2), "tflops": round(f / us / 1e6, 1),
                        "gbs": round(b / us / 1e3, 1), "roofline_frac": round(t_roof / us, 3),
                        "torch_us": round(tus, 2), "vs_torch": round(tus / us, 3)})
            del xs
        del W
        torch.cuda.empty_cache()
    return {"workload": "RMSNorm + projection in one call, Llama-3.1-8B qkv [6144,4096] and gate_up [28672,4096], "
                        "M in 1, 8, 32, 128, 1024, 4096, 8192; against F.rms_norm + torch.mm",
            "timing": GRAPH_TIMING, "sweep": res}


def run_lm_head(args, dist, peaks):
    """Llama-3.1-8B lm_head (V = 128256, K = 4096) and the per-token
    log-probabilities of given ids: bi_gemm_bf16 + bi_token_logprobs_bf16
    against torch.mm + log_softmax(float) + gather.  Also the full
    log-softmax kernel alone against its HBM roofline (B = 6 M V)."""
    from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
    dev = torch.device("cuda", dist.local_rank)
    V, K = 128256, 4096
    nw = copies_for(V * K * 2, cap=4)
    W = [inputs.device_normal((V, K), std=0.02, seed=dist.rank, stream=inputs.STREAM_W + 16 * i, device=dev)
         for i in range(nw)]
    pins = bd.bi_pins_default(V, K)
    pins = pins.replace(flags=pins.flags | bd.BI_FLAG_PREFETCH_W)
    res = []
    for M in (1, 32, 256):
        nx = copies_for(M * K * 2, cap=8)
        hs = [inputs.device_normal((M, K), seed=dist.rank, stream=inputs.STREAM_X + 16 * i, device=dev)
              for i in range(nx)]
        ids = torch.randint(0, V, (M,), dtype=torch.int32, device=dev,
                            generator=torch.Generator(device=dev).manual_seed(7))
        ids64 = ids.long().unsqueeze(1)
        logits = torch.empty((M, V), dtype=torch.bfloat16, device=dev)
        lp = torch.empty(M, dtype=torch.float32, device=dev)

        def ours(i):
            bd.bi_gemm_bf16(hs[i % nx], W[i % nw], out=logits, pins=pins)
            bd.bi_token_logprobs_bf16(logits, ids, out=lp)

        def theirs(i):
            lg = torch.mm(hs[i % nx], W[i % nw].t())
            torch.log_softmax(lg.float(), dim=-1).gather(1, ids64)

        us = time_graph(ours, args.per_m_reps)
        tus = time_graph(theirs, args.per_m_reps)
        # the log-softmax kernels alone, on resident logits
        nl = copies_for(M * V * 2, cap=16)
        ls = [inputs.device_normal((M, V), std=3.0, seed=dist.rank, stream=40 + i, device=dev) for i in range(nl)]
        yf = torch.empty((M, V), dtype=torch.float32, device=dev)
        us_tok = time_graph(lambda i: bd.bi_token_logprobs_bf16(ls[i % nl], ids, out=lp), args.per_m_reps)
        us_full = time_graph(lambda i: bd.bi_log_softmax_bf16(ls[i % nl], out=yf), args.per_m_reps)
        tus_full = time_graph(lambda i: torch.log_softmax(ls[i % nl].float(), dim=-1), args.per_m_reps)
        b_full = 6.0 * M * V
        res.append({"M": M, "us": round(us, 2), "torch_us": round(tus, 2), "vs_torch": round(tus / us, 3),
                    "token_logprobs_us": round(us_tok, 2), "log_softmax_us": round(us_full, 2),
                    "log_softmax_gbs": round(b_full / us_full / 1e3, 1),
                    "log_softmax_roofline_frac": round(b_full / (peaks["hbm_gbs"] * 1e3) / us_full, 3),
                    "torch_log_softmax_us": round(tus_full, 2)})
        del hs, ls
    del W
    torch.cuda.empty_cache()
    return {"timing": GRAPH_TIMING, "workload": "Llama-3.1-8B lm_head W[128256,4096] + per-token log-probabilities of given ids, "
                        "M in 1, 32, 256; against torch.mm + log_softmax + gather", "sweep": res}


def run_fp8(args, dist, peaks):
    """FP8 (E4M3, per-token and per-channel scales) on the down_proj shape:
    bi_quantize_rows_e4m3 of the activations + bi_gemm_fp8, against torch.mm
    in bf16 on the unquantised tensors.  Peak: the measured bf16 burst peak x 2,
    the nominal FP8 / bf16 ratio of dense tensor throughput."""
    from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
    dev = torch.device("cuda", dist.local_rank)
    N, K = DOWN_N, DOWN_K
    nw = copies_for(N * K, cap=6)
    Ws = [inputs.device_normal((N, K), std=0.02, seed=dist.rank, stream=inputs.STREAM_W + 16 * i, device=dev)
          for i in range(nw)]
    wq = [bd.bi_quantize_rows_e4m3(w) for w in Ws]
    pins = bd.bi_pins_default_fp8(N, K)
    pins = pins.replace(flags=pins.flags | bd.BI_FLAG_PREFETCH_W)
    peak8 = 2.0 * peaks["bf16_tflops"]
    baseline = "torch.mm in bf16 on the unquantised tensors"
    res = []
    for M in (1, 128, 512, 2048, 8192):
        nx = copies_for(M * K * 2, cap=8)
        xs = [inputs.device_normal((M, K), seed=dist.rank, stream=inputs.STREAM_X + 16 * i, device=dev)
              for i in range(nx)]
        xq = [bd.bi_quantize_rows_e4m3(x) for x in xs]
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        us_gemm = time_graph(lambda i: bd.bi_gemm_fp8(xq[i % nx][0], xq[i % nx][1], wq[i % nw][0], wq[i % nw][1],
                                                     out=y, pins=pins), args.per_m_reps)
        qbuf = (torch.empty((M, K), dtype=torch.uint8, device=dev), torch.empty(M, dtype=torch.float32, device=dev))

        def layer(i):
            q, sxv = bd.bi_quantize_rows_e4m3(xs[i % nx], q=qbuf[0], scale=qbuf[1])
            bd.bi_gemm_fp8(q, sxv, wq[i % nw][0], wq[i % nw][1], out=y, pins=pins)
        us_layer = time_graph(layer, args.per_m_reps)
        us_q = time_graph(lambda i: bd.bi_quantize_rows_e4m3(xs[i % nx], q=qbuf[0], scale=qbuf[1]), args.per_m_reps)
        bq = 3.0 * M * K + 4.0 * M   # bf16 in, E4M3 codes and fp32 scales out
        tus = time_graph(lambda i: torch.mm(xs[i % nx], Ws[i % nw].t(), out=y), args.per_m_reps)
        f = 2.0 * M * N * K
        b = float(N * K + M * K + 2 * M * N + 4 * (M + N))
        t_roof = max(f / (peak8 * 1e6), b / (peaks["hbm_gbs"] * 1e3))
        res.append({"M": M, "gemm_us": round(us_gemm, 2), "tflops": round(f / us_gemm / 1e6, 1),
                    "roofline_frac": round(t_roof / us_gemm, 3), "quantize_and_gemm_us": round(us_layer, 2),
                    "quantize_us": round(us_q, 2),
                    "quantize_hbm_frac": round(bq / us_q / 1e3 / peaks["hbm_gbs"], 3),
                    "baseline_us": round(tus, 2), "vs_baseline": round(tus / us_gemm, 3)})
        del xs, xq
    del Ws, wq
    torch.cuda.empty_cache()
    # the FP8 RMSNorm prologue (Llama-3.1-8B hidden 4096): one pass against
    # bi_rmsnorm_bf16 followed by bi_quantize_rows_e4m3
    H = 4096
    g = inputs.device_normal((H,), std=0.1, mean=1.0, seed=dist.rank, stream=inputs.STREAM_G, device=dev)
    pro = []
    for M in (1, 128, 2048, 8192):
        nx = copies_for(M * H * 2, cap=8)
        xs = [inputs.device_normal((M, H), seed=dist.rank, stream=inputs.STREAM_X + 16 * i, device=dev)
              for i in range(nx)]
        q = torch.empty((M, H), dtype=torch.uint8, device=dev)
        sc = torch.empty(M, dtype=torch.float32, device=dev)
        yb = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        us_f = time_graph(lambda i: bd.bi_rmsnorm_quantize_e4m3(xs[i % nx], g, EPS, q=q, scale=sc), args.per_m_reps)

        def two(i):
            bd.bi_rmsnorm_bf16(xs[i % nx], g, EPS, out=yb)
            bd.bi_quantize_rows_e4m3(yb, q=q, scale=sc)
        us_2 = time_graph(two, args.per_m_reps)
        bf = 3.0 * M * H + 4.0 * M + 2.0 * H   # bf16 in, codes and scales out, the gain
        pro.append({"M": M, "fused_us": round(us_f, 2), "fused_hbm_frac": round(bf / us_f / 1e3 / peaks["hbm_gbs"], 3),
                    "rmsnorm_then_quantize_us": round(us_2, 2), "speedup": round(us_2 / us_f, 3)})
        del xs
    torch.cuda.empty_cache()
    return {"timing": GRAPH_TIMING, "workload": "FP8 E4M3 down_proj W[4096,14336], per-token activation and per-channel weight scales",
            "peak_tflops": peak8, "peak_source": "measured bf16 burst x 2 (nominal FP8 / bf16 ratio)",
            "baseline": baseline, "sweep": res,
            "rmsnorm_quantize": {"workload": "bi_rmsnorm_quantize_e4m3, H = 4096, against bi_rmsnorm_bf16 + "
                                             "bi_quantize_rows_e4m3", "sweep": pro}}


ATTN_HEADS = (64, 8, 128, 16)   # query heads, key/value heads, head dim, page size
ATTN_MIXES = [("64 requests, lengths uniform on [512, 8192]", 64, (512, 8192)),
              ("256 requests, lengths uniform on [64, 2048]", 256, (64, 2048)),
              ("1 request of 32768", 1, (32768, 32768))]


def attention_case(mix, dist, dev):
    """(name, lengths, (k_cache, v_cache, block_table, seq_lens, q)) of one request mix."""
    from invariant_bi_gemm_bf16_gb300 import inputs
    Hq, Hkv, D, P = ATTN_HEADS
    name, B, (lo, hi) = ATTN_MIXES[mix]
    rng = np.random.default_rng(70 + dist.rank)
    lens = [int(x) for x in rng.integers(lo, hi + 1, size=B)]
    kc, vc, bt, sl = inputs.device_paged_kv(lens, Hkv, D, P, seed=70 + dist.rank, device=dev)
    q = inputs.device_normal((B, Hq, D), seed=70 + dist.rank, stream=0, device=dev)
    return name, lens, (kc, vc, bt, sl, q)


def run_attention(args, dist, peaks):
    """Decode attention over a paged cache (Llama-3.1-70B heads: 64 query
    heads, 8 key/value heads, D = 128; pages of 16 in shuffled order) against
    its HBM roofline, for three request mixes.  Algorithmic bytes per call:
    the keys and values of every request's positions, q and the output.  The
    caches are larger than L2, so consecutive calls find none of them there.
    Context: torch's scaled_dot_product_attention on the same requests padded
    to the longest, with a length mask (torch has no paged decode attention)."""
    from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
    import torch.nn.functional as F
    dev = torch.device("cuda", dist.local_rank)
    Hq, Hkv, D, P = ATTN_HEADS
    res = []
    for mix in range(len(ATTN_MIXES)):
        name, lens, (kc, vc, bt, sl, q) = attention_case(mix, dist, dev)
        B = len(lens)
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
        max_len = bt.shape[1] * P
        alg = sum(lens) * Hkv * D * 2 * 2 + 2 * B * Hq * D * 2
        row = {"mix": name, "kv_bytes": sum(lens) * Hkv * D * 4, "splits": []}
        for S in (128, 256, 320, 512, 576, 1024):
            ws = torch.empty(bd.bi_decode_attention_workspace_bytes(B, Hq, Hkv, max_len, S), dtype=torch.uint8,
                             device=dev)
            us = time_graph(lambda i: bd.bi_decode_attention_bf16(q, kc, vc, bt, sl, D ** -0.5, max_seq_len=max_len,
                                                                 split_size=S, out=out, workspace=ws),
                           args.per_m_reps)
            row["splits"].append({"split": S, "us": round(us, 2), "gbs": round(alg / us / 1e3, 1),
                                  "roofline_frac": round(alg / us / 1e3 / peaks["hbm_gbs"], 3)})
            del ws
        if bd.bi_last_device_status() != bd.BI_OK:
            raise RuntimeError("decode attention reported a device-side error")
        try:
            Lmax = max(lens)
            if B * Hkv * Lmax * D * 2 * 2 <= (8 << 30):
                Kd = torch.zeros((B, Hkv, Lmax, D), dtype=torch.bfloat16, device=dev)
                Vd = torch.zeros_like(Kd)
                for b, L in enumerate(lens):
                    pos = torch.arange(L, device=dev)
                    pages = bt[b].long()[pos // P]
                    Kd[b, :, :L] = kc[pages, pos % P].transpose(0, 1)
                    Vd[b, :, :L] = vc[pages, pos % P].transpose(0, 1)
                mask = (torch.arange(Lmax, device=dev)[None, :] < sl[:, None]).view(B, 1, 1, Lmax)
                q4 = q.view(B, Hq, 1, D)
                tus = time_reps(lambda i: F.scaled_dot_product_attention(q4, Kd, Vd, attn_mask=mask, enable_gqa=True),
                                args.per_m_reps)
                row["torch_sdpa_padded_us"] = round(tus, 2)
                del Kd, Vd
        except Exception as e:  # noqa: BLE001 - context only
            row["torch_sdpa_padded_us"] = None
            row["torch_sdpa_error"] = type(e).__name__
        res.append(row)
        del kc, vc, q
        torch.cuda.empty_cache()
    return {"timing": GRAPH_TIMING, "workload": "decode attention, Llama-3.1-70B heads (64 q, 8 kv, D 128), paged cache (pages of 16, "
                        "shuffled), fixed split sizes 128..1024", "mixes": res}


def time_steps(fn, steps, dist):
    dist.barrier()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        fn()
    e.record()
    torch.cuda.synchronize()
    dist.barrier()
    return s.elapsed_time(e) / 1e3  # seconds


def run_ours(args, dist):
    from invariant_bi_gemm_bf16_gb300 import binding as bd
    bd.load()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    wl = DownProjSweep(bd, dev, seed=dist.rank)
    L = wl.launches_per_step()

    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()

    # timed region: K whole steps between two CUDA events on the launching
    # stream (no events between launches, so consecutive kernels overlap their
    # ramp-up and drain exactly as in a real sweep)
    clocks = ClockSampler(smi_gpu_id(dist.local_rank))
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    t_start.record()
    for k in range(args.steps):
        wl.step()
    t_end.record()
    torch.cuda.synchronize()
    clocks.mark_end()
    dist.barrier()
    clk = clocks.stop()
    status = bd.bi_last_device_status()
    if status != bd.BI_OK:
        raise RuntimeError("device stall status: %s" % bd.status_string(status))
    wall = t_start.elapsed_time(t_end) / 1e3
    # per-M launch durations: R back-to-back launches of one M between two events
    per_launch = np.array([[wl.time_m(j, reps=args.per_m_reps)] for j in range(L)]).T  # us
    wall_max = dist.max(wall)
    flops, bytes_ = wl.work()
    total_flops = dist.sum(flops * args.steps)
    value = total_flops / wall_max / 1e12

    # torch.mm on the same tensors, same protocol
    torch_launch = np.array([[wl.time_m(j, reps=args.per_m_reps, use_torch=True)] for j in range(L)]).T
    med = [wl.median_m(j) for j in range(L)]
    torch_med = [wl.median_m(j, use_torch=True) for j in range(L)]
    def graph_m(j, use_torch):
        M = wl.ms[j]
        xs = wl.X[M]
        return time_graph(lambda i: wl._launch(M, xs[i % len(xs)], wl.W[i % wl.nw], use_torch), args.per_m_reps)
    gr = [graph_m(j, False) for j in range(L)]
    torch_gr = [graph_m(j, True) for j in range(L)]
    torch_wall = time_steps(lambda: wl.step(use_torch=True), args.steps, dist)
    sweep = []
    sum_roof = 0.0
    sum_meas = 0.0
    for j, M in enumerate(wl.ms):
        us = float(per_launch[0, j])
        tus = float(torch_launch[0, j])
        f, b = gemm_work(M, wl.N, wl.K)
        tr = roof_time_us(f, b, peaks)
        sum_roof += tr
        sum_meas += us
        bound = "tensor" if f / (peaks["bf16_tflops"] * 1e6) >= b / (peaks["hbm_gbs"] * 1e3) else "hbm"
        sweep.append({"M": M, "us": round(us, 2), "tflops": round(f / us / 1e6, 1),
                      "gbs": round(b / us / 1e3, 1), "bound": bound, "roofline_frac": round(tr / us, 3),
                      "torch_mm_us": round(tus, 2), "vs_torch_mm": round(tus / us, 3),
                      "us_median50": round(med[j], 2), "torch_mm_us_median50": round(torch_med[j], 2),
                      "us_graph": round(gr[j], 2), "torch_mm_us_graph": round(torch_gr[j], 2)})

    # e2e through the C ABI with host buffers
    host_x = {M: wl.X[M][0].cpu().pin_memory() for M in wl.ms}
    host_y = {M: torch.empty((M, wl.N), dtype=torch.bfloat16).pin_memory() for M in wl.ms}
    holder = {}
    # chunks of about e2e_chunk_mb MB of X for the batched call (a multiple of 128 rows)
    chunk_rows = max(128, ((args.e2e_chunk_mb << 20) // (2 * wl.K)) // 128 * 128)

    def e2e_time(batched):
        for _ in range(max(1, args.warmup // 2)):
            wl.e2e_step(host_x, host_y, batched, args.e2e_depth, chunk_rows)
        torch.cuda.synchronize()

        def e2e():
            holder["b"] = wl.e2e_step(host_x, host_y, batched, args.e2e_depth, chunk_rows)
        wall = dist.max(time_steps(e2e, args.steps, dist))
        return dist.sum(flops * args.steps) / wall / 1e12
    e2e_per_call = e2e_time(False)
    e2e_value = e2e_time(True)
    h2d, d2h = holder["b"]

    launch_sum = float(per_launch.sum()) / 1e6          # one sweep, seconds
    sweep_tflops = flops / launch_sum / 1e12
    traffic = NCU_TRAFFIC.get(build_fingerprint() or "", {})
    # the dominant launch of the step (largest M, the biggest share of its time)
    j_big = len(wl.ms) - 1
    M_big = wl.ms[j_big]
    f_big, b_big = gemm_work(M_big, wl.N, wl.K)
    ach_big = f_big / (float(per_launch[0, j_big]) * 1e-6) / 1e12
    roof = {"bound": "tensor", "achieved": round(ach_big, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(ach_big / peaks["bf16_tflops"], 3), "traffic": traffic.get(M_big),
            "algorithmic_bytes": int(b_big), "launch": "bi_gemm_bf16_ws at M=%d (%.0f%% of the step's time)" % (
                M_big, 100.0 * float(per_launch[0, j_big]) / float(per_launch.sum())),
            "peak_source": peaks["source"] + " (burst bf16; launches timed back to back)"}
    # the decode end of the sweep: HBM-bound
    M_small = wl.ms[0]
    f_s, b_s = gemm_work(M_small, wl.N, wl.K)
    ach_s = b_s / (float(per_launch[0, 0]) * 1e-6) / 1e9
    roof_decode = {"bound": "hbm", "achieved": round(ach_s, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                   "frac": round(ach_s / peaks["hbm_gbs"], 3), "traffic": traffic.get(M_small),
                   "algorithmic_bytes": int(b_s), "launch": "bi_gemm_bf16_ws at M=%d" % M_small,
                   "peak_source": peaks["source"] + " (copy bandwidth)"}
    sweep_roof = {"tflops": round(sweep_tflops, 1), "frac_of_bf16_peak": round(sweep_tflops / peaks["bf16_tflops"], 3),
                  "time_weighted_roofline_frac": round(sum_roof / sum_meas, 3),
                  "note": "whole sweep: FLOPs / summed per-launch times; per-M bound and fraction in sweep[]"}
    result = {
        "metric": "batch-invariant GEMM TFLOPS over the down_proj M sweep (M=1..8192)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(wall_max / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
        "config": {"workload": "Llama-3.1-8B down_proj W[4096,14336], M in 1,2,4..8192, one call per M",
                   "N": wl.N, "K": wl.K, "M_sweep": wl.ms, "pins": wl.pins.as_dict(),
                   "l2": "no flush; %d weight copies (%.0f MB) and rotating activations so no launch "
                         "reads what the previous launch left in L2" % (wl.nw, wl.nw * wl.N * wl.K * 2 / 1e6),
                   "parallelism": "replicas x%d (rows sharded, no collective)" % dist.world},
        "roofline": roof,
        "roofline_decode": roof_decode,
        "sweep_roofline": sweep_roof,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "api": "one bi_gemm_bf16_host_batch call over the sweep's 14 jobs (pinned host X and Y, "
                       "chunks of %d rows copied in and out while other chunks multiply, across the M "
                       "boundaries; ring of %d slots)" % (chunk_rows, args.e2e_depth)},
        "e2e_per_call": {"value": round(e2e_per_call, 2), "unit": "TFLOP/s",
                         "api": "bi_gemm_bf16_host once per M (default chunks of about 16 MB of X; ring of %d "
                                "slots)" % args.e2e_depth},
        "gpu_launches": L * args.steps,
        "per_m_timing": ("us: %d back-to-back launches of that M between two CUDA events (mean); us_median50: "
                         "median of 50 launches, each between its own events, after 10 warm-up launches; "
                         "us_graph: %d launches captured in one CUDA graph and replayed (device time only, no "
                         "host overhead)" % (args.per_m_reps, args.per_m_reps)),
        "clocks": clk,
        "sweep": sweep,
        "torch_mm_sweep_tflops": round(flops * args.steps / torch_wall / 1e12, 1),
    }
    if not args.no_stack:
        result["stack"] = run_stack(args, dist, peaks)
    if not args.no_fused:
        result["fused"] = run_fused(args, dist, peaks)
    if not args.no_rmsnorm:
        result["rmsnorm"] = run_rmsnorm(args, dist, peaks)
    if not args.no_lm_head:
        result["lm_head"] = run_lm_head(args, dist, peaks)
    if not args.no_fp8:
        result["fp8"] = run_fp8(args, dist, peaks)
    if not args.no_attention:
        result["attention"] = run_attention(args, dist, peaks)
    if dist.rank == 0 and not args.no_cpu_baseline:
        tf, secs, rows, threads = oracle_gemm_throughput(target_s=args.cpu_seconds)
        tf1, dt1 = oracle_gemm_1thread(16)
        result["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                  "sample": "oracle down_proj GEMM on %d rows x all 4096 outputs (K=14336), "
                                            "%.1f s" % (rows, secs), "model": cpu_model(),
                                  "value_1thread": round(tf1, 6), "sample_1thread": "%d rows, %.1f s" % (16, dt1)}
    return result


def run_single_m(args, dist):
    """Launches the sweep's GEMM (same tensors, pins and weight rotation) at one
    M, --launches times, for an ncu capture of that launch."""
    from invariant_bi_gemm_bf16_gb300 import binding as bd
    bd.load()
    torch.cuda.set_device(dist.local_rank)
    wl = DownProjSweep(bd, torch.device("cuda", dist.local_rank), seed=dist.rank, sweep=[args.single_m])
    for i in range(args.launches):
        wl._launch(args.single_m, wl.X[args.single_m][i % len(wl.X[args.single_m])], wl.W[i % wl.nw], False)
    torch.cuda.synchronize()
    st = bd.bi_last_device_status()
    if st != bd.BI_OK:
        raise RuntimeError(bd.status_string(st))


def run_single_gemm(args, dist):
    """Launches bi_gemm_bf16_ws with the default pins (plus the early weight
    stream) and a zeroed fold workspace on one shape N:K:M, --launches times
    on rotating weight copies larger than L2, for an ncu capture of those
    launches (the decode projections' GLOBAL schedule, for one)."""
    from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
    bd.load()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    N, K, M = (int(v) for v in args.single_gemm.split(":"))
    nw = copies_for(N * K * 2, cap=8)
    W = [inputs.device_normal((N, K), std=0.02, seed=dist.rank, stream=inputs.STREAM_W + 16 * i, device=dev)
         for i in range(nw)]
    x = inputs.device_normal((M, K), seed=dist.rank, stream=inputs.STREAM_X, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    pins = bd.bi_pins_default(N, K)
    pins = pins.replace(flags=pins.flags | bd.BI_FLAG_PREFETCH_W)
    ws = torch.zeros(max(bd.bi_gemm_bf16_workspace_bytes(M, N, K, pins), 256), dtype=torch.uint8, device=dev)
    plan = bd.bi_gemm_plan_describe_ws(M, N, K, pins, 0, ws.numel())
    print(json.dumps({"single_gemm": [N, K, M], "schedule": plan.schedule, "split_k": plan.split_k,
                      "tok_tile": plan.tok_tile, "grid": [plan.grid_x, plan.grid_y, plan.grid_z]}), flush=True)
    for i in range(args.launches):
        bd.bi_gemm_bf16(x, W[i % nw], out=y, pins=pins, workspace=ws)
    torch.cuda.synchronize()
    st = bd.bi_last_device_status()
    if st != bd.BI_OK:
        raise RuntimeError(bd.status_string(st))


def run_single_attention(args, dist):
    """Launches decode attention on one request mix (MIX:SPLIT), --launches
    times, for an ncu capture of those launches."""
    from invariant_bi_gemm_bf16_gb300 import binding as bd
    bd.load()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    mix, split = (int(x) for x in args.single_attention.split(":"))
    _, lens, (kc, vc, bt, sl, q) = attention_case(mix, dist, dev)
    D, P = ATTN_HEADS[2], ATTN_HEADS[3]
    for _ in range(args.launches):
        bd.bi_decode_attention_bf16(q, kc, vc, bt, sl, D ** -0.5, max_seq_len=bt.shape[1] * P, split_size=split)
    torch.cuda.synchronize()
    st = bd.bi_last_device_status()
    if st != bd.BI_OK:
        raise RuntimeError(bd.status_string(st))


def run_single_rmsnorm(args, dist):
    """Launches RMSNorm on one shape (H:M), or RMSNorm with the E4M3
    quantisation (H:M:q), --launches times on rotating inputs, for an ncu
    capture of those launches."""
    from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
    bd.load()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    parts = args.single_rmsnorm.split(":")
    H, M = int(parts[0]), int(parts[1])
    quant = len(parts) > 2 and parts[2] == "q"
    n = copies_for(M * H * 2, cap=8)
    xs = [inputs.device_normal((M, H), seed=dist.rank, stream=60 + i, device=dev) for i in range(n)]
    g = inputs.device_normal((H,), std=0.1, mean=1.0, seed=dist.rank, stream=inputs.STREAM_G, device=dev)
    y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    q = torch.empty((M, H), dtype=torch.uint8, device=dev)
    sc = torch.empty(M, dtype=torch.float32, device=dev)
    for i in range(args.launches):
        if quant:
            bd.bi_rmsnorm_quantize_e4m3(xs[i % n], g, EPS, q=q, scale=sc)
        else:
            bd.bi_rmsnorm_bf16(xs[i % n], g, EPS, out=y)
    torch.cuda.synchronize()


def run_single_quantize(args, dist):
    """Launches the per-row E4M3 quantisation on one shape (M:K), --launches
    times on rotating inputs, for an ncu capture of those launches."""
    from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
    bd.load()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    M, K = (int(x) for x in args.single_quantize.split(":"))
    n = copies_for(M * K * 2, cap=8)
    xs = [inputs.device_normal((M, K), seed=dist.rank, stream=80 + i, device=dev) for i in range(n)]
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sc = torch.empty((M,), dtype=torch.float32, device=dev)
    for i in range(args.launches):
        bd.bi_quantize_rows_e4m3(xs[i % n], q=q, scale=sc)
    torch.cuda.synchronize()


def run_single_logsoftmax(args, dist):
    """Launches the full log-softmax and the token log-probabilities on M rows
    of Llama-3.1-8B logits (V = 128256), --launches times each on rotating
    inputs, for an ncu capture of those launches."""
    from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
    bd.load()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    M, V = int(args.single_logsoftmax), 128256
    n = copies_for(M * V * 2, cap=8)
    xs = [inputs.device_normal((M, V), std=3.0, seed=dist.rank, stream=70 + i, device=dev) for i in range(n)]
    ids = torch.arange(M, dtype=torch.int32, device=dev) * 97 % V
    y = torch.empty((M, V), dtype=torch.float32, device=dev)
    for i in range(args.launches):
        bd.bi_log_softmax_bf16(xs[i % n], out=y)
        bd.bi_token_logprobs_bf16(xs[i % n], ids)
    torch.cuda.synchronize()


def run_reference(args, dist):
    """The reference arm: the CPU oracle on a bounded sample of the same workload."""
    if dist.rank != 0:
        return None
    step_s = min(args.ref_step_seconds, 150.0 / max(1, args.steps))
    oracle_inputs(2048)
    for _ in range(args.warmup):
        oracle_gemm_throughput(target_s=0.05, max_rows=2048)
    vals = []
    t0 = time.perf_counter()
    info = None
    for _ in range(args.steps):
        info = oracle_gemm_throughput(target_s=step_s, max_rows=2048)
        vals.append(info[0])
    total = time.perf_counter() - t0
    value = statistics.median(vals)
    return {"impl": "reference", "metric": "batch-invariant GEMM TFLOPS over the down_proj M sweep (M=1..8192)",
            "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
            "config": {"workload": "Llama-3.1-8B down_proj W[4096,14336], M in 1,2,4..8192, one call per M",
                       "N": DOWN_N, "K": DOWN_K},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": info[3], "kind": "oracle",
                             "sample": "per step: oracle down_proj GEMM on %d rows x 4096 outputs" % info[2]},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=6.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stack", action="store_true")
    ap.add_argument("--no-fused", action="store_true")
    ap.add_argument("--no-rmsnorm", action="store_true")
    ap.add_argument("--no-lm-head", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-attention", action="store_true")
    ap.add_argument("--per-m-reps", type=int, default=20)
    ap.add_argument("--e2e-depth", type=int, default=8, help="ring slots of the host-buffer GEMM's workspace")
    ap.add_argument("--e2e-chunk-mb", type=int, default=64, help="MB of X per chunk of the batched host GEMM")
    ap.add_argument("--single-quantize", default="",
                    help="M:K: only launch the E4M3 quantisation on that shape (for ncu)")
    ap.add_argument("--single-logsoftmax", default="",
                    help="M: only launch the log-softmax kernels on M rows of V = 128256 logits (for ncu)")
    ap.add_argument("--single-rmsnorm", default="",
                    help="H:M -- only launch RMSNorm on that shape (H:M:q: RMSNorm with the E4M3 quantisation) (for ncu)")
    ap.add_argument("--single-attention", default="",
                    help="MIX:SPLIT -- only launch decode attention on that request mix (for ncu)")
    ap.add_argument("--single-gemm", default="",
                    help="N:K:M -- only launch bi_gemm_bf16_ws on that shape --launches times (for ncu)")
    ap.add_argument("--single-m", type=int, default=0,
                    help="profiling helper: only launch the sweep's GEMM at this M --launches times")
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    dist = Dist()
    try:
        if args.single_attention:
            run_single_attention(args, dist)
            return
        if args.single_quantize:
            run_single_quantize(args, dist)
            return
        if args.single_logsoftmax:
            run_single_logsoftmax(args, dist)
            return
        if args.single_rmsnorm:
            run_single_rmsnorm(args, dist)
            return
        if args.single_m:
            run_single_m(args, dist)
            return
        if args.single_gemm:
            run_single_gemm(args, dist)
            return
        if args.impl == "reference":
            res = run_reference(args, dist)
        else:
            res = run_ours(args, dist)
        if dist.rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
