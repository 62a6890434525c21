"""Offline pin tuner for the GEMM family.

Detent: Batch-Invariant LLM Serving and RL Rollouts at Near-Stock Speed,
Sec. 6 (Tuner) and Eq. 3, restated for this library:

* A *family* is one GEMM shape (N, K).  Its pins are a ``bi_pins`` tuple
  (split count S, token tile T, CTA grouping, W ring depth, copy-size flag).
  The batch size M is never a pin and never reaches the choice: one tuple
  serves every M of the family.
* A recorded workload gives each family its distinct calls c (here: M) with
  counts n.  With C the time of all other work, the workload's time under a
  tuple a = (a_f) is T(a) = C + sum_f T_f(a_f), T_f(a_f) = sum_(c,n) n * t_f(c, a_f),
  so the best tuple is the per-family argmin of T_f, and the search costs the
  sum, not the product, of the families' grid sizes.
* If the sum holds only within a relative error delta, the per-family tuple is
  within (1 + delta) / (1 - delta) of the best tuple (``delta_bound``).
* Legality: every candidate passes ``bi_pins_validate`` before it is timed;
  the library checks the pins again on every call, and a tuned table is
  re-validated when it is loaded.
* Search: coordinate descent from the default pins over the grid's axes,
  measuring a part of the grid (``search``); ``exhaustive`` measures all of it.

Decode attention's split size is tuned the same way (Detent, Sec. 7: the tuner
also picks FA3's split stride like a pin).  A family is one head layout (query
heads, key/value heads, page size); its calls are decode steps, each a list of
request lengths with a count; the split size is the argmin of the family's
summed time over the legal sizes (multiples of 64 up to 4096), all measured.

Timing: each (candidate, M) is timed as calls of bi_gemm_bf16_ws (with a fold
workspace, so that the GLOBAL schedule is open to split counts whose clusters
would not fit the GPU at once) captured in a CUDA graph and replayed between
two CUDA events, on rotating weight copies (more bytes than L2), after
warm-up calls.  The graph keeps the binding's per-call host time out of the
measurement: a decode call takes about as long on the host as on the GPU, and
timed back to back from Python every candidate would look alike.  A
candidate's cost takes the fastest of a few repeats (the SM clock drifts under
the power cap).  The winner must then beat the default tuple by a margin
in interleaved re-measurements (``confirm``), else the default is kept.
"""
from __future__ import annotations

import itertools
import json
import math
from typing import Callable, Dict, Iterable, List, Sequence, Tuple

from . import binding as bd

FORMAT = "bi_gemm_pins/1"
L2_BYTES = 129 * 1024 * 1024

# Axes of the legal grid of one family, in the order coordinate descent visits them.
SPLITS = (1, 2, 3, 4, 5, 6, 7, 8, 12, 16)
TOK_TILES = (128, 256)
GROUPINGS = (0, 1, 2)
STAGES = (0, 4)
COPY_FLAGS = (0, bd.BI_FLAG_KTILE_PAIRS)


# --------------------------------------------------------------------------- workload

class Recorder:
    """Counts the GEMM calls of a workload per family: {(N, K): {M: n}}.

    Used as a context manager around code that calls the binding (the
    binding reports every bi_gemm_bf16 / bi_rmsnorm_gemm_bf16 call to the
    active recorders)."""

    def __init__(self):
        self.calls: Dict[Tuple[int, int], Dict[int, int]] = {}

    def add(self, M: int, N: int, K: int, n: int = 1):
        fam = self.calls.setdefault((int(N), int(K)), {})
        fam[int(M)] = fam.get(int(M), 0) + int(n)

    def __enter__(self):
        bd.add_call_hook(self.add)
        return self

    def __exit__(self, *exc):
        bd.remove_call_hook(self.add)
        return False

    def families(self) -> Dict[Tuple[int, int], List[Tuple[int, int]]]:
        return {k: sorted(v.items()) for k, v in self.calls.items()}


# --------------------------------------------------------------------------- grid

def candidate(N: int, K: int, S: int, T: int, ctas: int, stages: int, copy_flag: int,
              base_flags: int = bd.BI_FLAG_SCHEDULE_AUTO) -> bd.Pins:
    p = bd.bi_pins_default(N, K)
    return p.replace(split_k=S, tok_tile=T, mma_ctas=ctas, stages=stages,
                     flags=(base_flags & ~bd.BI_FLAG_KTILE_PAIRS) | copy_flag)


def axes(N: int, K: int) -> Dict[str, Sequence[int]]:
    kt = -(-K // bd.BI_BK)
    return {"S": tuple(s for s in SPLITS if s <= kt), "T": TOK_TILES, "ctas": GROUPINGS,
            "stages": STAGES, "copy": COPY_FLAGS}


def key_of(p: bd.Pins) -> Tuple[int, int, int, int, int]:
    return (p.split_k, p.tok_tile, p.mma_ctas, p.stages, p.flags & bd.BI_FLAG_KTILE_PAIRS)


def legal_grid(N: int, K: int, base_flags: int = bd.BI_FLAG_SCHEDULE_AUTO) -> List[bd.Pins]:
    """Every legal tuple of the family's grid (bi_pins_validate == BI_OK)."""
    ax = axes(N, K)
    out = []
    for S, T, c, st, cf in itertools.product(ax["S"], ax["T"], ax["ctas"], ax["stages"], ax["copy"]):
        p = candidate(N, K, S, T, c, st, cf, base_flags)
        if bd.bi_pins_validate(N, K, p) == bd.BI_OK:
            out.append(p)
    return out


# --------------------------------------------------------------------------- search

def family_cost(calls: Sequence[Tuple[int, int]], t: Callable[[int], float]) -> float:
    """T_f(a) = sum over the family's calls of n * t(M) (Eq. 3)."""
    return float(sum(n * t(M) for M, n in calls))


def exhaustive(grid: Sequence[bd.Pins], cost: Callable[[bd.Pins], float]):
    """Measures every candidate; returns (best, best_cost, measured)."""
    best, best_c = None, math.inf
    for p in grid:
        c = cost(p)
        if c < best_c:
            best, best_c = p, c
    return best, best_c, len(grid)


def search(grid: Sequence[bd.Pins], start: bd.Pins, cost: Callable[[bd.Pins], float], max_rounds: int = 4):
    """Coordinate descent over the grid's axes from `start` (which must be in
    the grid): one axis at a time, every legal value with the other axes held,
    keep the best; repeat until a round changes nothing.  Each tuple is
    measured at most once.  Returns (best, best_cost, measured)."""
    by_key = {key_of(p): p for p in grid}
    memo: Dict[tuple, float] = {}

    def c(k):
        if k not in memo:
            memo[k] = cost(by_key[k])
        return memo[k]

    cur = key_of(start)
    if cur not in by_key:
        raise ValueError("the start pins are not in the legal grid")
    values = [sorted({k[i] for k in by_key}) for i in range(5)]
    for _ in range(max_rounds):
        changed = False
        for axis in range(5):
            for v in values[axis]:
                k = cur[:axis] + (v,) + cur[axis + 1:]
                if k in by_key and c(k) < c(cur):
                    cur, changed = k, True
        if not changed:
            break
    return by_key[cur], memo[cur], len(memo)


def confirm(cost: Callable[[bd.Pins], float], default: bd.Pins, best: bd.Pins, rounds: int = 3,
            margin: float = 0.01):
    """Re-measures the default and the best tuple alternately; keeps the best
    only if its median cost is below the default's by `margin`.  Returns
    (chosen, median cost of the default, median cost of the best)."""
    import statistics
    if key_of(default) == key_of(best):
        c = statistics.median(cost(default) for _ in range(rounds))
        return default, c, c
    cd, cb = [], []
    for _ in range(rounds):
        cd.append(cost(default))
        cb.append(cost(best))
    md, mb = statistics.median(cd), statistics.median(cb)
    return (best if mb < md * (1.0 - margin) else default), md, mb


def delta_bound(delta: float) -> float:
    """Worst ratio of the per-family tuple's time to the best tuple's when
    additivity holds within relative error delta: (1 + delta) / (1 - delta)."""
    if not 0.0 <= delta < 1.0:
        raise ValueError("delta must be in [0, 1)")
    return (1.0 + delta) / (1.0 - delta)


def measured_delta(t_measured: float, c_other: float, family_costs: Iterable[float]) -> float:
    """Relative error of the additive model T^ = C + sum_f T_f against a
    measured workload time."""
    t_hat = c_other + sum(family_costs)
    return abs(t_measured - t_hat) / t_measured


# --------------------------------------------------------------------------- timing (GPU)

class GemmTimer:
    """t_f(M, pins) for one family on the current CUDA device."""

    def __init__(self, N: int, K: int, Ms: Sequence[int], reps: int = 10, seed: int = 0):
        import torch
        from . import inputs
        self.N, self.K = N, K
        wbytes = N * K * 2
        nw = max(2, math.ceil(2 * L2_BYTES / wbytes) + 1)
        self.W = [inputs.device_normal((N, K), std=0.02, seed=seed, stream=inputs.STREAM_W + 16 * i)
                  for i in range(min(nw, 8))]
        self.X = {}
        for M in Ms:
            nx = max(1, min(8, math.ceil(2 * L2_BYTES / max(M * K * 2, 1))))
            self.X[M] = [inputs.device_normal((M, K), seed=seed, stream=inputs.STREAM_X + 16 * i)
                         for i in range(nx)]
        self.Y = {M: torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for M in Ms}
        self.reps = reps
        self.ws = torch.zeros(256, dtype=torch.uint8, device="cuda")

    def _workspace(self, M: int, pins: bd.Pins):
        """A zeroed fold workspace large enough for this call (the counters
        stay zero between calls, so it is only replaced when too small)."""
        import torch
        need = bd.bi_gemm_bf16_workspace_bytes(M, self.N, self.K, pins)
        if need > self.ws.numel():
            self.ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        return self.ws

    def __call__(self, M: int, pins: bd.Pins) -> float:
        import torch
        xs, W, Y = self.X[M], self.W, self.Y[M]
        ws = self._workspace(M, pins)
        for i in range(3):
            bd.bi_gemm_bf16(xs[i % len(xs)], W[i % len(W)], out=Y, pins=pins, workspace=ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(self.reps):
                bd.bi_gemm_bf16(xs[i % len(xs)], W[i % len(W)], out=Y, pins=pins, workspace=ws)
        g.replay()
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        if bd.bi_last_device_status() != bd.BI_OK:
            raise bd.BiError(bd.bi_last_device_status(), "tuner timing")
        return s.elapsed_time(e) * 1e3 / self.reps   # us


def tune_family(N: int, K: int, calls: Sequence[Tuple[int, int]], mode: str = "search", reps: int = 10,
                base_flags: int = bd.BI_FLAG_SCHEDULE_AUTO, timer=None, repeats: int = 2) -> dict:
    """Tunes one family on the GPU; returns its JSON entry."""
    grid = legal_grid(N, K, base_flags)
    timer = timer or GemmTimer(N, K, [M for M, _ in calls], reps=reps)
    cost = lambda p: family_cost(calls, lambda M: min(timer(M, p) for _ in range(repeats)))
    d = bd.bi_pins_default(N, K)
    start = candidate(N, K, d.split_k, d.tok_tile, d.mma_ctas, d.stages, d.flags & bd.BI_FLAG_KTILE_PAIRS,
                      base_flags)
    if mode == "exhaustive":
        best, _, measured = exhaustive(grid, cost)
    else:
        best, _, measured = search(grid, start, cost)
    chosen, c_default, c_best = confirm(cost, start, best)
    return {"N": N, "K": K, "calls": [{"M": M, "n": n} for M, n in calls],
            "pins": chosen.as_dict(), "T_us": round(c_best if chosen is best else c_default, 2),
            "default_pins": start.as_dict(), "T_default_us": round(c_default, 2),
            "search_best_pins": best.as_dict(), "T_search_best_us": round(c_best, 2),
            "measured": measured, "legal": len(grid)}


# --------------------------------------------------------------------------- JSON

def dump(entries: Sequence[dict], path: str, **meta):
    doc = {"format": FORMAT, **meta, "families": list(entries)}
    with open(path, "w") as f:
        json.dump(doc, f, indent=1, sort_keys=False)
        f.write("\n")


def load(path: str) -> Dict[tuple, object]:
    """{(N, K): Pins, ("attention", Hq, Hkv, page_size): split_size} from a
    tuned table; every GEMM entry must pass bi_pins_validate for its shape and
    every split size must be legal (an illegal table is refused whole)."""
    with open(path) as f:
        doc = json.load(f)
    if doc.get("format") != FORMAT:
        raise ValueError("not a %s file: %r" % (FORMAT, doc.get("format")))
    table = {}
    for fam in doc["families"]:
        if "attention" in fam:
            att = fam["attention"]
            key = ("attention", int(att["Hq"]), int(att["Hkv"]), int(att["page_size"]))
            split = int(att["split_size"])
            if split % 64 or not 64 <= split <= bd.BI_ATTN_MAX_SPLIT:
                raise ValueError("split size %d for %r is illegal" % (split, key))
            if key in table:
                raise ValueError("two entries for %r" % (key,))
            table[key] = split
            continue
        N, K = int(fam["N"]), int(fam["K"])
        p = bd.Pins(**{k: int(v) for k, v in fam["pins"].items()})
        st = bd.bi_pins_validate(N, K, p)
        if st != bd.BI_OK:
            raise ValueError("pins for (N=%d, K=%d) are illegal: %s" % (N, K, bd.status_string(st)))
        if (N, K) in table:
            raise ValueError("two entries for (N=%d, K=%d)" % (N, K))
        table[(N, K)] = p
    return table


# --------------------------------------------------------------------------- decode attention

# Powers of two, and every multiple of 64 between 256 and 1024: a few long
# requests are shared out among the CTAs (request, split) item by item, so the
# split size that balances them need not be a power of two.
ATTN_SPLITS = (64, 128, 256, 320, 384, 448, 512, 576, 640, 704, 768, 832, 896, 960, 1024, 2048, 4096)


def attn_legal_splits(splits: Sequence[int] = ATTN_SPLITS) -> List[int]:
    """The legal split sizes among `splits`: multiples of 64 up to BI_ATTN_MAX_SPLIT."""
    return [S for S in splits if S % 64 == 0 and 64 <= S <= bd.BI_ATTN_MAX_SPLIT]


class AttnTimer:
    """t(split) of one recorded decode-attention workload on the current CUDA
    device: `calls` is a list of (request lengths, count); each call is timed
    as back-to-back decode steps over a paged cache (pages of `page_size`,
    shuffled) larger than L2."""

    def __init__(self, Hq: int, Hkv: int, page_size: int, calls, reps: int = 10, seed: int = 0):
        import torch
        from . import inputs
        self.calls = [(list(map(int, lens)), int(n)) for lens, n in calls]
        self.Hq, self.Hkv, self.P = Hq, Hkv, page_size
        self.data = []
        for i, (lens, _) in enumerate(self.calls):
            kc, vc, bt, sl = inputs.device_paged_kv(lens, Hkv, bd.BI_ATTN_HEAD_DIM, page_size, seed=seed + i)
            q = inputs.device_normal((len(lens), Hq, bd.BI_ATTN_HEAD_DIM), seed=seed + i, stream=0)
            out = torch.empty_like(q)
            self.data.append((q, kc, vc, bt, sl, out))
        self.reps = reps

    def call_time(self, i: int, split: int) -> float:
        import torch
        q, kc, vc, bt, sl, out = self.data[i]
        ml = bt.shape[1] * self.P
        ws = torch.empty(bd.bi_decode_attention_workspace_bytes(q.shape[0], self.Hq, self.Hkv, ml, split),
                         dtype=torch.uint8, device=q.device)
        run = lambda: bd.bi_decode_attention_bf16(q, kc, vc, bt, sl, bd.BI_ATTN_HEAD_DIM ** -0.5, max_seq_len=ml,
                                                  split_size=split, out=out, workspace=ws)
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(self.reps):
            run()
        e.record()
        torch.cuda.synchronize()
        if bd.bi_last_device_status() != bd.BI_OK:
            raise bd.BiError(bd.bi_last_device_status(), "tuner timing")
        return s.elapsed_time(e) * 1e3 / self.reps

    def __call__(self, split: int) -> float:
        return float(sum(n * self.call_time(i, split) for i, (_, n) in enumerate(self.calls)))


def tune_attention(Hq: int, Hkv: int, page_size: int, calls, splits: Sequence[int] = ATTN_SPLITS,
                   timer=None, repeats: int = 2, margin: float = 0.01) -> dict:
    """Picks the split size of one attention family: every legal size is
    measured (the best of `repeats`), then the winner must beat the library
    default by `margin` in interleaved re-measurements (else the default is
    kept).  Returns the table entry."""
    import statistics
    legal = attn_legal_splits(splits)
    if not legal:
        raise ValueError("no legal split size")
    timer = timer or AttnTimer(Hq, Hkv, page_size, calls)
    cost = {S: min(timer(S) for _ in range(repeats)) for S in legal}
    best = min(legal, key=lambda S: (cost[S], S))
    default = bd.BI_ATTN_DEFAULT_SPLIT
    chosen, t_default, t_best = default, None, None
    if best == default:
        t_default = t_best = cost[best]
    else:
        cd, cb = [], []
        for _ in range(3):
            cd.append(timer(default))
            cb.append(timer(best))
        t_default, t_best = statistics.median(cd), statistics.median(cb)
        if t_best < t_default * (1.0 - margin):
            chosen = best
    return {"attention": {"Hq": Hq, "Hkv": Hkv, "page_size": page_size,
                          "calls": [{"lengths": len(lens), "max": max(lens), "total": sum(lens), "n": n}
                                    for lens, n in [(list(c[0]), c[1]) for c in calls]],
                          "split_size": chosen, "T_us": round(t_best if chosen == best else t_default, 2),
                          "default_split": default, "T_default_us": round(t_default, 2),
                          "measured": {str(S): round(c, 2) for S, c in cost.items()}}}
