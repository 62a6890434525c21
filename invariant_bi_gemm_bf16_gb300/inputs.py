"""Seeded synthetic inputs for the batch-invariant linear layer.

This module only draws random numbers and stores them as bf16.  It holds none
of the layer's arithmetic, so both the CUDA path and the CPU oracle can be fed
from it without sharing any computation.

Recipes (the shapes and distributions of the Llama-3.1 projection workloads):
  - activations X ~ N(0, 1), weights W ~ N(0, 0.02), gains g ~ N(1, 0.1);
  - RMSNorm sweep rows: row m ~ N(0, s_m) with s_m = exp(U(ln 0.1, ln 10)),
    i.e. log-uniform on [0.1, 10] per row;
  - integer-valued tensors for the exactness cases.

Host draws use numpy's PCG64 generator seeded with ``[seed, stream]``; each
tensor of a problem gets its own stream id (X = 0, W = 1, g = 2, further
weights 3, 4, ...), so adding a tensor never shifts another tensor's values.
Values are drawn in float32 and rounded to bf16 by torch's round-to-nearest-even
conversion.  Device draws (for the multi-gigabyte benchmark tensors) use a
seeded ``torch.Generator`` on the GPU with the same distributions.
"""
from __future__ import annotations

import math

import numpy as np
import torch

STREAM_X = 0
STREAM_W = 1
STREAM_G = 2


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 numpy array -> CPU bf16 tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns (copied to host)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> CPU bf16 tensor."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)


def normal(shape, std: float = 1.0, mean: float = 0.0, seed: int = 0, stream: int = 0) -> torch.Tensor:
    """CPU bf16 tensor with entries ~ N(mean, std)."""
    r = _rng(seed, stream)
    a = r.standard_normal(size=tuple(shape), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return to_bf16(a)


def rows_loguniform(M: int, H: int, lo: float = 0.1, hi: float = 10.0, seed: int = 0,
                    stream: int = 0) -> torch.Tensor:
    """[M, H] bf16; row m ~ N(0, s_m), s_m log-uniform on [lo, hi]."""
    r = _rng(seed, stream)
    s = np.exp(r.uniform(math.log(lo), math.log(hi), size=(M, 1))).astype(np.float32)
    a = r.standard_normal(size=(M, H), dtype=np.float32) * s
    return to_bf16(a)


def integers(shape, lo: int, hi: int, seed: int = 0, stream: int = 0) -> torch.Tensor:
    """CPU bf16 tensor of integers uniform in [lo, hi] (exact in bf16 for |v| <= 256)."""
    r = _rng(seed, stream)
    a = r.integers(lo, hi + 1, size=tuple(shape)).astype(np.float32)
    return to_bf16(a)


def device_normal(shape, std: float = 1.0, mean: float = 0.0, seed: int = 0, stream: int = 0,
                  device="cuda") -> torch.Tensor:
    """bf16 tensor drawn on the device (for tensors too large to draw on the host)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + int(stream))
    out = torch.empty(tuple(shape), dtype=torch.bfloat16, device=device)
    # Draw in slices so that the float32 staging buffer stays small.
    flat = out.view(-1)
    step = 1 << 26
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        v = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        if mean != 0.0:
            v.add_(mean)
        flat[i:i + n].copy_(v)
    return out


def scatter_rows(target: torch.Tensor, batch: int, seed: int = 0, stream: int = 9,
                 corunner_std: float = 1.0, corunner_fill=None):
    """Embed the rows of ``target`` [m, K] at distinct random positions of a
    [batch, K] batch whose other rows are co-runners: N(0, corunner_std) draws,
    or a constant ``corunner_fill`` (e.g. +-65504, +-inf, nan).
    Returns (batch tensor, positions)."""
    m, K = target.shape
    if batch < m:
        raise ValueError("batch smaller than the target set")
    r = _rng(seed, stream)
    pos = np.sort(r.choice(batch, size=m, replace=False)).astype(np.int64)
    if corunner_fill is None:
        co = r.standard_normal(size=(batch, K), dtype=np.float32) * np.float32(corunner_std)
        full = to_bf16(co)
    else:
        full = torch.full((batch, K), float(corunner_fill), dtype=torch.bfloat16)
    full[torch.from_numpy(pos)] = target.to(torch.bfloat16).cpu()
    return full, pos


STREAM_KV = 20


def paged_kv(lens, Hkv: int, D: int, page_size: int, seed: int = 0, stream: int = STREAM_KV,
             spare_pages: int = 0, stale: float = float("nan"), std: float = 1.0):
    """Seeded keys and values for requests of the given lengths, in a paged
    cache whose pages are handed out in a shuffled order (host tensors):
    k_cache, v_cache [num_pages, page_size, Hkv, D] bf16; block_table [B, P]
    int32 (P = the most pages any request needs, unused entries -1); seq_lens
    [B] int32.  Cache rows past a request's length and the spare pages hold
    ``stale``.  Layout only: no arithmetic of the method."""
    lens = [int(x) for x in lens]
    need = [-(-L // page_size) for L in lens]
    total = sum(need) + int(spare_pages)
    r = _rng(seed, stream)
    order = r.permutation(max(total, 1))
    k = np.full((max(total, 1), page_size, Hkv, D), stale, dtype=np.float32)
    v = np.full((max(total, 1), page_size, Hkv, D), stale, dtype=np.float32)
    bt = np.full((len(lens), max(max(need, default=0), 1)), -1, dtype=np.int32)
    slot = 0
    for b, L in enumerate(lens):
        kd = r.standard_normal(size=(L, Hkv, D), dtype=np.float32) * np.float32(std)
        vd = r.standard_normal(size=(L, Hkv, D), dtype=np.float32) * np.float32(std)
        for i in range(need[b]):
            pg = int(order[slot])
            slot += 1
            lo, hi = i * page_size, min((i + 1) * page_size, L)
            k[pg, :hi - lo], v[pg, :hi - lo] = kd[lo:hi], vd[lo:hi]
            bt[b, i] = pg
    return to_bf16(k), to_bf16(v), torch.from_numpy(bt), torch.tensor(lens, dtype=torch.int32)


def device_paged_kv(lens, Hkv: int, D: int, page_size: int, seed: int = 0, stream: int = STREAM_KV,
                    device="cuda"):
    """The same layout drawn on the device, for caches too large for the host:
    every cache row is N(0, 1) (no stale marker), pages handed out in a seeded
    shuffled order.  Returns (k_cache, v_cache, block_table, seq_lens) on the
    device."""
    lens = [int(x) for x in lens]
    need = [-(-L // page_size) for L in lens]
    total = max(sum(need), 1)
    k = device_normal((total, page_size, Hkv, D), seed=seed, stream=stream, device=device)
    v = device_normal((total, page_size, Hkv, D), seed=seed, stream=stream + 1, device=device)
    order = _rng(seed, stream + 2).permutation(total)
    bt = np.full((len(lens), max(max(need, default=0), 1)), -1, dtype=np.int32)
    slot = 0
    for b in range(len(lens)):
        bt[b, :need[b]] = order[slot:slot + need[b]]
        slot += need[b]
    return (k, v, torch.from_numpy(bt).to(device),
            torch.tensor(lens, dtype=torch.int32, device=device))
