"""Shared checks for the parity and invariance tests."""
from __future__ import annotations

import hashlib

import numpy as np
import torch

EPS = 1e-5


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    a = np.maximum(a, 2.0 ** -126)
    e = np.floor(np.log2(a))
    return 2.0 ** (e - 7)


def gemm_tolerance(y_ref_f32: np.ndarray, y_gpu: np.ndarray, K: int) -> np.ndarray:
    """Per-element bound: 2e-2 * sqrt(K/4096) * rms(row of the oracle's fp32
    output) plus half a bf16 ulp of the larger of the two values (the output
    rounding alone can reach half an ulp, which the first term does not cover
    for K < 4096 or for elements far above the row's RMS)."""
    ref = y_ref_f32.astype(np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    big = np.maximum(np.abs(ref), np.abs(y_gpu))
    return 2e-2 * np.sqrt(K / 4096.0) * rms + 0.5 * ulp_bf16(big)


def check_gemm_parity(y_gpu_bits: np.ndarray, y_ref_f32: np.ndarray, K: int, what: str = ""):
    """The GEMM bar: max |err| within the per-element tolerance and relative
    Frobenius error <= 5e-3 (errors taken against the oracle's fp32 result)."""
    g = bits_to_f64(y_gpu_bits)
    ref = y_ref_f32.astype(np.float64)
    assert np.all(np.isfinite(g)), what + ": non-finite output"
    err = np.abs(g - ref)
    tol = gemm_tolerance(y_ref_f32, g, K)
    bad = err > tol
    assert not bad.any(), "%s: %d elements over tolerance, worst excess %.3g at %s" % (
        what, int(bad.sum()), float((err - tol).max()), np.unravel_index(np.argmax(err - tol), err.shape))
    den = np.linalg.norm(ref)
    if den > 0:
        rel = np.linalg.norm(g - ref) / den
        assert rel <= 5e-3, "%s: relative Frobenius error %.3g" % (what, rel)


def ordered(bits16: np.ndarray) -> np.ndarray:
    b = bits16.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def check_ulp(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, max_ulp: int = 1, what: str = ""):
    """bf16 patterns within max_ulp steps (both NaN counts as equal, +-0 equal)."""
    a = y_gpu_bits.astype(np.uint16)
    b = y_ref_bits.astype(np.uint16)
    nan_a = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nan_b = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    assert np.array_equal(nan_a, nan_b), what + ": NaN positions differ"
    d = np.abs(ordered(a) - ordered(b))
    d[nan_a] = 0
    assert d.max(initial=0) <= max_ulp, "%s: %d elements more than %d ulp apart (max %d)" % (
        what, int((d > max_ulp).sum()), max_ulp, int(d.max()))


def row_hashes(t: torch.Tensor) -> list:
    """64-bit hash of each row's bytes."""
    b = bf16_bits(t)
    return [hashlib.blake2b(r.tobytes(), digest_size=8).hexdigest() for r in b]
