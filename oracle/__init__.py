"""CPU oracle for the batch-invariant linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product (``invariant_bi_gemm_bf16_gb300``)
never imports it, and it imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, built with ``-ffp-contract=off``)
and is documented there, function by function, with the passages it follows.
This module only builds that file with gcc and marshals numpy arrays of bf16
bit patterns (``uint16``) in and out through ctypes.

Pins (checks against things other than the oracle itself) live in
``tests/test_oracle_pins.py``.  Parity status of each function:
  - ``gemm``, ``gemm_sampled``: pinned (integer-exact cases, the hand-worked
    summation-order example, Higham's bound against an fp64 brute force,
    identity / permutation / one-hot weights).
  - ``rmsnorm``, ``inv_rms``: pinned (zero rows, +-c rows with closed forms,
    fp64 brute force within one bf16 ulp, Higham's bound on the sum of squares).
  - ``rmsnorm_gemm``: pinned through its two pinned parts plus a composed
    closed-form case.
  - ``bf16_rne``: pinned against hand-derived bit patterns (ties, NaN, overflow).
  - ``silu_mul``, ``residual_add``, ``attention_ctx1``, ``decode_layer``:
    pinned by closed forms (silu(0)=0, large-|x| limits, zero weights give the
    identity layer, selector weights route v exactly, and selector gate/up and
    down weights with a gain for the second RMSNorm that differs from the
    first reproduce a numpy closed form of the MLP half).
  - ``log_softmax``, ``token_logprobs``: pinned by closed forms (uniform rows
    give -log V, two-logit rows the stable softplus form), normalisation
    (sum of exp = 1), shift invariance, -Inf entries and undefined rows.
  - ``e4m3_encode``/``e4m3_decode``, ``quantize_rows_e4m3``, ``gemm_e4m3``:
    pinned by hand-derived codes (1.0, 448, subnormals, ties, saturation,
    NaN), the decode/encode round trip over all codes, exact scales for
    power-of-two rows, integer-exact GEMMs, and non-power-of-two scales for
    which each other order of applying sx and sw changes the bf16 result.
  - ``decode_attention``: pinned by closed forms (one position gives its
    value row; equal keys or scale 0 give the mean of the values; two
    positions give the logistic form; a dominant key selects its value),
    the grouped-query head mapping, position-order and page-placement
    invariance, convexity, and cache rows past the length being ignored.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no fused multiply-add)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        # -fno-tree-vrp -fno-thread-jumps: gcc 13 at -O2 threaded a branch on
        # a float range and folded amax / 448 to 0 for a subnormal amax (the
        # quotient is a nonzero subnormal); the oracle gives up those passes.
        cmd = ["gcc", "-O2", "-fno-tree-vrp", "-fno-thread-jumps", "-std=c11", "-ffp-contract=off",
               "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_rmsnorm.argtypes = [_u16p, _u16p, _u16p, _i64, _i64, ctypes.c_float, ctypes.c_int]
            lib.oracle_rmsnorm_inv_rms.restype = ctypes.c_float
            lib.oracle_rmsnorm_inv_rms.argtypes = [_u16p, _i64, ctypes.c_float]
            lib.oracle_gemm.argtypes = [_u16p, _u16p, _f32p, _u16p, _i64, _i64, _i64, ctypes.c_int]
            lib.oracle_gemm_sampled.argtypes = [_u16p, _u16p, _i64p, _i64p, _f32p, _i64, _i64, ctypes.c_int]
            lib.oracle_rmsnorm_gemm.argtypes = [_u16p, _u16p, _u16p, _f32p, _u16p, _u16p, _i64, _i64,
                                                _i64, ctypes.c_float, ctypes.c_int]
            lib.oracle_residual_add.argtypes = [_u16p, _u16p, _u16p, _i64]
            lib.oracle_silu_mul.argtypes = [_u16p, _u16p, _i64, _i64]
            lib.oracle_attention_ctx1.argtypes = [_u16p, _u16p, _i64, _i64, _i64, _i64]
            lib.oracle_decode_layer.restype = ctypes.c_int
            lib.oracle_decode_layer.argtypes = [_u16p, _u16p, _u16p, _u16p, _u16p, _u16p, _u16p, _u16p,
                                                _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_float,
                                                ctypes.c_int]
            lib.oracle_log_softmax.argtypes = [_u16p, _f64p, _i64, _i64, ctypes.c_int]
            lib.oracle_token_logprobs.argtypes = [_u16p, _i32p, _f64p, _i64, _i64, ctypes.c_int]
            lib.oracle_e4m3_to_f32.restype = ctypes.c_float
            lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_rne_sat.restype = ctypes.c_uint8
            lib.oracle_e4m3_rne_sat.argtypes = [ctypes.c_float]
            lib.oracle_quantize_rows_e4m3.argtypes = [_u16p, _u8p, _f32p, _i64, _i64, ctypes.c_int]
            lib.oracle_gemm_e4m3.argtypes = [_u8p, _f32p, _u8p, _f32p, _f32p, _u16p, _i64, _i64, _i64,
                                             ctypes.c_int]
            lib.oracle_decode_attention.argtypes = [_u16p, _u16p, _u16p, _i32p, _i64, _i32p, _i64p, _i64,
                                                    _f64p, _i64, _i64, _i64, _i64, _i64, ctypes.c_double,
                                                    ctypes.c_int]
            lib.oracle_bf16_rne_array.argtypes = [_f32p, _u16p, _i64]
            lib.oracle_bf16_to_f32_array.argtypes = [_u16p, _f32p, _i64]
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("expected bf16 bit patterns as uint16, got %s" % a.dtype)
    return a


def _p16(a: np.ndarray):
    return a.ctypes.data_as(_u16p)


def _pf(a: np.ndarray):
    return a.ctypes.data_as(_f32p)


# --------------------------------------------------------------------------
# conversions
# --------------------------------------------------------------------------

def bf16_rne(values) -> np.ndarray:
    """fp32 values -> bf16 bit patterns, round to nearest even."""
    f = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    out = np.empty(f.shape, dtype=np.uint16)
    _load().oracle_bf16_rne_array(_pf(f), _p16(out), f.size)
    return out


def bf16_to_f32(bits) -> np.ndarray:
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float32)
    _load().oracle_bf16_to_f32_array(_p16(b), _pf(out), b.size)
    return out


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------

def rmsnorm(X, g, eps: float, nthreads: int | None = None) -> np.ndarray:
    """X [M,H] bf16 bits, g [H] bf16 bits -> Y [M,H] bf16 bits."""
    X = _u16(X)
    g = _u16(g)
    M, H = X.shape
    if g.shape != (H,):
        raise ValueError("gain must have shape (H,)")
    Y = np.empty_like(X)
    _load().oracle_rmsnorm(_p16(X), _p16(g), _p16(Y), M, H, float(eps), nthreads or default_threads())
    return Y


def inv_rms(x_row, eps: float) -> np.float32:
    x = _u16(x_row).reshape(-1)
    return np.float32(_load().oracle_rmsnorm_inv_rms(_p16(x), x.size, float(eps)))


def gemm(X, W, nthreads: int | None = None):
    """X [M,K], W [N,K] bf16 bits -> (Y fp32 [M,N], Y bf16 bits [M,N])."""
    X = _u16(X)
    W = _u16(W)
    M, K = X.shape
    N, K2 = W.shape
    if K != K2:
        raise ValueError("K mismatch")
    Yf = np.empty((M, N), dtype=np.float32)
    Yb = np.empty((M, N), dtype=np.uint16)
    _load().oracle_gemm(_p16(X), _p16(W), _pf(Yf), _p16(Yb), M, N, K, nthreads or default_threads())
    return Yf, Yb


def gemm_sampled(X, W, rows, cols, nthreads: int | None = None) -> np.ndarray:
    """fp32 Y[rows[i], cols[i]] for each i, without computing the rest."""
    X = _u16(X)
    W = _u16(W)
    K = X.shape[1]
    if W.shape[1] != K:
        raise ValueError("K mismatch")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows/cols shape mismatch")
    if rows.size and (rows.min() < 0 or rows.max() >= X.shape[0] or cols.min() < 0 or cols.max() >= W.shape[0]):
        raise IndexError("sample index out of range")
    out = np.empty(rows.shape, dtype=np.float32)
    _load().oracle_gemm_sampled(_p16(X), _p16(W), rows.ctypes.data_as(_i64p), cols.ctypes.data_as(_i64p),
                                _pf(out), rows.size, K, nthreads or default_threads())
    return out


def rmsnorm_gemm(X, g, W, eps: float, nthreads: int | None = None):
    """Fused layer -> (Y fp32, Y bf16 bits, Xhat bf16 bits)."""
    X = _u16(X)
    g = _u16(g)
    W = _u16(W)
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K or g.shape != (K,):
        raise ValueError("shape mismatch")
    Yf = np.empty((M, N), dtype=np.float32)
    Yb = np.empty((M, N), dtype=np.uint16)
    Xh = np.empty((M, K), dtype=np.uint16)
    _load().oracle_rmsnorm_gemm(_p16(X), _p16(g), _p16(W), _pf(Yf), _p16(Yb), _p16(Xh), M, N, K,
                                float(eps), nthreads or default_threads())
    return Yf, Yb, Xh


def residual_add(a, b) -> np.ndarray:
    a = _u16(a)
    b = _u16(b)
    if a.shape != b.shape:
        raise ValueError("shape mismatch")
    out = np.empty_like(a)
    _load().oracle_residual_add(_p16(a), _p16(b), _p16(out), a.size)
    return out


def silu_mul(gu) -> np.ndarray:
    """[M, 2I] gate|up bits -> [M, I] bits."""
    gu = _u16(gu)
    M, I2 = gu.shape
    if I2 % 2:
        raise ValueError("gate/up width must be even")
    out = np.empty((M, I2 // 2), dtype=np.uint16)
    _load().oracle_silu_mul(_p16(gu), _p16(out), M, I2 // 2)
    return out


def attention_ctx1(qkv, nq: int, nkv: int, D: int) -> np.ndarray:
    qkv = _u16(qkv)
    M, width = qkv.shape
    if width != (nq + 2 * nkv) * D or nq % nkv:
        raise ValueError("bad head layout")
    out = np.empty((M, nq * D), dtype=np.uint16)
    _load().oracle_attention_ctx1(_p16(qkv), _p16(out), M, nq, nkv, D)
    return out


def decode_layer(x, layer: dict, nq: int, nkv: int, D: int, eps: float,
                 nthreads: int | None = None) -> np.ndarray:
    """One decode layer (see oracle.c); ``layer`` holds bf16 bit arrays
    g_attn, Wqkv, Wo, g_mlp, Wgu, Wd."""
    x = _u16(x)
    M, Hd = x.shape
    Wqkv, Wo, Wgu, Wd = (_u16(layer[k]) for k in ("Wqkv", "Wo", "Wgu", "Wd"))
    g1, g2 = _u16(layer["g_attn"]), _u16(layer["g_mlp"])
    I = Wd.shape[1]
    if Wqkv.shape != ((nq + 2 * nkv) * D, Hd) or Wo.shape != (Hd, nq * D) or \
            Wgu.shape != (2 * I, Hd) or Wd.shape != (Hd, I) or g1.shape != (Hd,) or g2.shape != (Hd,):
        raise ValueError("bad layer shapes")
    out = np.empty_like(x)
    rc = _load().oracle_decode_layer(_p16(x), _p16(out), _p16(g1), _p16(Wqkv), _p16(Wo), _p16(g2),
                                     _p16(Wgu), _p16(Wd), M, Hd, nq, nkv, D, I, float(eps),
                                     nthreads or default_threads())
    if rc != 0:
        raise MemoryError("oracle_decode_layer: allocation failed")
    return out


def stack(x, layers, nq: int, nkv: int, D: int, eps: float, nthreads: int | None = None) -> np.ndarray:
    """The decode-step linear stack: the layers applied in order."""
    for layer in layers:
        x = decode_layer(x, layer, nq, nkv, D, eps, nthreads)
    return x


# --------------------------------------------------------------------------
# lm_head log-probabilities
# --------------------------------------------------------------------------

def log_softmax(X, nthreads: int | None = None) -> np.ndarray:
    """X [M,V] bf16 bits -> [M,V] float64 log-probabilities."""
    x = _u16(X)
    M, V = x.shape
    out = np.empty((M, V), dtype=np.float64)
    _load().oracle_log_softmax(_p16(x), out.ctypes.data_as(_f64p), M, V, nthreads or default_threads())
    return out


def token_logprobs(X, ids, nthreads: int | None = None) -> np.ndarray:
    """X [M,V] bf16 bits, ids [M] int -> [M] float64 log-probabilities of the ids."""
    x = _u16(X)
    M, V = x.shape
    i = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    if i.shape != (M,):
        raise ValueError("ids must have shape [M]")
    out = np.empty(M, dtype=np.float64)
    _load().oracle_token_logprobs(_p16(x), i.ctypes.data_as(_i32p), out.ctypes.data_as(_f64p), M, V,
                                  nthreads or default_threads())
    return out


# --------------------------------------------------------------------------
# FP8 (E4M3) with per-row scales
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    lib = _load()
    return np.array([lib.oracle_e4m3_to_f32(int(v)) for v in c.ravel()], dtype=np.float32).reshape(c.shape)


def e4m3_encode(values) -> np.ndarray:
    f = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    lib = _load()
    return np.array([lib.oracle_e4m3_rne_sat(float(v)) for v in f.ravel()], dtype=np.uint8).reshape(f.shape)


def quantize_rows_e4m3(X, nthreads: int | None = None):
    """X [M,K] bf16 bits -> (codes [M,K] uint8, scales [M] float32)."""
    x = _u16(X)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.uint8)
    sc = np.empty(M, dtype=np.float32)
    _load().oracle_quantize_rows_e4m3(_p16(x), q.ctypes.data_as(_u8p), _pf(sc), M, K,
                                      nthreads or default_threads())
    return q, sc


def gemm_e4m3(Xq, sx, Wq, sw, nthreads: int | None = None):
    """(fp32 unscaled sums [M,N], bf16 bits of the scaled result [M,N])."""
    xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    sxa = np.ascontiguousarray(sx, dtype=np.float32)
    swa = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = xq.shape
    N = wq.shape[0]
    yf = np.empty((M, N), dtype=np.float32)
    yb = np.empty((M, N), dtype=np.uint16)
    _load().oracle_gemm_e4m3(xq.ctypes.data_as(_u8p), _pf(sxa), wq.ctypes.data_as(_u8p), _pf(swa), _pf(yf),
                             _p16(yb), M, N, K, nthreads or default_threads())
    return yf, yb


# --------------------------------------------------------------------------
# Decode attention over a paged key/value cache
# --------------------------------------------------------------------------

def decode_attention(q, k_cache, v_cache, block_table, seq_lens, scale: float, pairs=None,
                     nthreads: int | None = None) -> np.ndarray:
    """q [B,Hq,D] bf16 bits; k_cache, v_cache [num_pages, page_size, Hkv, D]
    bf16 bits; block_table [B, P] int32; seq_lens [B] int32.  Returns fp64
    [B,Hq,D], or [n,D] for the (b, h) rows listed in ``pairs`` ([n,2])."""
    qa, ka, va = _u16(q), _u16(k_cache), _u16(v_cache)
    B, Hq, D = qa.shape
    _, page_size, Hkv, Dk = ka.shape
    if va.shape != ka.shape or Dk != D or Hq % Hkv:
        raise ValueError("shape mismatch")
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    if bt.ndim != 2 or bt.shape[0] != B or sl.shape != (B,):
        raise ValueError("block_table must be [B, P] and seq_lens [B]")
    if np.any(sl > bt.shape[1] * page_size) or np.any(sl < 0):
        raise ValueError("a length exceeds the pages of its block-table row")
    for b in range(B):
        used = bt[b, :(int(sl[b]) + page_size - 1) // page_size]
        if np.any(used < 0) or np.any(used >= ka.shape[0]):
            raise ValueError("request %d uses a page id outside the cache" % b)
    lib = _load()
    nt = nthreads or default_threads()
    if pairs is None:
        out = np.empty((B, Hq, D), dtype=np.float64)
        lib.oracle_decode_attention(_p16(qa), _p16(ka), _p16(va), bt.ctypes.data_as(_i32p), bt.shape[1],
                                    sl.ctypes.data_as(_i32p), None, 0, out.ctypes.data_as(_f64p), B, Hq,
                                    Hkv, D, page_size, float(scale), nt)
        return out
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    out = np.empty((pr.shape[0], D), dtype=np.float64)
    lib.oracle_decode_attention(_p16(qa), _p16(ka), _p16(va), bt.ctypes.data_as(_i32p), bt.shape[1],
                                sl.ctypes.data_as(_i32p), pr.ctypes.data_as(_i64p), pr.shape[0],
                                out.ctypes.data_as(_f64p), B, Hq, Hkv, D, page_size, float(scale), nt)
    return out
