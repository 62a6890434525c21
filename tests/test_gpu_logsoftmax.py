"""GPU log-probabilities (bi_log_softmax_bf16, bi_token_logprobs_bf16) against
the fp64 oracle, special rows, and batch invariance (bit-exact rows across M,
positions and permutations).

Tolerance, from the arithmetic: each thread sums n = 8*ceil(V/32768) terms
exp(x - m) (m its own maximum), then three 5-level butterflies combine the
pairs; every step rounds once (2^-24); a term exp(d) = 2^(d log2 e) by
ex2.approx is off by about 2^-22 relative plus |d| 2^-24 from the rounded
product, and since d e^d <= 1/e that adds below n 2^-25 to the sum, so the sum's
relative error is below (n + 20) * 2^-23 and lse moves by at most that plus
the rounding of logf and of m + log(s); the final x - lse rounds once more:
    |gpu - ref| <= (n + 30) * 2^-23 + 2^-22 * (|lse| + |ref|)."""
import math

import numpy as np
import pytest
import torch

from helpers import bf16_bits
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


def tol(V, lse, ref):
    n = 8 * -(-V // 32768)
    return (n + 30) * 2.0 ** -23 + 2.0 ** -22 * (np.abs(lse)[:, None] + np.abs(ref))


def check(got, ref, x, what):
    """x: the logits as float64 [M,V] (to recover each row's lse = x - ref)."""
    got = got.astype(np.float64)
    finite = np.isfinite(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), what + ": NaN pattern"
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)]), what + ": infinities"
    V = ref.shape[1]
    lse = np.zeros(ref.shape[0])
    for r in range(ref.shape[0]):
        j = np.flatnonzero(finite[r])
        if j.size:
            lse[r] = x[r, j[0]] - ref[r, j[0]]
    err = np.zeros_like(ref)
    err[finite] = np.abs(got[finite] - ref[finite])
    t = tol(V, lse, np.where(finite, ref, 0.0))
    assert np.all(err <= t), "%s: worst error %.3g (tolerance %.3g)" % (what, err.max(), t.max())


def f64(X):
    return X.float().numpy().astype(np.float64)


@pytest.mark.parametrize("V", [8, 1000, 4104, 128256])
@pytest.mark.parametrize("M,std", [(1, 1.0), (3, 4.0), (37, 8.0), (100, 2.0), (130, 3.0)])
def test_log_softmax_parity(lib, oracle, V, M, std):
    X = inputs.normal((M, V), std=std, seed=20, stream=0)
    ref = oracle.log_softmax(inputs.bits(X))
    got = lib.bi_log_softmax_bf16(X.cuda()).cpu().numpy()
    check(got, ref, f64(X), "V=%d M=%d" % (V, M))


def test_special_rows(lib, oracle):
    V = 64
    rows = np.zeros((6, V), dtype=np.float32)
    rows[1, ::3] = -np.inf                  # -Inf entries
    rows[2, 5] = np.nan                     # undefined rows
    rows[3, 7] = np.inf
    rows[4, :] = -np.inf
    rows[5, :] = np.linspace(-40, 40, V)
    X = torch.from_numpy(rows).to(torch.bfloat16)
    ref = oracle.log_softmax(inputs.bits(X))
    got = lib.bi_log_softmax_bf16(X.cuda()).cpu().numpy()
    assert np.allclose(got[0], -math.log(V), rtol=0, atol=1e-6)
    assert np.all(np.isnan(got[2:5]))
    check(got, ref, f64(X), "special rows")


def test_rows_independent_of_batch_and_position(lib):
    V = 32000
    X = inputs.normal((300, V), std=4.0, seed=21, stream=0).cuda()
    full = lib.bi_log_softmax_bf16(X).cpu().numpy().view(np.uint32)
    for r in (0, 151, 299):
        alone = lib.bi_log_softmax_bf16(X[r:r + 1].contiguous()).cpu().numpy().view(np.uint32)
        assert np.array_equal(alone[0], full[r])
    perm = torch.randperm(300, generator=torch.Generator().manual_seed(6))
    shuffled = lib.bi_log_softmax_bf16(X[perm.cuda()].contiguous()).cpu().numpy().view(np.uint32)
    assert np.array_equal(shuffled, full[perm.numpy()])


@pytest.mark.parametrize("V", [8, 1000, 128256, 140008])
def test_cluster_and_cta_variants_give_the_same_bits(lib, V):
    """Rows of a batch of 130 run on a CTA pair per row; a row alone runs on
    an 8-CTA cluster.  Both follow the same tree: identical bits, including
    rows longer than the on-chip cache (V > 131072) and special rows."""
    X = inputs.normal((130, V), std=5.0, seed=24, stream=0)
    X[5, :] = float("-inf")
    X[6, V // 2] = float("nan")
    X[7, V - 1] = float("-inf")
    X = X.cuda()
    full = lib.bi_log_softmax_bf16(X).cpu().numpy().view(np.uint32)
    ids = torch.arange(130, dtype=torch.int32, device="cuda") % V
    tok = lib.bi_token_logprobs_bf16(X, ids).cpu().numpy().view(np.uint32)
    for r in (0, 5, 6, 7, 129):
        alone = lib.bi_log_softmax_bf16(X[r:r + 1].contiguous()).cpu().numpy().view(np.uint32)
        assert np.array_equal(alone[0], full[r]), r
        t1 = lib.bi_token_logprobs_bf16(X[r:r + 1].contiguous(), ids[r:r + 1]).cpu().numpy().view(np.uint32)
        assert t1[0] == tok[r], r


def test_token_logprobs_are_the_same_bits(lib, oracle):
    M, V = 40, 128256
    X = inputs.normal((M, V), std=3.0, seed=22, stream=0).cuda()
    ids = torch.from_numpy(inputs.integers((M,), 0, V - 1, seed=22, stream=1).float().numpy().astype(np.int32))
    ids[3] = -1
    ids[7] = V
    full = lib.bi_log_softmax_bf16(X).cpu().numpy()
    tok = lib.bi_token_logprobs_bf16(X, ids.cuda()).cpu().numpy()
    idn = ids.numpy()
    for r in range(M):
        if r in (3, 7):
            assert np.isnan(tok[r])
        else:
            assert tok[r].view(np.uint32) == full[r, idn[r]].view(np.uint32)
    ref = oracle.token_logprobs(inputs.bits(X.cpu()), np.where((idn >= 0) & (idn < V), idn, 0))
    ok = (idn >= 0) & (idn < V)
    assert np.all(np.abs(tok[ok] - ref[ok]) <= 64 * 2.0 ** -23 + 2.0 ** -21 * np.abs(ref[ok]) + 4e-5)


def test_lm_head_logprobs_batch_invariant(lib, oracle):
    """lm_head GEMM (Llama-3.1-8B shape: V = 128256, K = 4096) then token
    log-probabilities: a token's value is the same bits alone, in a batch of
    64 and at another position."""
    V, K = 128256, 4096
    W = inputs.device_normal((V, K), std=0.02, seed=23, stream=1)
    H = inputs.device_normal((64, K), seed=23, stream=0)
    ids = torch.arange(64, dtype=torch.int32, device="cuda") * 1999
    lp = lib.bi_token_logprobs_bf16(lib.bi_gemm_bf16(H, W), ids).cpu().numpy()
    for r in (0, 33, 63):
        alone = lib.bi_token_logprobs_bf16(lib.bi_gemm_bf16(H[r:r + 1].contiguous(), W), ids[r:r + 1]).cpu().numpy()
        assert alone[0].view(np.uint32) == lp[r].view(np.uint32)
    # and the log-softmax part against the oracle, on the GPU's own logits
    logits = lib.bi_gemm_bf16(H[:4].contiguous(), W)
    ref = oracle.token_logprobs(bf16_bits(logits), ids[:4].cpu().numpy())
    got = lib.bi_token_logprobs_bf16(logits, ids[:4]).cpu().numpy()
    assert np.all(np.abs(got - ref) <= 300 * 2.0 ** -23 + 2.0 ** -21 * np.abs(ref))


@pytest.mark.parametrize("V", [1000, 128256, 140008])
def test_token_logprobs_on_persistent_pairs(lib, V):
    """From 256 rows the token variant runs one CTA pair per SM, each pair
    taking every P-th row and staging its next row while it reduces this one.
    Each row's log-probability keeps its bits: equal to the full
    log-softmax's element (one pair per row) and to the row computed alone
    (an 8-CTA cluster), for rows longer than the on-chip cache and special
    rows; ids outside [0, V) give NaN."""
    M = 400
    X = inputs.normal((M, V), std=4.0, seed=25, stream=0)
    X[5, :] = float("-inf")
    X[160, V // 3] = float("nan")
    X[399, V - 1] = float("inf")
    X = X.cuda()
    ids = torch.from_numpy(np.random.default_rng(25).integers(0, V, size=M).astype(np.int32))
    ids[11] = -1
    ids[300] = V
    tok = lib.bi_token_logprobs_bf16(X, ids.cuda()).cpu().numpy().view(np.uint32)
    full = lib.bi_log_softmax_bf16(X).cpu().numpy().view(np.uint32)
    idn = ids.numpy()
    for r in range(M):
        if r in (11, 300):
            assert np.isnan(tok[r].view(np.float32)), r
        else:
            assert tok[r] == full[r, idn[r]], r
    for r in (0, 5, 151, 152, 160, 303, 304, 399):
        t1 = lib.bi_token_logprobs_bf16(X[r:r + 1].contiguous(), ids[r:r + 1].cuda()).cpu().numpy().view(np.uint32)
        assert t1[0] == tok[r], r
