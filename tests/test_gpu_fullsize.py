"""Parity at the full workload sizes, in the launch configurations the
benchmark times, on sampled outputs the oracle computes one by one."""
import numpy as np
import pytest
import torch

from helpers import EPS, bf16_bits, bits_to_f64, check_ulp, ulp_bf16
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu

SHAPES = [
    # (N, K, Ms)
    (4096, 14336, [1, 64, 512, 8192]),    # Llama-3.1-8B down_proj (the benchmark sweep)
    (6144, 4096, [1, 8, 1024]),           # 8B qkv
    (28672, 4096, [1, 32, 4096]),         # 8B gate_up
    (10240, 8192, [32]),                  # 70B qkv
    (8192, 8192, [32]),                   # 70B o_proj
    (57344, 8192, [32]),                  # 70B gate_up
    (8192, 28672, [32]),                  # 70B down_proj
]


def sampled_parity(oracle, X, W, Y, n_samples, seed, what):
    M, K = X.shape
    N = W.shape[0]
    r = np.random.default_rng(seed)
    rows = r.integers(0, M, n_samples)
    cols = r.integers(0, N, n_samples)
    # always include the corners and the last row / column
    rows[:4] = [0, 0, M - 1, M - 1]
    cols[:4] = [0, N - 1, 0, N - 1]
    xs = inputs.bits(X[torch.from_numpy(np.unique(rows)).to(X.device)])
    remap = {m: i for i, m in enumerate(np.unique(rows))}
    want = oracle.gemm_sampled(xs, inputs.bits(W), np.array([remap[m] for m in rows]), cols)
    got = bits_to_f64(bf16_bits(Y[torch.from_numpy(rows).to(Y.device), torch.from_numpy(cols).to(Y.device)]))
    # rms(row) of the oracle's row: estimate from the GPU row (within tolerance of it)
    yrows = Y[torch.from_numpy(rows).to(Y.device)].float()
    rms = torch.sqrt(torch.mean(yrows * yrows, dim=1)).cpu().numpy().astype(np.float64)
    ref = want.astype(np.float64)
    tol = 2e-2 * np.sqrt(K / 4096.0) * rms + 0.5 * ulp_bf16(np.maximum(np.abs(ref), np.abs(got)))
    err = np.abs(got - ref)
    assert np.all(err <= tol), "%s: %d of %d samples over tolerance (worst %.3g x tol)" % (
        what, int((err > tol).sum()), n_samples, float((err / tol).max()))
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 5e-3, "%s: relative error %.3g" % (what, rel)


@pytest.mark.parametrize("N,K,Ms", SHAPES)
def test_fullsize_gemm_sampled_parity(lib, oracle, N, K, Ms):
    W = inputs.device_normal((N, K), std=0.02, seed=0, stream=inputs.STREAM_W)
    for M in Ms:
        X = inputs.device_normal((M, K), seed=0, stream=inputs.STREAM_X)
        Y = lib.bi_gemm_bf16(X, W)
        torch.cuda.synchronize()
        assert lib.bi_last_device_status() == lib.BI_OK
        sampled_parity(oracle, X, W, Y, 1500, seed=M, what="N=%d K=%d M=%d" % (N, K, M))


@pytest.mark.parametrize("N", [6144, 28672])
def test_fullsize_fused_sampled_parity(lib, oracle, N):
    K = 4096
    W = inputs.device_normal((N, K), std=0.02, seed=0, stream=inputs.STREAM_W)
    g = inputs.device_normal((K,), std=0.1, mean=1.0, seed=0, stream=inputs.STREAM_G)
    for M in (1, 32, 1024):
        X = inputs.device_normal((M, K), seed=0, stream=inputs.STREAM_X)
        Y = lib.bi_rmsnorm_gemm_bf16(X, g, W, EPS)
        xh = lib.bi_rmsnorm_bf16(X, g, EPS)
        torch.cuda.synchronize()
        # the normalisation within one ulp of the oracle, on a subset of rows
        sub = list(range(0, M, max(1, M // 16)))
        check_ulp(bf16_bits(xh[sub]), oracle.rmsnorm(inputs.bits(X[sub]), inputs.bits(g), EPS), 1, "norm")
        sampled_parity(oracle, xh, W, Y, 1500, seed=M, what="fused N=%d M=%d" % (N, M))
