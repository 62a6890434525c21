"""GPU parity of bi_rmsnorm_bf16 (within one bf16 ulp of the oracle) and of the
fused bi_rmsnorm_gemm_bf16 (bit-equal to the two calls in sequence)."""
import numpy as np
import pytest
import torch

from helpers import EPS, bf16_bits, check_gemm_parity, check_ulp
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H", [256, 2048, 4096, 8192, 16384, 8, 72, 1000, 2048 + 8])
@pytest.mark.parametrize("M", [1, 3, 37, 257, 1500])
def test_rmsnorm_parity(lib, oracle, M, H):
    """1500 rows exceed the warps of one grid at H >= 2048, so each warp's ring
    of row buffers wraps around."""
    X = inputs.rows_loguniform(M, H, seed=0, stream=0)
    g = inputs.normal((H,), std=0.1, mean=1.0, seed=0, stream=2)
    want = oracle.rmsnorm(inputs.bits(X), inputs.bits(g), EPS)
    got = bf16_bits(lib.bi_rmsnorm_bf16(X.cuda(), g.cuda(), EPS))
    check_ulp(got, want, 1, "rmsnorm M=%d H=%d" % (M, H))


def test_rmsnorm_special_rows(lib):
    H = 256
    g1 = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((2, H), dtype=torch.bfloat16, device="cuda")
    assert torch.all(lib.bi_rmsnorm_bf16(x, g1).float() == 0)
    sign = torch.where(torch.rand(3, H) < 0.5, -1.0, 1.0).to(torch.bfloat16).cuda()
    assert torch.equal(lib.bi_rmsnorm_bf16(sign, g1), sign)   # +-1 rows are fixed points
    nanrow = torch.full((1, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert torch.isnan(lib.bi_rmsnorm_bf16(nanrow, g1).float()).all()


@pytest.mark.parametrize("M,H", [(9, 4096), (2000, 8192), (700, 16384)])
def test_rmsnorm_in_place(lib, oracle, M, H):
    X = inputs.rows_loguniform(M, H, seed=1, stream=0)
    g = inputs.normal((H,), std=0.1, mean=1.0, seed=1, stream=2)
    want = oracle.rmsnorm(inputs.bits(X), inputs.bits(g), EPS)
    x = X.cuda()
    lib.bi_rmsnorm_bf16(x, g.cuda(), EPS, out=x)
    check_ulp(bf16_bits(x), want, 1, "in place")


@pytest.mark.parametrize("H,M", [(2048, 3000), (4096, 5000), (8192, 3000)])
def test_rmsnorm_rows_independent_of_batch(lib, H, M):
    """A row's bits are the same alone, in a batch of M and at another position.
    The batch and the single row run different kernels at H = 4096 and 8192
    (the row in shared memory against registers)."""
    X = inputs.rows_loguniform(M, H, seed=3, stream=0).cuda()
    g = inputs.normal((H,), std=0.1, mean=1.0, seed=3, stream=2).cuda()
    full = bf16_bits(lib.bi_rmsnorm_bf16(X, g, EPS))
    for r in (0, 1234, M - 1):
        alone = bf16_bits(lib.bi_rmsnorm_bf16(X[r:r + 1].contiguous(), g, EPS))
        assert np.array_equal(alone[0], full[r])
    for m in (37, 1215, 1216, 4095):  # the block-size and kernel switches
        assert np.array_equal(bf16_bits(lib.bi_rmsnorm_bf16(X[:m].contiguous(), g, EPS)), full[:m]), m
    perm = torch.randperm(M, generator=torch.Generator().manual_seed(5))
    shuffled = bf16_bits(lib.bi_rmsnorm_bf16(X[perm.cuda()].contiguous(), g, EPS))
    assert np.array_equal(shuffled, full[perm.numpy()])


@pytest.mark.parametrize("M,H", [(4100, 4096), (1300, 8192)])
def test_rmsnorm_parity_large_batches(lib, oracle, M, H):
    """The kernel of large batches (the row in shared memory) against the
    oracle."""
    X = inputs.rows_loguniform(M, H, seed=4, stream=0)
    g = inputs.normal((H,), std=0.1, mean=1.0, seed=4, stream=2)
    want = oracle.rmsnorm(inputs.bits(X), inputs.bits(g), EPS)
    check_ulp(bf16_bits(lib.bi_rmsnorm_bf16(X.cuda(), g.cuda(), EPS)), want, 1, "rmsnorm M=%d H=%d" % (M, H))


@pytest.mark.parametrize("M,N,K", [(1, 384, 4096), (33, 256, 512), (130, 640, 256)])
def test_fused_equals_composition_and_oracle(lib, oracle, M, N, K):
    X = inputs.normal((M, K), seed=2, stream=0)
    g = inputs.normal((K,), std=0.1, mean=1.0, seed=2, stream=2)
    W = inputs.normal((N, K), std=0.02, seed=2, stream=1)
    x, gg, w = X.cuda(), g.cuda(), W.cuda()
    fused = lib.bi_rmsnorm_gemm_bf16(x, gg, w, EPS)
    xh = lib.bi_rmsnorm_bf16(x, gg, EPS)
    comp = lib.bi_gemm_bf16(xh, w)
    torch.cuda.synchronize()
    assert torch.equal(fused, comp)
    # the GEMM part against the oracle, fed the GPU's own normalised rows
    yf, _ = oracle.gemm(bf16_bits(xh), inputs.bits(W))
    check_gemm_parity(bf16_bits(fused), yf, K, "fused")
    # and the normalisation against the oracle's
    check_ulp(bf16_bits(xh), oracle.rmsnorm(inputs.bits(X), inputs.bits(g), EPS), 1, "fused norm")
