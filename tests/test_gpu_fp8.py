"""FP8 (E4M3) path on the GPU: per-row quantisation bit-exact against the
oracle, the scaled FP8 GEMM within the GEMM bar (bit-exact on integer codes),
and batch invariance -- including across schedules and CTA groupings, which
the open grouping relies on for kind::f8f6f4 MMAs as for bf16 (H1)."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_parity
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


def u8(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 16), (37, 4096), (300, 14336), (5, 1040), (3, 28672), (4, 33024)])
def test_quantize_bit_exact(lib, oracle, M, K):
    X = inputs.rows_loguniform(M, K, lo=1e-3, hi=1e3, seed=40, stream=0)
    want_q, want_s = oracle.quantize_rows_e4m3(inputs.bits(X))
    q, s = lib.bi_quantize_rows_e4m3(X.cuda())
    assert np.array_equal(u8(q), want_q)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), want_s.view(np.uint32))


def test_quantize_special_rows(lib, oracle):
    K = 64
    rows = np.ones((6, K), dtype=np.float32)
    rows[5] = np.linspace(-1e-38, 1e-38, K)      # amax below 448 / FLT_MAX: inv is clamped
    rows[0] = 0.0
    rows[1, 3] = np.nan
    rows[2, 7] = -np.inf
    rows[3] = -0.0
    rows[4] = np.linspace(-1e-30, 1e-30, K)      # bf16 subnormal-range values
    X = torch.from_numpy(rows).to(torch.bfloat16)
    want_q, want_s = oracle.quantize_rows_e4m3(inputs.bits(X))
    q, s = lib.bi_quantize_rows_e4m3(X.cuda())
    assert np.array_equal(u8(q), want_q)
    got_s = s.cpu().numpy()
    assert np.array_equal(np.isnan(got_s), np.isnan(want_s))
    assert np.array_equal(got_s[~np.isnan(got_s)], want_s[~np.isnan(want_s)])


def quantized(lib, M, N, K, seed):
    X = inputs.normal((M, K), seed=seed, stream=0).cuda()
    W = inputs.normal((N, K), std=0.02, seed=seed, stream=1).cuda()
    xq, sx = lib.bi_quantize_rows_e4m3(X)
    wq, sw = lib.bi_quantize_rows_e4m3(W)
    return xq, sx, wq, sw


SHAPES = [(200, 300, 1024), (1, 640, 4096), (129, 256, 1040), (300, 512, 14336)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_fp8_parity(lib, oracle, M, N, K):
    xq, sx, wq, sw = quantized(lib, M, N, K, seed=41)
    yf, _ = oracle.gemm_e4m3(u8(xq), sx.cpu().numpy(), u8(wq), sw.cpu().numpy())
    ref = (yf.astype(np.float64) * sx.cpu().numpy()[:, None] * sw.cpu().numpy()[None, :]).astype(np.float32)
    got = bf16_bits(lib.bi_gemm_fp8(xq, sx, wq, sw))
    check_gemm_parity(got, ref, K, "fp8 M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("S", [1, 2, 3, 4])
def test_gemm_fp8_integer_codes_bit_exact_in_every_schedule(lib, oracle, S):
    """Codes of small integers: every product and partial sum is an exact
    integer, so any tree gives the oracle's bits."""
    M, N, K = 150, 384, 2048
    rng = np.random.default_rng(42)
    vx = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    vw = rng.integers(-4, 5, size=(N, K)).astype(np.float32)
    qx, qw = oracle.e4m3_encode(vx), oracle.e4m3_encode(vw)
    sx = (2.0 ** rng.integers(-3, 4, size=M)).astype(np.float32)
    sw = (2.0 ** rng.integers(-3, 4, size=N)).astype(np.float32)
    _, yb = oracle.gemm_e4m3(qx, sx, qw, sw)
    d = [torch.from_numpy(a).cuda() for a in (qx, sx, qw, sw)]
    base = lib.bi_pins_default_fp8(N, K).replace(split_k=S)
    for flags in (lib.BI_FLAG_SCHEDULE_LOCAL, lib.BI_FLAG_SCHEDULE_CLUSTER, lib.BI_FLAG_SCHEDULE_AUTO):
        for ctas in (1, 2):
            p = base.replace(flags=flags | lib.BI_FLAG_KTILE_PAIRS, mma_ctas=ctas)
            assert np.array_equal(bf16_bits(lib.bi_gemm_fp8(*d, pins=p)), yb), (flags, ctas)


def test_gemm_fp8_schedules_groupings_and_copies_agree(lib):
    M, N, K = 700, 4096, 14336
    xq, sx, wq, sw = quantized(lib, M, N, K, seed=43)
    base = lib.bi_pins_default_fp8(N, K)
    ref = None
    for flags in (lib.BI_FLAG_SCHEDULE_LOCAL, lib.BI_FLAG_SCHEDULE_CLUSTER, lib.BI_FLAG_SCHEDULE_CHAIN,
                  lib.BI_FLAG_SCHEDULE_AUTO):
        for ctas in (0, 1, 2):
            for kp in (0, lib.BI_FLAG_KTILE_PAIRS):
                p = base.replace(flags=flags | kp, mma_ctas=ctas)
                got = bf16_bits(lib.bi_gemm_fp8(xq, sx, wq, sw, pins=p))
                if ref is None:
                    ref = got
                assert np.array_equal(got, ref), (flags, ctas, kp)


def test_fp8_rows_independent_of_batch(lib):
    """Quantisation and GEMM together: a token's output bits are the same alone,
    in a batch of 1000 and at another position."""
    N, K = 4096, 14336
    X = inputs.device_normal((1000, K), seed=44, stream=0)
    W = inputs.device_normal((N, K), std=0.02, seed=44, stream=1)
    wq, sw = lib.bi_quantize_rows_e4m3(W)

    def layer(x):
        xq, sx = lib.bi_quantize_rows_e4m3(x)
        return bf16_bits(lib.bi_gemm_fp8(xq, sx, wq, sw))
    full = layer(X)
    for r in (0, 517, 999):
        assert np.array_equal(layer(X[r:r + 1].contiguous())[0], full[r])
    # batches on either side of the decode tiles (64 and 128 tokens)
    for m in (8, 64, 65, 128, 129):
        assert np.array_equal(layer(X[:m].contiguous()), full[:m]), m
    perm = torch.randperm(1000, generator=torch.Generator().manual_seed(8))
    assert np.array_equal(layer(X[perm.cuda()].contiguous()), full[perm.numpy()])


@pytest.mark.parametrize("M,H", [(1, 4096), (37, 8192), (300, 4096), (5, 16384), (3, 1040), (2000, 2048),
                                 (1023, 4096), (1024, 4096), (4100, 4096), (8192, 4096), (5001, 2048)])
def test_rmsnorm_quantize_is_the_composition(lib, oracle, M, H):
    """One pass gives the codes and scales of bi_quantize_rows_e4m3 applied to
    bi_rmsnorm_bf16's output, bit for bit, and those are the oracle's
    quantisation of that output; zero and NaN rows included."""
    X = inputs.rows_loguniform(M, H, lo=1e-3, hi=1e3, seed=45, stream=0)
    if M >= 3:
        X[1] = 0
        X[2, H // 3] = float("nan")
    if M >= 5:
        X[3, 7] = -float("inf")   # an infinity flags its row like a NaN
        X[4] = -0.0               # signed zeros: the row's maximum is 0
    g = inputs.normal((H,), std=0.1, mean=1.0, seed=45, stream=2)
    x, gg = X.cuda(), g.cuda()
    q, sc = lib.bi_rmsnorm_quantize_e4m3(x, gg, 1e-5)
    y = lib.bi_rmsnorm_bf16(x, gg, 1e-5)
    q2, sc2 = lib.bi_quantize_rows_e4m3(y)
    assert np.array_equal(u8(q), u8(q2))
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), sc2.cpu().numpy().view(np.uint32))
    want_q, want_s = oracle.quantize_rows_e4m3(bf16_bits(y))
    assert np.array_equal(u8(q), want_q)
    got_s, want_s = sc.cpu().numpy(), np.asarray(want_s, dtype=np.float32)
    assert np.array_equal(np.isnan(got_s), np.isnan(want_s))
    ok = ~np.isnan(want_s)
    assert np.array_equal(got_s[ok].view(np.uint32), want_s[ok].view(np.uint32))


@pytest.mark.parametrize("H", [2048, 4096])
def test_rmsnorm_quantize_bits_across_the_kernel_switch(lib, H):
    """Below 1024 rows a warp holds its row in registers; from 1024 rows the
    rows stream through per-warp rings in shared memory (a persistent grid,
    each warp taking every G-th row).  A row's codes and scale are the same
    bits either way, and whatever batch the row is in: every row of a
    4096 + 1900 row batch equals the same row computed in batches of 1000
    (registers), 1 (registers), 3099 and 3000 (the ring)."""
    M = 4096 + 1900
    X = inputs.rows_loguniform(M, H, lo=1e-2, hi=1e2, seed=46, stream=0)
    X[5] = 0
    X[4097, 11] = float("nan")
    g = inputs.normal((H,), std=0.1, mean=1.0, seed=46, stream=2)
    x, gg = X.cuda(), g.cuda()
    q, sc = lib.bi_rmsnorm_quantize_e4m3(x, gg, 1e-5)
    q, sc = u8(q), sc.cpu().numpy().view(np.uint32)
    for a, b in ((0, 1000), (1000, 1001), (1001, 4100), (M - 3000, M)):
        qa, sa = lib.bi_rmsnorm_quantize_e4m3(x[a:b].contiguous(), gg, 1e-5)
        assert np.array_equal(u8(qa), q[a:b]), (a, b)
        assert np.array_equal(sa.cpu().numpy().view(np.uint32), sc[a:b]), (a, b)
