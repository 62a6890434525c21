"""The fused RMSNorm -> GEMM layer (bi_rmsnorm_gemm_bf16), through the C ABI.

The layer has two forms with the same bits: the RMSNorm kernel stages the
normalised rows for the GEMM (the default, or BI_FLAG_NORM_STAGED), or the
GEMM applies the RMSNorm to each X tile in shared memory, with the per-row
scale r computed beforehand by the RMSNorm's own lane partition and butterfly
(BI_FLAG_NORM_SMEM).  The
layer is defined as the composition of the two calls through the bf16
normalised rows, so the check is bit equality with
bi_gemm_bf16(bi_rmsnorm_bf16(X)) under the same pins, in both forms, for every
schedule, CTA grouping, copy size and token-tile width the planner can
choose, plus parity of the result with the oracle (its GEMM fed the GPU's
normalised rows, its RMSNorm within one ulp)."""
import numpy as np
import pytest
import torch

from helpers import EPS, bf16_bits, check_gemm_parity, check_ulp
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


def problem(M, N, K, seed):
    X = inputs.normal((M, K), seed=seed, stream=0)
    g = inputs.normal((K,), std=0.1, mean=1.0, seed=seed, stream=2)
    W = inputs.normal((N, K), std=0.02, seed=seed, stream=1)
    return X, g, W


def fused_and_composed(lib, x, gg, w, pins=None):
    fused = lib.bi_rmsnorm_gemm_bf16(x, gg, w, EPS, pins=pins)
    comp = lib.bi_gemm_bf16(lib.bi_rmsnorm_bf16(x, gg, EPS), w, pins=pins)
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_OK
    return fused, comp


def forms(lib, pins):
    """The pins with each form of the fused layer forced."""
    return [pins.replace(flags=pins.flags | f) for f in (lib.BI_FLAG_NORM_SMEM, lib.BI_FLAG_NORM_STAGED)]


def same_bits(a, b) -> bool:
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


# Default pins; the planner's choice at each size is noted (single-CTA decode
# tiles of 64 / 128 tokens with 2-D copies, CTA pairs with narrowed tiles,
# clusters of pairs, the chained schedule, single-CTA 256-token tiles).
PLANNED = [
    (1, 640, 1024),       # decode T=64, clusters of 8
    (37, 640, 1024),      # decode T=64, 40 valid rows copied
    (65, 640, 1024),      # decode T=128
    (128, 1024, 512),     # decode T=128, every row valid
    (129, 640, 1024),     # pairs, T=160, persistent
    (300, 384, 640),      # pairs, T=160, one split
    (129, 6144, 4096),    # clusters of pairs, T=256 (qkv shape)
    (512, 6144, 4096),    # pairs, T=192 (qkv shape)
    (1000, 4096, 14336),  # chained clusters of pairs / pairs (down_proj shape)
    (200, 4096, 14336),   # single CTAs, T=256, one K tile per copy
]


@pytest.mark.parametrize("M,N,K", PLANNED)
def test_fused_equals_composition_planned(lib, M, N, K):
    X, g, W = problem(M, N, K, seed=M + N)
    x, gg, w = X.cuda(), g.cuda(), W.cuda()
    fused, comp = fused_and_composed(lib, x, gg, w)
    assert same_bits(fused, comp)
    for pins in forms(lib, lib.bi_pins_default(N, K)):
        f, _ = fused_and_composed(lib, x, gg, w, pins)
        assert same_bits(f, comp), "flags=%#x" % pins.flags


SHAPES = [
    (200, 300, 200),     # K tail (200 = 3*64 + 8), N tail, M tail
    (129, 256, 512),
    (1, 640, 1024),
    (300, 128, 64),
    (65, 136, 8),        # a single partial K tile
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("S,T", [(1, 128), (2, 64), (3, 256), (5, 256)])
@pytest.mark.parametrize("ctas", [0, 1, 2])
def test_fused_equals_composition_pinned(lib, M, N, K, S, T, ctas):
    kt = -(-K // 64)
    if S > kt:
        pytest.skip("more splits than K tiles")
    X, g, W = problem(M, N, K, seed=7)
    x, gg, w = X.cuda(), g.cuda(), W.cuda()
    scheds = [lib.BI_FLAG_SCHEDULE_LOCAL, lib.BI_FLAG_SCHEDULE_CLUSTER,
              lib.BI_FLAG_SCHEDULE_AUTO | lib.BI_FLAG_KTILE_PAIRS,
              lib.BI_FLAG_SCHEDULE_AUTO | lib.BI_FLAG_KTILE_PAIRS | lib.BI_FLAG_PREFETCH_W]
    if S >= 3:
        scheds.append(lib.BI_FLAG_SCHEDULE_CHAIN | lib.BI_FLAG_KTILE_PAIRS)
    outs = []
    for flags in scheds:
        pins = lib.bi_pins_default(N, K).replace(split_k=S, tok_tile=T, mma_ctas=ctas, flags=flags)
        for p in forms(lib, pins):
            fused, comp = fused_and_composed(lib, x, gg, w, p)
            assert same_bits(fused, comp), "S=%d T=%d ctas=%d flags=%#x" % (S, T, ctas, p.flags)
            outs.append(fused)
    assert all(same_bits(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("M,N,K", [(1, 384, 4096), (33, 256, 512), (130, 640, 256), (257, 512, 1000)])
def test_fused_parity_with_the_oracle(lib, oracle, M, N, K):
    X, g, W = problem(M, N, K, seed=2)
    x, gg, w = X.cuda(), g.cuda(), W.cuda()
    fused = lib.bi_rmsnorm_gemm_bf16(x, gg, w, EPS)
    xh = lib.bi_rmsnorm_bf16(x, gg, EPS)
    torch.cuda.synchronize()
    # the normalisation within one ulp of the oracle's; the GEMM part against
    # the oracle fed the GPU's normalised rows
    check_ulp(bf16_bits(xh), oracle.rmsnorm(inputs.bits(X), inputs.bits(g), EPS), 1, "fused norm")
    yf, _ = oracle.gemm(bf16_bits(xh), inputs.bits(W))
    check_gemm_parity(bf16_bits(fused), yf, K, "fused M=%d N=%d K=%d" % (M, N, K))
    # end to end against the oracle's composition (its own normalised rows)
    yf2, _, _ = oracle.rmsnorm_gemm(inputs.bits(X), inputs.bits(g), inputs.bits(W), EPS)
    check_gemm_parity(bf16_bits(fused), yf2, K, "fused vs oracle composition")


def test_fused_rows_are_isolated_from_nan_inf_and_huge_co_runners(lib):
    """A co-runner row of NaN, +-Inf or +-65504 gives that row a NaN or
    extreme r; no other row's bits change."""
    M, N, K = 40, 640, 1024
    X, g, W = problem(M, N, K, seed=11)
    x, gg, w = X.cuda(), g.cuda(), W.cuda()
    ref = lib.bi_rmsnorm_gemm_bf16(x, gg, w, EPS)
    bad = x.clone()
    bad[3] = float("nan")
    bad[17] = float("inf")
    bad[18] = -float("inf")
    bad[25] = 65504.0
    bad[26, ::2] = -65504.0
    got = lib.bi_rmsnorm_gemm_bf16(bad, gg, w, EPS)
    comp = lib.bi_gemm_bf16(lib.bi_rmsnorm_bf16(bad, gg, EPS), w)
    staged = lib.bi_rmsnorm_gemm_bf16(bad, gg, w, EPS, pins=forms(lib, lib.bi_pins_default(N, K))[1])
    torch.cuda.synchronize()
    assert same_bits(got, comp) and same_bits(staged, comp)
    keep = [m for m in range(M) if m not in (3, 17, 18, 25, 26)]
    assert same_bits(got[keep], ref[keep])
    assert torch.isnan(got[3].float()).all()


def test_fused_workspace_contents_do_not_matter(lib):
    M, N, K = 70, 512, 2048
    X, g, W = problem(M, N, K, seed=12)
    x, gg, w = X.cuda(), g.cuda(), W.cuda()
    need = lib.bi_rmsnorm_gemm_workspace_bytes(M, K)
    assert need >= 4 * M and need % 256 == 0
    outs = []
    for pins in forms(lib, lib.bi_pins_default(N, K)):
        for fill in (0, 0xFF, 0x7F):
            ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
            outs.append(lib.bi_rmsnorm_gemm_bf16(x, gg, w, EPS, pins=pins, workspace=ws))
    torch.cuda.synchronize()
    assert all(same_bits(outs[0], o) for o in outs[1:])


def test_fused_stalled_producer_reports_timeout_and_recovers(lib):
    M, N, K = 3, 128, 256
    X, g, W = problem(M, N, K, seed=13)
    x, gg, w = X.cuda(), g.cuda(), W.cuda()
    for ctas, flags in ((1, lib.BI_FLAG_SCHEDULE_LOCAL), (2, lib.BI_FLAG_SCHEDULE_LOCAL),
                        (1, lib.BI_FLAG_SCHEDULE_CLUSTER)):
        pins = lib.bi_pins_default(N, K).replace(split_k=2, tok_tile=128, mma_ctas=ctas,
                                                 flags=flags | lib.BI_FLAG_NORM_SMEM)
        flags = pins.flags
        assert lib.bi_last_device_status() == lib.BI_OK
        lib.bi_rmsnorm_gemm_bf16(x, gg, w, EPS, pins=pins.replace(flags=flags | lib.BI_FLAG_DEBUG_STALL_PRODUCER))
        assert lib.bi_last_device_status() == lib.BI_ERR_DEVICE_TIMEOUT
        assert lib.bi_last_device_status() == lib.BI_OK
        fused, comp = fused_and_composed(lib, x, gg, w, pins)
        assert same_bits(fused, comp)


def test_fused_tiny_batches_every_m(lib):
    """In shared memory, up to 4 rows the GEMM computes the rows' RMSNorm
    scales itself (one launch); from 5 a row-scale kernel does.  Every M
    across the switch, with a NaN and an infinite row among them, gives the
    composition's bits."""
    N, K = 384, 4096
    X, g, W = problem(17, N, K, seed=14)
    x, gg, w = X.cuda(), g.cuda(), W.cuda()
    x[2] = float("nan")
    x[11, 7] = float("inf")
    pins = forms(lib, lib.bi_pins_default(N, K))[0]
    comp = lib.bi_gemm_bf16(lib.bi_rmsnorm_bf16(x, gg, EPS), w)
    for M in range(1, 18):
        for p in (pins, pins.replace(flags=pins.flags | lib.BI_FLAG_PREFETCH_W)):
            got = lib.bi_rmsnorm_gemm_bf16(x[:M], gg, w, EPS, pins=p)
            torch.cuda.synchronize()
            assert same_bits(got, comp[:M]), "M=%d flags=%#x" % (M, p.flags)
    assert lib.bi_last_device_status() == lib.BI_OK


@pytest.mark.parametrize("M", [1, 9, 64, 100])
def test_fused_with_a_fold_workspace(lib, M):
    """A fused-call workspace with room for the GEMM's fold in front: the
    GLOBAL schedule folds the split partials there; both forms keep the
    composition's bits, and the fold counters at the front are zero after
    every call, whatever M the calls use."""
    N, K = 1024, 4096
    X, g, W = problem(128, N, K, seed=15)
    x, gg, w = X.cuda(), g.cuda(), W.cuda()
    pins = lib.bi_pins_default(N, K).replace(split_k=3)
    pins = pins.replace(flags=pins.flags | lib.BI_FLAG_SCHEDULE_GLOBAL)
    front = max(lib.bi_gemm_bf16_workspace_bytes(m, N, K, pins) for m in (1, 128))
    assert front > 0
    ws = torch.zeros(front + lib.bi_rmsnorm_gemm_workspace_bytes(128, K), dtype=torch.uint8, device="cuda")
    comp = lib.bi_gemm_bf16(lib.bi_rmsnorm_bf16(x, gg, EPS), w, pins=pins)
    for p in forms(lib, pins):
        for m in (M, 128, M):
            got = lib.bi_rmsnorm_gemm_bf16(x[:m], gg, w, EPS, pins=p, workspace=ws)
            torch.cuda.synchronize()
            assert same_bits(got, comp[:m]), "M=%d flags=%#x" % (m, p.flags)
            assert bool((ws[: 8 * 4] == 0).all())        # the counters of the 8 W tiles
    assert lib.bi_last_device_status() == lib.BI_OK
