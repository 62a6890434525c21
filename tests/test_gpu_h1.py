"""H1: for a fixed K-tile and split sequence, the MMA's N extent (the token
tile T = 64, 128, 256) and its CTA grouping (tcgen05.mma cta_group::1, 128
weight rows per MMA, against cta_group::2, 256 rows across a CTA pair) leave
every output bit unchanged; so do copies of one or two K tiles.

Each output element is one dot-product chain of k16 MMA steps in a fixed
order; these knobs only change how many such chains one instruction computes
side by side and which SM computes them.  The library relies on this result
when the pins leave the token tile or the CTA grouping open (0): it then picks
them per launch, for speed.  The inputs span a wide exponent range so that
every accumulation step rounds.
"""
import numpy as np
import pytest
import torch

from helpers import bf16_bits
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = [
    # (M, N, K, S)
    (300, 512, 1024, 2),
    (77, 6144, 4096, 3),
    (513, 1280, 8192, 2),
    (256, 640, 704, 1),      # K % 64 != 0 never takes two-tile copies
    (1024, 4096, 14336, 4),  # Llama-3.1-8B down_proj
]


def wide_range(shape, seed, stream, std=1.0):
    """N(0, std) entries times 2^e, e uniform in [-24, 24]: bf16 values over ~48 binades."""
    x = inputs.normal(shape, std=std, seed=seed, stream=stream).float()
    e = inputs.integers(shape, -24, 24, seed=seed, stream=stream + 100).float()
    return (x * torch.exp2(e)).to(torch.bfloat16)


@pytest.mark.parametrize("M,N,K,S", CASES)
def test_mma_shape_and_grouping_leave_bits_unchanged(lib, M, N, K, S):
    X = wide_range((M, K), seed=21, stream=0).cuda()
    W = wide_range((N, K), seed=21, stream=1, std=0.02).cuda()
    base = lib.bi_pins_default(N, K).replace(split_k=S, flags=lib.BI_FLAG_SCHEDULE_AUTO)
    ref = None
    seen = []
    for T in (64, 128, 256):
        for ctas in (1, 2):
            for kp in (0, lib.BI_FLAG_KTILE_PAIRS):
                pins = base.replace(tok_tile=T, mma_ctas=ctas, flags=base.flags | kp)
                plan = lib.bi_gemm_plan_describe(M, N, K, pins)
                y = lib.bi_gemm_bf16(X, W, pins=pins)
                torch.cuda.synchronize()
                assert lib.bi_last_device_status() == lib.BI_OK
                got = bf16_bits(y)
                seen.append((T, ctas, plan.kps))
                if ref is None:
                    ref = got
                else:
                    diff = int((got != ref).sum())
                    assert diff == 0, "T=%d ctas=%d kps=%d: %d of %d elements differ from T=64 ctas=1" % (
                        T, ctas, plan.kps, diff, ref.size)
    if K % 64 == 0 and M > 128:
        assert (256, 2, 2) in seen  # the two-tile pair path ran (a short X box keeps one-tile copies)


# (M, N, K, S, token tile the open layout narrows to)
NARROW = [
    (4096, 4096, 14336, 4, 224),   # down_proj: 19 token tiles fill 4 waves of 76 pairs
    (1024, 6144, 4096, 3, 192),    # Llama-3.1-8B qkv: 144 tiles in 2 waves
    (513, 4096, 14336, 4, 160),    # down_proj just past 512
    (1500, 4096, 4096, 2, 192),
]


@pytest.mark.parametrize("M,N,K,S,T", NARROW)
def test_narrowed_token_tiles_leave_bits_unchanged(lib, M, N, K, S, T):
    """Persistent paired launches may narrow their token tile per M (224, 192,
    160) when the pins leave the layout open.  The bits must equal those of
    the pinned 256-wide paired layout and of one CTA per MMA."""
    X = wide_range((M, K), seed=22, stream=0).cuda()
    W = wide_range((N, K), seed=22, stream=1, std=0.02).cuda()
    base = lib.bi_pins_default(N, K).replace(split_k=S, flags=lib.BI_FLAG_SCHEDULE_AUTO | lib.BI_FLAG_KTILE_PAIRS)
    open_pins = base.replace(mma_ctas=0)
    plan = lib.bi_gemm_plan_describe(M, N, K, open_pins)
    assert (plan.tok_tile, plan.mma_ctas, plan.kps) == (T, 2, 2), (plan.tok_tile, plan.mma_ctas, plan.kps)
    got = bf16_bits(lib.bi_gemm_bf16(X, W, pins=open_pins))
    for ctas in (2, 1):
        ref = bf16_bits(lib.bi_gemm_bf16(X, W, pins=base.replace(mma_ctas=ctas, tok_tile=256)))
        assert np.array_equal(got, ref), ctas
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_OK


@pytest.mark.parametrize("N,K", [(4096, 14336), (6144, 4096), (640, 704)])
def test_decode_tiles_leave_bits_unchanged(lib, N, K):
    """With the grouping left open, a single token tile of up to 128 tokens
    on single-CTA MMAs runs at T = 64 or 128 with two K tiles per stage (2-D
    copies); pinning one CTA per MMA keeps the pinned T = 256 and one K tile
    per stage.  Both give the same bits, in bf16 and in FP8 (K = 704 has a
    partial last K tile); larger M cross into the pinned plans."""
    X = wide_range((256, K), seed=14, stream=0)
    W = wide_range((N, K), seed=14, stream=1, std=0.05)
    x, w = X.cuda(), W.cuda()
    base = lib.bi_pins_default(N, K)
    for M in (1, 7, 64, 65, 128, 129, 192, 256):
        open_ = lib.bi_gemm_plan_describe(M, N, K, base)
        pinned = base.replace(mma_ctas=1)
        assert lib.bi_gemm_plan_describe(M, N, K, pinned).tok_tile == 256
        got = bf16_bits(lib.bi_gemm_bf16(x[:M].contiguous(), w, pins=base))
        ref = bf16_bits(lib.bi_gemm_bf16(x[:M].contiguous(), w, pins=pinned))
        assert np.array_equal(got, ref), (M, open_.tok_tile, open_.kps)
    if K % 128 == 0:
        wq, sw = lib.bi_quantize_rows_e4m3(w)
        xq, sx = lib.bi_quantize_rows_e4m3(x)
        fb = lib.bi_pins_default_fp8(N, K)
        for M in (1, 64, 65, 128, 200):
            got = bf16_bits(lib.bi_gemm_fp8(xq[:M].contiguous(), sx[:M].contiguous(), wq, sw, pins=fb))
            ref = bf16_bits(lib.bi_gemm_fp8(xq[:M].contiguous(), sx[:M].contiguous(), wq, sw,
                                            pins=fb.replace(mma_ctas=1)))
            assert np.array_equal(got, ref), ("fp8", M)
