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
