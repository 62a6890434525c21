"""Host-side pieces of bench.py that every reported number rests on: the
algorithmic work of a GEMM (W counted once), the roofline
time, the L2-defeating copy counts and the kernel fingerprint."""
import math
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_gemm_work_counts_w_once():
    f, b = bench.gemm_work(1, 4096, 14336)
    assert f == 2.0 * 4096 * 14336
    assert b == 2.0 * (4096 * 14336 + 14336 + 4096)        # W, X and Y in bf16
    f, b = bench.gemm_work(8192, 4096, 14336)
    assert f == pytest.approx(962.07e9, rel=1e-4)          # 2 M N K
    assert b == 2.0 * (4096 * 14336 + 8192 * 14336 + 8192 * 4096)


def test_roofline_time_takes_the_slower_bound():
    peaks = {"bf16_tflops": 1905.4, "hbm_gbs": 6782.8}
    # decode: bytes bound (W streamed once)
    f, b = bench.gemm_work(1, 4096, 14336)
    assert bench.roof_time_us(f, b, peaks) == pytest.approx(b / (6782.8 * 1e3))
    # large M: tensor bound
    f, b = bench.gemm_work(8192, 4096, 14336)
    assert bench.roof_time_us(f, b, peaks) == pytest.approx(f / (1905.4 * 1e6))


def test_copies_defeat_l2():
    for nbytes in (1, 10 << 20, 117 << 20, 470 << 20, 4 << 30):
        n = bench.copies_for(nbytes)
        assert n >= 1
        if n < 64:
            assert n * nbytes >= 2 * bench.L2_BYTES or n == 1 and nbytes >= 2 * bench.L2_BYTES
    assert bench.copies_for(117 << 20) == math.ceil(2 * bench.L2_BYTES / (117 << 20)) + 1


def test_fingerprint_is_a_sha256_of_the_kernel_sources():
    fp = bench.build_fingerprint()
    assert fp is None or (len(fp) == 64 and all(c in "0123456789abcdef" for c in fp))
