"""The GLOBAL schedule of bi_gemm_bf16_ws: split chains on any SMs, their
partials folded in ascending split order in a caller workspace by the chain
that finishes its tile's set last.

The tree is a function of (N, K, pins) only, so for the same pins the GLOBAL
schedule must give the bits of LOCAL and CLUSTER at every M of a single token
tile, in any order of arrival; and parity with the oracle follows from the
GEMM tests.  The workspace's counters must be zero after every completed
call (the call leaves them ready for the next one)."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_parity
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


def same_bits(a, b) -> bool:
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def fold_workspace(lib, M, N, K, pins):
    need = lib.bi_gemm_bf16_workspace_bytes(M, N, K, pins)
    assert need > 0
    return torch.zeros(need, dtype=torch.uint8, device="cuda"), need


def counters_zero(ws, N) -> bool:
    tiles = -(-N // 128)
    return bool((ws[: tiles * 4] == 0).all())


@pytest.mark.parametrize("M", [1, 7, 33, 64, 65, 100, 128])
@pytest.mark.parametrize("N,K", [(640, 1024), (300, 200), (1024, 4096)])
@pytest.mark.parametrize("S", [2, 3, 4, 7, 8])
def test_global_equals_local_and_cluster(lib, oracle, M, N, K, S):
    if S > -(-K // 64):
        pytest.skip("more splits than K tiles")
    X = inputs.normal((M, K), seed=M + S, stream=0)
    W = inputs.normal((N, K), std=0.02, seed=M + S, stream=1)
    x, w = X.cuda(), W.cuda()
    base = lib.bi_pins_default(N, K).replace(split_k=S)
    pins_g = base.replace(flags=base.flags | lib.BI_FLAG_SCHEDULE_GLOBAL)
    ws, need = fold_workspace(lib, M, N, K, pins_g)
    plan = lib.bi_gemm_plan_describe_ws(M, N, K, pins_g, 0, need)
    assert plan.schedule == lib.BI_FLAG_SCHEDULE_GLOBAL
    # a workspace one byte short: the call runs without the GLOBAL schedule
    assert lib.bi_gemm_plan_describe_ws(M, N, K, pins_g, 0, need - 1).schedule != lib.BI_FLAG_SCHEDULE_GLOBAL
    got = [lib.bi_gemm_bf16(x, w, pins=pins_g, workspace=ws) for _ in range(3)]   # reuses the counters
    loc = lib.bi_gemm_bf16(x, w, pins=base.replace(flags=base.flags | lib.BI_FLAG_SCHEDULE_LOCAL))
    clu = lib.bi_gemm_bf16(x, w, pins=base.replace(flags=base.flags | lib.BI_FLAG_SCHEDULE_CLUSTER))
    auto = lib.bi_gemm_bf16(x, w, pins=base, workspace=ws)
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_OK
    for g in got + [clu, auto]:
        assert same_bits(g, loc)
    assert counters_zero(ws, N)
    yf, _ = oracle.gemm(inputs.bits(X), inputs.bits(W))
    check_gemm_parity(bf16_bits(got[0]), yf, K, "GLOBAL M=%d N=%d K=%d S=%d" % (M, N, K, S))


@pytest.mark.parametrize("N,K,S", [(6144, 4096, 3), (28672, 4096, 2), (4096, 14336, 4), (10240, 8192, 3),
                                   (8192, 8192, 7), (8192, 28672, 5)])
def test_global_full_shapes_every_decode_m_switch(lib, N, K, S):
    """Full projection shapes: every split count the GLOBAL schedule takes,
    across the 64/65 token-tile switch, against the cluster schedule."""
    x = inputs.device_normal((70, K), seed=N, stream=0, device=torch.device("cuda"))
    w = inputs.device_normal((N, K), std=0.02, seed=N, stream=1, device=torch.device("cuda"))
    base = lib.bi_pins_default(N, K).replace(split_k=S)
    pins_g = base.replace(flags=base.flags | lib.BI_FLAG_SCHEDULE_GLOBAL)
    ws, _ = fold_workspace(lib, 70, N, K, pins_g)
    ref = lib.bi_gemm_bf16(x, w, pins=base.replace(flags=base.flags | lib.BI_FLAG_SCHEDULE_LOCAL))
    for M in (1, 2, 31, 64, 65, 70):
        got = lib.bi_gemm_bf16(x[:M], w, pins=pins_g, workspace=ws)
        torch.cuda.synchronize()
        assert same_bits(got, ref[:M]), "M=%d" % M
    assert counters_zero(ws, N)
    assert lib.bi_last_device_status() == lib.BI_OK


def test_global_partials_region_contents_do_not_matter(lib):
    M, N, K = 20, 512, 2048
    x = inputs.normal((M, K), seed=5, stream=0).cuda()
    w = inputs.normal((N, K), std=0.02, seed=5, stream=1).cuda()
    pins = lib.bi_pins_default(N, K).replace(split_k=3,
                                             flags=lib.bi_pins_default(N, K).flags | lib.BI_FLAG_SCHEDULE_GLOBAL)
    ws, need = fold_workspace(lib, M, N, K, pins)
    a = lib.bi_gemm_bf16(x, w, pins=pins, workspace=ws)
    tiles = -(-N // 128)
    cstart = (tiles * 4 + 255) // 256 * 256
    ws[cstart:] = 0xFF          # NaN patterns where the partials go
    b = lib.bi_gemm_bf16(x, w, pins=pins, workspace=ws)
    torch.cuda.synchronize()
    assert same_bits(a, b)


def test_global_stalled_producer_reports_timeout_and_recovers(lib):
    M, N, K = 3, 256, 512
    x = inputs.normal((M, K), seed=6, stream=0).cuda()
    w = inputs.normal((N, K), std=0.02, seed=6, stream=1).cuda()
    base = lib.bi_pins_default(N, K).replace(split_k=2)
    pins = base.replace(flags=base.flags | lib.BI_FLAG_SCHEDULE_GLOBAL)
    ws, _ = fold_workspace(lib, M, N, K, pins)
    assert lib.bi_last_device_status() == lib.BI_OK
    lib.bi_gemm_bf16(x, w, pins=pins.replace(flags=pins.flags | lib.BI_FLAG_DEBUG_STALL_PRODUCER), workspace=ws)
    assert lib.bi_last_device_status() == lib.BI_ERR_DEVICE_TIMEOUT
    assert lib.bi_last_device_status() == lib.BI_OK
    ws.zero_()                 # an abandoned call may leave counts behind
    got = lib.bi_gemm_bf16(x, w, pins=pins, workspace=ws)
    ref = lib.bi_gemm_bf16(x, w, pins=base)
    torch.cuda.synchronize()
    assert same_bits(got, ref)
    assert counters_zero(ws, N)
    assert lib.bi_last_device_status() == lib.BI_OK
