"""GPU parity of bi_gemm_bf16 against the CPU oracle, through the C ABI.

Bar (from the oracle's fp32 result): per element |err| <= 2e-2*sqrt(K/4096)*rms(row)
+ half a bf16 ulp, relative Frobenius error <= 5e-3; bit-exact where every
summation order is exact (integer inputs, identity / permutation weights)."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_parity
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


def run(lib, X, W, pins=None):
    x = X.cuda()
    w = W.cuda()
    y = lib.bi_gemm_bf16(x, w, pins=pins)
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_OK
    return bf16_bits(y)


def pins_for(lib, N, K, **kw):
    return lib.bi_pins_default(N, K).replace(**kw)


@pytest.mark.parametrize("M", [1, 3, 7, 16, 33])
@pytest.mark.parametrize("ctas", [1, 2])
def test_tiny_config_parity(lib, oracle, M, ctas):
    """X [M,256] ~N(0,1), W [128,256] ~N(0,0.02), seed 0."""
    X = inputs.normal((M, 256), seed=0, stream=inputs.STREAM_X)
    W = inputs.normal((128, 256), std=0.02, seed=0, stream=inputs.STREAM_W)
    yf, _ = oracle.gemm(inputs.bits(X), inputs.bits(W))
    outs = []
    for flags in (lib.BI_FLAG_SCHEDULE_LOCAL, lib.BI_FLAG_SCHEDULE_CLUSTER):
        got = run(lib, X, W, pins_for(lib, 128, 256, flags=flags, mma_ctas=ctas))
        check_gemm_parity(got, yf, 256, "tiny M=%d flags=%d ctas=%d" % (M, flags, ctas))
        outs.append(got)
    assert np.array_equal(outs[0], outs[1])


SHAPES = [
    # (M, N, K): several tiles and ragged tails in every dimension
    (200, 300, 200),     # K tail (200 = 3*64 + 8), N tail, M tail
    (129, 256, 512),
    (1, 640, 1024),
    (300, 128, 64),
    (65, 136, 8),        # a single partial K tile
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("S,T", [(1, 128), (2, 64), (3, 128), (2, 256), (4, 64), (5, 256)])
@pytest.mark.parametrize("ctas", [1, 2])
def test_ragged_parity_and_schedules_agree(lib, oracle, M, N, K, S, T, ctas):
    kt = -(-K // 64)
    if S > kt:
        pytest.skip("more splits than K tiles")
    X = inputs.normal((M, K), seed=1, stream=0)
    W = inputs.normal((N, K), std=0.02, seed=1, stream=1)
    yf, _ = oracle.gemm(inputs.bits(X), inputs.bits(W))
    outs = []
    scheds = [lib.BI_FLAG_SCHEDULE_LOCAL, lib.BI_FLAG_SCHEDULE_CLUSTER, lib.BI_FLAG_SCHEDULE_AUTO,
              lib.BI_FLAG_SCHEDULE_AUTO | lib.BI_FLAG_PREFETCH_W]
    if S >= 3:
        scheds.append(lib.BI_FLAG_SCHEDULE_CHAIN)
    for flags in scheds:
        got = run(lib, X, W, pins_for(lib, N, K, split_k=S, tok_tile=T, flags=flags, mma_ctas=ctas))
        check_gemm_parity(got, yf, K, "M=%d N=%d K=%d S=%d T=%d ctas=%d flags=%d" % (M, N, K, S, T, ctas, flags))
        outs.append(got)
    # the schedule and the early weight stream change when and where things are
    # computed, never a bit
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("M,N,K", [(300, 256, 1472), (513, 384, 640), (256, 200, 704), (1, 256, 1472)])
@pytest.mark.parametrize("S", [1, 2, 3])
@pytest.mark.parametrize("ctas", [1, 2])
def test_ktile_pairs_change_no_bit(lib, oracle, M, N, K, S, ctas):
    """Copies of two K tiles (3-D tensor maps) against one-tile copies, with
    odd K-tile counts per split (the last copy of a split reaches past it) and a
    short X box at M=1 (which keeps one tile per copy)."""
    X = inputs.normal((M, K), seed=11, stream=0)
    W = inputs.normal((N, K), std=0.02, seed=11, stream=1)
    yf, _ = oracle.gemm(inputs.bits(X), inputs.bits(W))
    outs = []
    for extra in (0, lib.BI_FLAG_KTILE_PAIRS):
        for sched in (lib.BI_FLAG_SCHEDULE_LOCAL, lib.BI_FLAG_SCHEDULE_CLUSTER) + \
                ((lib.BI_FLAG_SCHEDULE_CHAIN,) if S >= 3 else ()):
            pins = pins_for(lib, N, K, split_k=S, tok_tile=256, mma_ctas=ctas, flags=sched | extra)
            plan = lib.bi_gemm_plan_describe(M, N, K, pins)
            assert plan.kps == (2 if extra and ctas == 2 and plan.x_box_rows == 128 else 1)
            got = run(lib, X, W, pins)
            check_gemm_parity(got, yf, K, "M=%d N=%d K=%d S=%d ctas=%d flags=%d" % (M, N, K, S, ctas, sched | extra))
            outs.append(got)
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("S,T", [(1, 128), (3, 64), (2, 256)])
@pytest.mark.parametrize("ctas", [1, 2])
def test_integer_inputs_bit_exact(lib, oracle, S, T, ctas):
    """Integer inputs: every partial sum is an exact integer, so every reduction
    tree gives the same bits as the oracle."""
    M, N, K = 77, 260, 704
    X = inputs.integers((M, K), -8, 8, seed=2, stream=0)
    W = inputs.integers((N, K), -8, 8, seed=2, stream=1)
    _, yb = oracle.gemm(inputs.bits(X), inputs.bits(W))
    got = run(lib, X, W, pins_for(lib, N, K, split_k=S, tok_tile=T, mma_ctas=ctas))
    assert np.array_equal(got, yb)


def test_observation_mma_pairing(lib):
    """Not a requirement (the pairing is a pin, part of the tree): records
    whether cta_group::1 and cta_group::2 MMAs of the same chain give the same
    bits on this GPU."""
    M, N, K = 300, 512, 1024
    X = inputs.normal((M, K), seed=7, stream=0)
    W = inputs.normal((N, K), std=0.02, seed=7, stream=1)
    a = run(lib, X, W, pins_for(lib, N, K, split_k=2, tok_tile=128, mma_ctas=1))
    b = run(lib, X, W, pins_for(lib, N, K, split_k=2, tok_tile=128, mma_ctas=2))
    print("cta_group::1 vs ::2: %d of %d elements differ" % (int((a != b).sum()), a.size))


def test_identity_and_permutation_weights(lib):
    K = 256
    X = inputs.normal((150, K), seed=3, stream=0)
    eye = inputs.to_bf16(np.eye(K, dtype=np.float32))
    assert np.array_equal(run(lib, X, eye), inputs.bits(X))
    perm = np.random.default_rng(3).permutation(K)
    P = np.zeros((K, K), dtype=np.float32)
    P[np.arange(K), perm] = 1.0
    got = run(lib, X, inputs.to_bf16(P), pins_for(lib, K, K, split_k=2))
    assert np.array_equal(got, inputs.bits(X)[:, perm])


def test_one_hot_rows_exact(lib, oracle):
    """One non-zero per X row: each output is a single exact product."""
    M, N, K = 40, 200, 512
    r = np.random.default_rng(4)
    Xf = np.zeros((M, K), dtype=np.float32)
    Xf[np.arange(M), r.integers(0, K, M)] = r.standard_normal(M).astype(np.float32)
    X = inputs.to_bf16(Xf)
    W = inputs.normal((N, K), std=0.02, seed=4, stream=1)
    _, yb = oracle.gemm(inputs.bits(X), inputs.bits(W))
    assert np.array_equal(run(lib, X, W, pins_for(lib, N, K, split_k=4)), yb)


def test_zero_rows_and_m_zero(lib):
    x = torch.zeros((5, 128), dtype=torch.bfloat16, device="cuda")
    w = inputs.normal((64, 128), std=0.02, seed=5, stream=1).cuda()
    y = lib.bi_gemm_bf16(x, w)
    assert torch.all(y.float() == 0)
    empty = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    assert lib.bi_gemm_bf16(empty, w).shape == (0, 64)


def test_errors_launch_nothing(lib):
    w = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    y = torch.full((4, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    bad = lib.bi_pins_default(64, 128).replace(split_k=5)
    with pytest.raises(lib.BiError) as e:
        lib.bi_gemm_bf16(x, w, out=y, pins=bad)
    assert e.value.status == lib.BI_ERR_ILLEGAL_PINS
    torch.cuda.synchronize()
    assert torch.all(y.float() == 7.0)
    # a misaligned view (offset of one element = 2 bytes)
    buf = torch.zeros(4 * 128 + 1, dtype=torch.bfloat16, device="cuda")
    xm = buf[1:].view(4, 128)
    with pytest.raises(lib.BiError) as e:
        lib.bi_gemm_bf16(xm, w, out=y)
    assert e.value.status == lib.BI_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert torch.all(y.float() == 7.0)


def test_stores_stay_inside_y(lib):
    """Guard bands around Y stay untouched for ragged M and N."""
    M, N, K = 70, 200, 256
    X = inputs.normal((M, K), seed=6, stream=0).cuda()
    W = inputs.normal((N, K), std=0.02, seed=6, stream=1).cuda()
    guard = 4096
    buf = torch.full((guard + M * N + guard,), 123.0, dtype=torch.bfloat16, device="cuda")
    y = buf[guard:guard + M * N].view(M, N)
    for S, T, ctas in [(1, 64, 1), (2, 128, 1), (4, 256, 1), (1, 64, 2), (2, 128, 2), (4, 256, 2)]:
        for flags in (lib.BI_FLAG_SCHEDULE_LOCAL, lib.BI_FLAG_SCHEDULE_CLUSTER):
            lib.bi_gemm_bf16(X, W, out=y, pins=lib.bi_pins_default(N, K).replace(
                split_k=S, tok_tile=T, flags=flags, mma_ctas=ctas))
            torch.cuda.synchronize()
            assert torch.all(buf[:guard].float() == 123.0) and torch.all(buf[guard + M * N:].float() == 123.0)


@pytest.mark.parametrize("M", [1, 300, 2500])
def test_host_buffers_give_the_device_bits(lib, M):
    """bi_gemm_bf16_host (X and Y in host memory, rows in 512-row chunks for
    down_proj: 2500 rows are 5 chunks, the last one partial) gives the bits of
    bi_gemm_bf16 on device copies, from page-locked and from pageable memory."""
    N, K = 4096, 14336
    X = inputs.normal((M, K), seed=30, stream=0)
    W = inputs.device_normal((N, K), std=0.02, seed=30, stream=1)
    want = bf16_bits(lib.bi_gemm_bf16(X.cuda(), W))
    y = lib.bi_gemm_bf16_host(X.contiguous().pin_memory(), W)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(y), want)
    y2 = torch.empty((M, N), dtype=torch.bfloat16)
    lib.bi_gemm_bf16_host(X.contiguous(), W, out=y2)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(y2), want)


def test_host_buffer_calls_back_to_back(lib):
    """Consecutive calls on one stream and one workspace, with no
    synchronisation between them, each give their own bits."""
    N, K = 6144, 4096
    W = inputs.device_normal((N, K), std=0.02, seed=31, stream=1)
    Ms = (5000, 1, 2049, 700)
    xs = [inputs.normal((M, K), seed=31, stream=10 + i).pin_memory() for i, M in enumerate(Ms)]
    ws = torch.empty(lib.bi_gemm_bf16_host_workspace_bytes(max(Ms), N, K), dtype=torch.uint8, device="cuda")
    outs = [lib.bi_gemm_bf16_host(x, W, workspace=ws) for x in xs]
    torch.cuda.synchronize()
    for x, y in zip(xs, outs):
        assert np.array_equal(bf16_bits(y), bf16_bits(lib.bi_gemm_bf16(x.cuda(), W)))


@pytest.mark.parametrize("depth,chunk_rows", [(0, 0), (3, 0), (8, 0), (0, 1000), (4, 128), (2, 4999), (8, 2304)])
def test_host_batch_gives_each_job_its_device_bits(lib, depth, chunk_rows):
    """bi_gemm_bf16_host_batch over jobs of one (N, K) (an empty job, one row,
    ragged counts, jobs sharing W and jobs with their own W) gives each job
    the bits of bi_gemm_bf16 alone, with the two-slot ring the workspace query
    sizes (depth 0 here) or a deeper one, and the default chunk (2048 rows at
    K = 4096) or an explicit one (ragged, small, larger than most jobs)."""
    N, K = 6144, 4096
    Wa = inputs.device_normal((N, K), std=0.02, seed=32, stream=1)
    Wb = inputs.device_normal((N, K), std=0.02, seed=32, stream=2)
    Ms = (0, 1, 5000, 3, 2049, 700)
    Wl = [Wa, Wb, Wa, Wb, Wb, Wa]
    xs = [inputs.normal((M, K), seed=32, stream=10 + i).pin_memory() for i, M in enumerate(Ms)]
    ws = None
    if depth:
        ws = torch.empty(depth * lib.bi_gemm_bf16_host_slot_bytes(list(Ms), N, K, chunk_rows), dtype=torch.uint8,
                         device="cuda")
    outs = lib.bi_gemm_bf16_host_batch(xs, Wl, workspace=ws, chunk_rows=chunk_rows)
    torch.cuda.synchronize()
    for x, w, y in zip(xs, Wl, outs):
        assert y.shape == (x.shape[0], N)
        if x.shape[0]:
            assert np.array_equal(bf16_bits(y), bf16_bits(lib.bi_gemm_bf16(x.cuda(), w)))


def test_host_batch_calls_back_to_back(lib):
    """Two job lists enqueued on one stream and one workspace without a
    synchronisation between them, then a single-job call: each keeps its own
    bits (down_proj shape, 512-row chunks)."""
    N, K = 4096, 14336
    W = inputs.device_normal((N, K), std=0.02, seed=33, stream=1)
    lists = [(1, 1100, 64), (513, 2, 1024)]
    ws = torch.empty(lib.bi_gemm_bf16_host_batch_workspace_bytes([1100, 1024, 700], N, K), dtype=torch.uint8,
                     device="cuda")
    xs = [[inputs.normal((M, K), seed=33, stream=100 * a + i).pin_memory() for i, M in enumerate(Ms)]
          for a, Ms in enumerate(lists)]
    outs = [lib.bi_gemm_bf16_host_batch(x, [W] * len(x), workspace=ws) for x in xs]
    x1 = inputs.normal((700, K), seed=33, stream=999).pin_memory()
    y1 = lib.bi_gemm_bf16_host(x1, W, workspace=ws)
    torch.cuda.synchronize()
    for xl, yl in zip(xs, outs):
        for x, y in zip(xl, yl):
            assert np.array_equal(bf16_bits(y), bf16_bits(lib.bi_gemm_bf16(x.cuda(), W)))
    assert np.array_equal(bf16_bits(y1), bf16_bits(lib.bi_gemm_bf16(x1.cuda(), W)))
