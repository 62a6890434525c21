"""Batch invariance on the GPU, bit for bit (GPU against GPU).

CoRun (Padding is Simple and Efficient for Deterministic LLM Inference),
Sec. III-B, Def. 1: x_i = x'_j implies F_n(X)_i = F_m(X')_j for all batch sizes
n, m and positions i, j; Def. 2 (position invariance) is the permutation case.
Detent, Sec. 8.1, tests reruns, co-batch changes and row moves bitwise.  Here:
  - M sweeps: row i's output bits are the same for every M > i;
  - permutations: F(PX) = P F(X);
  - co-runners: target rows embedded at random positions among other rows,
    including rows of +-65504, +-inf and NaN, give the same bits;
  - reruns give the same bits;
  - a negative control: an M-dependent split count (what a shape-picking
    library does) is caught by the same comparison."""
import numpy as np
import pytest
import torch

from helpers import EPS
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


def bits16(t):
    return t.view(torch.int16)


def rows_equal(a, b):
    return torch.equal(bits16(a), bits16(b))


# ---------------------------------------------------------------------------
# configuration 2: down_proj, every M from 1 to 8192
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def down_proj(lib):
    N, K = 4096, 14336
    W = inputs.device_normal((N, K), std=0.02, seed=0, stream=inputs.STREAM_W)
    X = inputs.device_normal((8192, K), seed=0, stream=inputs.STREAM_X)
    ref = lib.bi_gemm_bf16(X, W)
    torch.cuda.synchronize()
    return X, W, ref


def test_down_proj_every_m_1_to_8192(lib, down_proj):
    X, W, ref = down_proj
    out = torch.empty_like(ref)
    bad = []
    for M in range(1, 8193):
        lib.bi_gemm_bf16(X[:M], W, out=out[:M])
        if not rows_equal(out[:M], ref[:M]):
            bad.append(M)
        if M % 512 == 0:
            torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_OK
    assert not bad, "row bits changed with M at M = %s" % bad[:10]


def test_down_proj_reruns_and_schedules(lib, down_proj):
    X, W, ref = down_proj
    pins = lib.bi_pins_default(4096, 14336)
    for M in (1, 64, 300):
        for flags in (lib.BI_FLAG_SCHEDULE_LOCAL, lib.BI_FLAG_SCHEDULE_CLUSTER):
            y = lib.bi_gemm_bf16(X[:M], W, pins=pins.replace(flags=flags))
            assert rows_equal(y, ref[:M]), (M, flags)
    assert rows_equal(lib.bi_gemm_bf16(X, W), ref)


@pytest.mark.parametrize("M", [1, 2, 8, 33, 128, 1024, 4096, 8192])
def test_down_proj_permutations(lib, down_proj, M):
    X, W, ref = down_proj
    perm = torch.from_numpy(np.random.default_rng(M).permutation(M)).cuda()
    y = lib.bi_gemm_bf16(X[:M][perm].contiguous(), W)
    assert rows_equal(y, ref[:M][perm])


def test_negative_control_m_dependent_split(lib, down_proj):
    """A library that picks the split count from M (1 split for a large batch,
    4 for a single token, as shape-aware split-K does) changes row bits; the
    same comparison that passes above must fail here."""
    X, W, ref = down_proj
    pins = lib.bi_pins_default(4096, 14336)
    y_split1 = lib.bi_gemm_bf16(X[:64], W, pins=pins.replace(split_k=1))
    y_split4 = lib.bi_gemm_bf16(X[:64], W, pins=pins.replace(split_k=4))
    assert not rows_equal(y_split1, y_split4)
    differing = (bits16(y_split1) != bits16(y_split4)).any(dim=1).sum().item()
    assert differing > 0


def test_observation_torch_mm(lib, down_proj):
    """Not a requirement: records whether cuBLAS (torch.mm) keeps row bits
    across M on this GPU (it picks kernels by shape)."""
    X, W, _ = down_proj
    ref = torch.mm(X[:4096], W.t())
    changed = []
    for M in (1, 8, 64, 256, 1024):
        if not rows_equal(torch.mm(X[:M], W.t()), ref[:M]):
            changed.append(M)
    print("torch.mm row bits differ from the M=4096 result at M in", changed)


# ---------------------------------------------------------------------------
# configuration 1: tiny shape, rows among co-runners
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M", [1, 3, 7, 16, 33])
def test_tiny_corunners(lib, M):
    W = inputs.normal((128, 256), std=0.02, seed=0, stream=inputs.STREAM_W).cuda()
    target = inputs.normal((M, 256), seed=0, stream=inputs.STREAM_X)
    ref = lib.bi_gemm_bf16(target.cuda(), W)
    cases = [(b, None) for b in (M, 64, 1000, 8192) if b >= M]
    cases += [(300, 65504.0), (300, -65504.0), (300, float("inf")), (300, float("-inf")),
              (300, float("nan"))]
    for i, (batch, fill) in enumerate(cases):
        full, pos = inputs.scatter_rows(target, batch, seed=100 + i, corunner_fill=fill)
        y = lib.bi_gemm_bf16(full.cuda(), W)
        assert rows_equal(y[torch.from_numpy(pos).cuda()], ref), (batch, fill)
    xh_ref = lib.bi_rmsnorm_bf16(target.cuda(), torch.ones(256, dtype=torch.bfloat16, device="cuda"))
    full, pos = inputs.scatter_rows(target, 97, seed=7, corunner_fill=float("nan"))
    xh = lib.bi_rmsnorm_bf16(full.cuda(), torch.ones(256, dtype=torch.bfloat16, device="cuda"))
    assert rows_equal(xh[torch.from_numpy(pos).cuda()], xh_ref)


# ---------------------------------------------------------------------------
# configuration 3: fused RMSNorm + qkv / gate_up projections
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N", [6144, 28672])
def test_fused_projection_invariance(lib, N):
    K = 4096
    W = inputs.device_normal((N, K), std=0.02, seed=0, stream=inputs.STREAM_W)
    g = inputs.device_normal((K,), std=0.1, mean=1.0, seed=0, stream=inputs.STREAM_G)
    X = inputs.device_normal((8192, K), seed=0, stream=inputs.STREAM_X)
    ref = lib.bi_rmsnorm_gemm_bf16(X, g, W, EPS)
    for M in (1, 8, 32, 128, 1024, 4096):
        assert rows_equal(lib.bi_rmsnorm_gemm_bf16(X[:M], g, W, EPS), ref[:M]), M
        perm = torch.from_numpy(np.random.default_rng(M).permutation(M)).cuda()
        assert rows_equal(lib.bi_rmsnorm_gemm_bf16(X[:M][perm].contiguous(), g, W, EPS), ref[:M][perm]), M
    # co-runner swap: the first 32 rows, with every other row replaced
    Xs = X[:1024].clone()
    Xs[32:] = inputs.device_normal((1024 - 32, K), seed=5, stream=77)
    assert rows_equal(lib.bi_rmsnorm_gemm_bf16(Xs, g, W, EPS)[:32], ref[:32])


# ---------------------------------------------------------------------------
# configuration 4: RMSNorm token-count sweep
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H", [4096, 8192])
def test_rmsnorm_token_count_sweep(lib, H):
    x = inputs.rows_loguniform(16384, H, seed=0, stream=0).cuda()
    g = inputs.normal((H,), std=0.1, mean=1.0, seed=0, stream=2).cuda()
    ref = lib.bi_rmsnorm_bf16(x, g, EPS)
    counts = [1 << i for i in range(15)] + [3, 37, 1001]
    for M in counts:
        assert rows_equal(lib.bi_rmsnorm_bf16(x[:M], g, EPS), ref[:M]), M
    perm = torch.from_numpy(np.random.default_rng(1).permutation(1001)).cuda()
    assert rows_equal(lib.bi_rmsnorm_bf16(x[:1001][perm].contiguous(), g, EPS), ref[:1001][perm])
