"""Parity at the full workload sizes, in the launch configurations the
benchmark times, on whole rows the oracle computes (a few distinct rows of
each batch, every output column)."""
import numpy as np
import pytest
import torch

from helpers import EPS, bf16_bits, check_gemm_parity, check_ulp
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


def sampled_parity(oracle, X, W, Y, n_rows, seed, what):
    """Whole rows: up to n_rows distinct rows (the first and the last among
    them), every column, against the oracle's fp32 rows; the bar is the GEMM
    tolerance with rms(row) taken from the oracle's row (check_gemm_parity)."""
    M, K = X.shape
    r = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, M - 1], r.integers(0, M, n_rows)]))[:n_rows]
    idx = torch.from_numpy(rows).to(X.device)
    yf, _ = oracle.gemm(inputs.bits(X[idx]), inputs.bits(W))
    check_gemm_parity(bf16_bits(Y[idx]), yf, K, what)


@pytest.mark.parametrize("N,K,Ms", SHAPES)
def test_fullsize_gemm_sampled_parity(lib, oracle, N, K, Ms):
    W = inputs.device_normal((N, K), std=0.02, seed=0, stream=inputs.STREAM_W)
    # the benchmark's launch configuration: bi_gemm_bf16_ws with a zeroed fold
    # workspace and the early weight stream
    pins = lib.bi_pins_default(N, K)
    pins = pins.replace(flags=pins.flags | lib.BI_FLAG_PREFETCH_W)
    for M in Ms:
        X = inputs.device_normal((M, K), seed=0, stream=inputs.STREAM_X)
        ws = torch.zeros(max(lib.bi_gemm_bf16_workspace_bytes(M, N, K, pins), 256), dtype=torch.uint8, device="cuda")
        Y = lib.bi_gemm_bf16(X, W, pins=pins, workspace=ws)
        torch.cuda.synchronize()
        assert lib.bi_last_device_status() == lib.BI_OK
        sampled_parity(oracle, X, W, Y, 6, seed=M, what="N=%d K=%d M=%d" % (N, K, M))


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
        sampled_parity(oracle, xh, W, Y, 6, seed=M, what="fused N=%d M=%d" % (N, M))


def test_fullsize_fp8_sampled_parity(lib, oracle):
    """The FP8 workload at full size (down_proj W [4096, 14336]; M = 1, 512,
    8192), in the benchmark's launch configuration (the FP8 default pins plus
    the early weight stream): whole sampled rows against the oracle's E4M3
    GEMM on the same codes and scales, with the same GEMM tolerance."""
    N, K = 4096, 14336
    W = inputs.device_normal((N, K), std=0.02, seed=1, stream=inputs.STREAM_W)
    wq, sw = lib.bi_quantize_rows_e4m3(W)
    pins = lib.bi_pins_default_fp8(N, K)
    pins = pins.replace(flags=pins.flags | lib.BI_FLAG_PREFETCH_W)
    wq_np = wq.cpu().numpy()
    sw_np = sw.cpu().numpy()
    for M in (1, 512, 8192):
        X = inputs.device_normal((M, K), seed=1, stream=inputs.STREAM_X)
        xq, sx = lib.bi_quantize_rows_e4m3(X)
        Y = lib.bi_gemm_fp8(xq, sx, wq, sw, pins=pins)
        torch.cuda.synchronize()
        assert lib.bi_last_device_status() == lib.BI_OK
        r = np.random.default_rng(M)
        rows = np.unique(np.concatenate([[0, M - 1], r.integers(0, M, 4)]))
        sx_np = sx.cpu().numpy()[rows]
        yf, _ = oracle.gemm_e4m3(xq.cpu().numpy()[rows], sx_np, wq_np, sw_np)
        ref = (yf.astype(np.float64) * sx_np[:, None] * sw_np[None, :]).astype(np.float32)
        idx = torch.from_numpy(rows).cuda()
        check_gemm_parity(bf16_bits(Y[idx]), ref, K, "fp8 N=%d K=%d M=%d" % (N, K, M))


def test_fullsize_host_batch_sweep(lib, oracle):
    """The end-to-end launch configuration of the benchmark: the whole
    down_proj M sweep (M = 1, 2, 4 .. 8192, 16383 rows) as one
    bi_gemm_bf16_host_batch call from page-locked memory, 2304-row chunks and
    a ring of 8 slots (so the last rows go in halving chunks), two weight
    copies alternating between the jobs.  Every job's rows are the bits
    bi_gemm_bf16 gives on device copies; sampled whole rows of the largest
    job are the oracle's within the GEMM tolerance."""
    N, K = 4096, 14336
    Ws = [inputs.device_normal((N, K), std=0.02, seed=0, stream=inputs.STREAM_W + 16 * i) for i in range(2)]
    Ms = [1 << i for i in range(14)]
    xs = [inputs.device_normal((M, K), seed=0, stream=inputs.STREAM_X + 16 * j).cpu().pin_memory()
          for j, M in enumerate(Ms)]
    wl = [Ws[j % 2] for j in range(len(Ms))]
    ws = torch.empty(8 * lib.bi_gemm_bf16_host_slot_bytes(Ms, N, K, 2304), dtype=torch.uint8, device="cuda")
    outs = lib.bi_gemm_bf16_host_batch(xs, wl, workspace=ws, chunk_rows=2304)
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_OK
    for x, w, y in zip(xs, wl, outs):
        assert np.array_equal(bf16_bits(y), bf16_bits(lib.bi_gemm_bf16(x.cuda(), w))), x.shape[0]
    sampled_parity(oracle, xs[-1], Ws[13 % 2].cpu(), outs[-1], 4, 7, "host batch M=8192")
