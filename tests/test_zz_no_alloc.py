"""The fused layer for callers that cannot allocate device memory.

bi_rmsnorm_gemm_bf16_noalloc serves callers with no allocator of their own
(for instance a plugin inside a host runtime that has reserved all device
memory up front, or a latency-critical path where cudaMalloc/cudaFree would
synchronise the device).  It keeps each row's RMSNorm scale in the library's
static device array instead of a caller workspace.  Its output must match the
workspace entry point bi_rmsnorm_gemm_bf16 on two calls in a row (the array
keeps the previous call's contents), and an oversized call must be refused
without launching anything.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from helpers import EPS, bf16_bits, bits_to_f64, check_gemm_parity
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


def _problem(M, N, K, seed):
    X = inputs.normal((M, K), seed=seed, stream=0).cuda()
    g = inputs.normal((K,), std=0.1, mean=1.0, seed=seed, stream=2).cuda()
    W = inputs.normal((N, K), std=0.02, seed=seed, stream=1).cuda()
    return X, g, W


def test_noalloc_matches_workspace_entry_point_twice(lib):
    # in shared memory; staged in the array (the second call reuses it); and a
    # batch whose staged rows would not fit the array, normalised in shared
    # memory instead
    cases = [(37, 640, 4096, 1), (300, 384, 1024, 2), (2100, 256, 4096, 3)]
    for M, N, K, seed in cases:
        X, g, W = _problem(M, N, K, seed)
        want = lib.bi_rmsnorm_gemm_bf16(X, g, W, EPS)
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        lib.bi_rmsnorm_gemm_bf16_noalloc(X, g, W, out, EPS)
        torch.cuda.synchronize()
        assert lib.bi_last_device_status() == lib.BI_OK
        # within the GEMM tolerance the other tests use (reference: the workspace call)
        check_gemm_parity(bf16_bits(out), bits_to_f64(bf16_bits(want)).astype(np.float32), K, "noalloc")
        # and in fact the same kernels give the same bits
        assert torch.equal(out.view(torch.int16), want.view(torch.int16))


def test_noalloc_allocates_nothing_and_refuses_oversize(lib):
    M, N, K = 64, 256, 2048
    X, g, W = _problem(M, N, K, 3)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    lib.bi_rmsnorm_gemm_bf16_noalloc(X, g, W, out, EPS)      # first call on this device: set-up
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    lib.bi_rmsnorm_gemm_bf16_noalloc(X, g, W, out, EPS)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    # one fp32 value per row: M * 4 above the static capacity is refused, output untouched
    Kb, Nb = 8, 8
    Mb = lib.bi_noalloc_scratch_bytes() // 4 + 1
    xb = torch.zeros((Mb, Kb), dtype=torch.bfloat16, device="cuda")
    gb = torch.ones(Kb, dtype=torch.bfloat16, device="cuda")
    wb = torch.zeros((Nb, Kb), dtype=torch.bfloat16, device="cuda")
    ob = torch.full((Mb, Nb), 5.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.BiError) as e:
        lib.bi_rmsnorm_gemm_bf16_noalloc(xb, gb, wb, ob, EPS)
    assert e.value.status == lib.BI_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(ob.float() == 5.0)
