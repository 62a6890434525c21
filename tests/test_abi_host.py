"""Host-side tests of the C ABI: the library loads, exports every entry point
declared in include/*.h, and its host-only logic (the pin table, validation,
the launch plan) behaves -- in particular the reduction tree never depends on M.
No GPU work is done here."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bd():
    from invariant_bi_gemm_bf16_gb300 import binding, build
    build.build()
    binding.load()
    return binding


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(bi_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("bi_gemm_bf16", "bi_rmsnorm_bf16", "bi_rmsnorm_gemm_bf16", "bi_pins_default",
                     "bi_pins_validate", "bi_status_string", "bi_last_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(bd):
    lib = ctypes.CDLL(bd.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, "not exported: %s" % missing
    assert set(declared_functions()) <= set(bd._SIGNATURES), "binding lacks a declared entry point"


def test_abi_version_and_status_strings(bd):
    lib = bd.load()
    assert lib.bi_abi_version() == bd.BI_PINS_ABI_VERSION
    for s in range(8):
        assert bd.status_string(s).startswith("BI_")
    assert bd.status_string(999) == "BI_ERR_UNKNOWN"


TABLE_SHAPES = [(128, 256), (4096, 14336), (6144, 4096), (28672, 4096), (10240, 8192), (8192, 8192),
                (57344, 8192), (8192, 28672)]


@pytest.mark.parametrize("N,K", TABLE_SHAPES + [(300, 200), (1000, 8), (64, 65536)])
def test_default_pins_are_legal(bd, N, K):
    p = bd.bi_pins_default(N, K)
    assert p.abi_version == 1 and p.bk == 64
    assert 1 <= p.split_k <= min(16, -(-K // 64))
    assert p.tok_tile in (64, 128, 256) and p.mma_ctas in (0, 1, 2)
    assert bd.bi_pins_validate(N, K, p) == bd.BI_OK


def test_pins_validation_refuses(bd):
    N, K = 4096, 14336
    good = bd.bi_pins_default(N, K)
    bad = [good.replace(abi_version=2), good.replace(bk=32), good.replace(split_k=0),
           good.replace(split_k=17), good.replace(tok_tile=96), good.replace(tok_tile=512),
           good.replace(stages=1), good.replace(stages=99), good.replace(flags=0x8000),
           good.replace(split_k=2, flags=bd.BI_FLAG_SCHEDULE_CHAIN), good.replace(split_k=9, flags=bd.BI_FLAG_SCHEDULE_CLUSTER),
           good.replace(mma_ctas=-1), good.replace(mma_ctas=4)]
    for p in bad:
        assert bd.bi_pins_validate(N, K, p) == bd.BI_ERR_ILLEGAL_PINS, p
    # more splits than K tiles
    assert bd.bi_pins_validate(128, 64, good.replace(split_k=2)) == bd.BI_ERR_ILLEGAL_PINS
    # bad shapes
    assert bd.bi_pins_validate(128, 100, good) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert bd.bi_pins_validate(0, 64, good) == bd.BI_ERR_INVALID_ARG


def test_null_and_bad_arguments_rejected_before_any_launch(bd):
    """These return before touching CUDA, so they run without a GPU."""
    lib = bd.load()
    p = bd.bi_pins_default(128, 256)
    # negative M, K not a multiple of 8, null pointers with M > 0
    assert lib.bi_gemm_bf16(None, None, None, -1, 128, 256, None, None) == bd.BI_ERR_INVALID_ARG
    assert lib.bi_gemm_bf16(None, None, None, 4, 128, 250, None, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_gemm_bf16(None, None, None, 4, 128, 256, None, None) == bd.BI_ERR_INVALID_ARG
    # misaligned pointers
    assert lib.bi_gemm_bf16(16, 18, 32, 4, 128, 256, None, None) == bd.BI_ERR_ALIGNMENT
    # illegal pins win over a launch
    assert lib.bi_gemm_bf16(16, 32, 48, 4, 128, 256, ctypes.byref(p.replace(tok_tile=7)), None) == \
        bd.BI_ERR_ILLEGAL_PINS
    # M == 0 is a no-op even with null pointers
    assert lib.bi_gemm_bf16(None, None, None, 0, 128, 256, None, None) == bd.BI_OK
    assert lib.bi_rmsnorm_bf16(None, None, None, 0, 256, 1e-5, None) == bd.BI_OK
    assert lib.bi_rmsnorm_bf16(None, None, None, 3, 256, 0.0, None) == bd.BI_ERR_INVALID_ARG
    assert lib.bi_rmsnorm_bf16(None, None, None, 3, 250, 1e-5, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_rmsnorm_bf16(16, 32, 40, 3, 256, 1e-5, None) == bd.BI_ERR_ALIGNMENT
    # fused: workspace checks
    assert lib.bi_rmsnorm_gemm_bf16(16, 32, 48, 64, 4, 128, 256, 1e-5, None, None, 0, None) == \
        bd.BI_ERR_WORKSPACE
    ws = bd.bi_rmsnorm_gemm_workspace_bytes(4, 256)
    assert ws >= 4 * 4 + 4 * 256 * 2 and ws % 256 == 0     # r, then room for the staged rows
    assert bd.bi_rmsnorm_gemm_workspace_bytes(1000, 4096) == 4096 + 1000 * 4096 * 2
    assert bd.bi_rmsnorm_gemm_workspace_bytes(0, 4096) == 0
    # the two forms of the fused layer cannot both be forced
    both = p.replace(flags=p.flags | bd.BI_FLAG_NORM_SMEM | bd.BI_FLAG_NORM_STAGED)
    assert lib.bi_pins_validate(128, 256, ctypes.byref(both)) == bd.BI_ERR_ILLEGAL_PINS
    for one in (bd.BI_FLAG_NORM_SMEM, bd.BI_FLAG_NORM_STAGED):
        assert lib.bi_pins_validate(128, 256, ctypes.byref(p.replace(flags=p.flags | one))) == bd.BI_OK
    assert lib.bi_rmsnorm_gemm_bf16(16, 32, 48, 64, 4, 128, 256, 1e-5, None, 256, ws - 1, None) == \
        bd.BI_ERR_WORKSPACE
    # the no-alloc capacity: one fp32 per row, refused before any CUDA call
    cap = lib.bi_noalloc_scratch_bytes()
    assert cap == 16 * 1024 * 1024
    assert lib.bi_rmsnorm_gemm_bf16_noalloc(16, 32, 48, 64, cap // 4 + 1, 128, 64, 1e-5, None, None) == \
        bd.BI_ERR_WORKSPACE
    # RMSNorm fused with the quantisation: H % 16 == 0 and at most 16384
    assert lib.bi_rmsnorm_quantize_e4m3(None, None, None, None, 0, 4096, 1e-5, None) == bd.BI_OK
    assert lib.bi_rmsnorm_quantize_e4m3(16, 32, 48, 64, 2, 4104, 1e-5, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_rmsnorm_quantize_e4m3(16, 32, 48, 64, 2, 16384 + 16, 1e-5, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_rmsnorm_quantize_e4m3(16, 32, 48, 64, 2, 4096, 0.0, None) == bd.BI_ERR_INVALID_ARG
    assert lib.bi_rmsnorm_quantize_e4m3(16, 32, 48, None, 2, 4096, 1e-5, None) == bd.BI_ERR_INVALID_ARG
    assert lib.bi_rmsnorm_quantize_e4m3(16, 32, 48, 66, 2, 4096, 1e-5, None) == bd.BI_ERR_ALIGNMENT
    assert lib.bi_rmsnorm_quantize_e4m3(16, 32, 40, 64, 2, 4096, 1e-5, None) == bd.BI_ERR_ALIGNMENT
    # GEMM on host buffers: argument, pin and workspace checks before any CUDA call
    assert lib.bi_gemm_bf16_host(None, None, None, 0, 128, 256, None, None, 0, None) == bd.BI_OK
    assert lib.bi_gemm_bf16_host(None, None, None, -1, 128, 256, None, None, 0, None) == bd.BI_ERR_INVALID_ARG
    assert lib.bi_gemm_bf16_host(None, None, None, 4, 128, 250, None, None, 0, None) == \
        bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_gemm_bf16_host(16, None, 48, 4, 128, 256, None, 256, 1 << 20, None) == bd.BI_ERR_INVALID_ARG
    assert lib.bi_gemm_bf16_host(16, 40, 48, 4, 128, 256, None, 256, 1 << 20, None) == bd.BI_ERR_ALIGNMENT
    assert lib.bi_gemm_bf16_host(16, 32, 48, 4, 128, 256, ctypes.byref(p.replace(tok_tile=7)), 256, 1 << 20,
                                 None) == bd.BI_ERR_ILLEGAL_PINS
    hws = bd.bi_gemm_bf16_host_workspace_bytes(4, 128, 256)
    assert lib.bi_gemm_bf16_host(16, 32, 48, 4, 128, 256, None, 256, hws - 1, None) == bd.BI_ERR_WORKSPACE
    assert lib.bi_gemm_bf16_host(16, 32, 48, 4, 128, 256, None, 512 + 16, hws, None) == bd.BI_ERR_ALIGNMENT
    # glue
    assert lib.bi_residual_add_bf16(16, 32, 48, 12, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_silu_mul_bf16(16, 32, 2, 12, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_attention_ctx1_bf16(16, 32, 2, 6, 4, 8, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    # FP8: K must give 16-byte rows of 1-byte codes; pins with bk = 128 and T = 256
    assert lib.bi_quantize_rows_e4m3(16, 32, 48, 2, 24, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_quantize_rows_e4m3(16, 32, 50, 2, 32, None) == bd.BI_ERR_ALIGNMENT
    assert lib.bi_gemm_fp8(16, 48, 32, 64, 80, 2, 128, 24, None, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_gemm_fp8(16, None, 32, 64, 80, 2, 128, 32, None, None) == bd.BI_ERR_INVALID_ARG
    p8 = bd.bi_pins_default_fp8(4096, 14336)
    assert p8.bk == 128 and p8.tok_tile == 256 and bd.bi_pins_validate_fp8(4096, 14336, p8) == bd.BI_OK
    assert bd.bi_pins_validate_fp8(4096, 14336, p8.replace(bk=64)) == bd.BI_ERR_ILLEGAL_PINS
    assert bd.bi_pins_validate_fp8(4096, 14336, p8.replace(tok_tile=128)) == bd.BI_ERR_ILLEGAL_PINS
    plan8 = bd.bi_gemm_plan_describe_fp8(8192, 4096, 14336)
    assert (plan8.bk, plan8.k_tiles, plan8.mma_k) == (128, 112, 32)
    # log-probabilities: V must be a multiple of 8; errors before any launch
    assert lib.bi_log_softmax_bf16(16, 32, 2, 12, None) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_log_softmax_bf16(16, 32, -1, 16, None) == bd.BI_ERR_INVALID_ARG
    assert lib.bi_log_softmax_bf16(None, 32, 2, 16, None) == bd.BI_ERR_INVALID_ARG
    assert lib.bi_log_softmax_bf16(8, 32, 2, 16, None) == bd.BI_ERR_ALIGNMENT
    assert lib.bi_log_softmax_bf16(0, 0, 0, 16, None) == bd.BI_OK        # M = 0: nothing to do
    assert lib.bi_token_logprobs_bf16(16, None, 32, 2, 16, None) == bd.BI_ERR_INVALID_ARG
    assert lib.bi_token_logprobs_bf16(16, 34, 32, 2, 16, None) == bd.BI_ERR_ALIGNMENT



def test_decode_attention_arguments_rejected_before_any_launch(bd):
    """Decode attention's host checks: shapes, the split-size pin, alignment
    and the workspace, all before anything touches CUDA."""
    lib = bd.load()

    def call(q=16, k=32, v=48, bt=64, bts=4, sl=80, out=96, B=2, Hq=8, Hkv=2, D=128, pages=10, P=16,
             max_len=64, split=0, scale=0.088, ws=112, ws_bytes=1 << 30):
        return lib.bi_decode_attention_bf16(q, k, v, bt, bts, sl, out, B, Hq, Hkv, D, pages, P, max_len, split,
                                            scale, ws, ws_bytes, None)
    assert call(D=64) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert call(Hq=6, Hkv=4) == bd.BI_ERR_UNSUPPORTED_SHAPE      # Hq % Hkv
    assert call(Hq=34, Hkv=2) == bd.BI_ERR_UNSUPPORTED_SHAPE     # 17 query heads per group
    assert call(P=12) == bd.BI_ERR_UNSUPPORTED_SHAPE             # not a power of two
    assert call(P=4) == bd.BI_ERR_UNSUPPORTED_SHAPE              # below 8
    assert call(split=100) == bd.BI_ERR_UNSUPPORTED_SHAPE        # not a multiple of 64
    assert call(split=8192) == bd.BI_ERR_UNSUPPORTED_SHAPE       # above BI_ATTN_MAX_SPLIT
    assert call(split=-64) == bd.BI_ERR_INVALID_ARG
    assert call(max_len=65, bts=4) == bd.BI_ERR_INVALID_ARG      # the block table is too short
    assert call(scale=float("nan")) == bd.BI_ERR_INVALID_ARG
    assert call(q=None) == bd.BI_ERR_INVALID_ARG
    assert call(q=18) == bd.BI_ERR_ALIGNMENT
    assert call(sl=82) == bd.BI_ERR_ALIGNMENT
    assert call(ws_bytes=100) == bd.BI_ERR_WORKSPACE
    assert call(B=0, q=None, k=None, v=None, bt=None, sl=None, out=None, ws=None) == bd.BI_OK
    # workspace: 256 + list (B * n_split * 4, to 256) + B * Hkv * n_split * (128 + 2) * GP * 4
    assert bd.bi_decode_attention_workspace_bytes(2, 8, 2, 1000, 256) == 256 + 256 + 2 * 2 * 4 * 130 * 8 * 4
    assert bd.bi_decode_attention_workspace_bytes(3, 32, 2, 64, 64) == 256 + 256 + 3 * 2 * 1 * 130 * 16 * 4
    assert bd.bi_decode_attention_workspace_bytes(1, 8, 8, 0, 0) == 256 + 256 + 1 * 8 * 1 * 130 * 8 * 4
    assert bd.bi_decode_attention_workspace_bytes(100, 8, 8, 4096, 64) == \
        256 + (100 * 64 * 4 + 255) // 256 * 256 + 100 * 8 * 64 * 130 * 8 * 4
    assert bd.bi_decode_attention_workspace_bytes(1, 8, 8, 1000, 0) == \
        bd.bi_decode_attention_workspace_bytes(1, 8, 8, 1000, bd.BI_ATTN_DEFAULT_SPLIT)

ALL_M = list(range(1, 300)) + [511, 512, 513, 1000, 1023, 1024, 2048, 4095, 4096, 8191, 8192]



def test_host_gemm_workspace_is_two_chunk_slots(bd):
    """Rows travel in chunks of about 16 MB of X (a multiple of 128 rows,
    128..8192); the workspace holds two slots of a chunk's X and Y, each
    rounded to 256 bytes, or one slot when one chunk holds every row."""
    def r256(b):
        return (b + 255) // 256 * 256

    def slot(R, N, K):
        return r256(R * K * 2) + r256(R * N * 2)
    assert bd.bi_gemm_bf16_host_workspace_bytes(0, 4096, 14336) == 0
    # down_proj: 16 MB / 28 KB per row = 585 rows -> 512-row chunks
    assert bd.bi_gemm_bf16_host_workspace_bytes(8192, 4096, 14336) == 2 * slot(512, 4096, 14336)
    assert bd.bi_gemm_bf16_host_workspace_bytes(512, 4096, 14336) == slot(512, 4096, 14336)
    assert bd.bi_gemm_bf16_host_workspace_bytes(3, 4096, 14336) == slot(3, 4096, 14336)
    # K = 4096: 2048-row chunks; tiny K: at most 8192 rows
    assert bd.bi_gemm_bf16_host_workspace_bytes(5000, 6144, 4096) == 2 * slot(2048, 6144, 4096)
    assert bd.bi_gemm_bf16_host_workspace_bytes(100000, 128, 256) == 2 * slot(8192, 128, 256)

def test_host_batch_workspace_follows_the_largest_job(bd):
    """A job list chunks every job with the row count of its largest job; the
    workspace is two slots of that chunk, or one when a single chunk holds
    every row of every job; one job sizes as bi_gemm_bf16_host."""
    def r256(b):
        return (b + 255) // 256 * 256

    def slot(R, N, K):
        return r256(R * K * 2) + r256(R * N * 2)
    N, K = 4096, 14336
    sweep = [1 << i for i in range(14)]
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes(sweep, N, K) == 2 * slot(512, N, K)
    assert bd.bi_gemm_bf16_host_slot_bytes(sweep, N, K) == slot(512, N, K)
    # 3 rows and 5 rows: one 5-row chunk each, two chunks in all
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes([3, 5], N, K) == 2 * slot(5, N, K)
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes([0, 7, 0], N, K) == slot(7, N, K)
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes([0, 0], N, K) == 0
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes([], N, K) == 0
    assert bd.bi_gemm_bf16_host_slot_bytes([0], N, K) == 0
    for M in (1, 300, 512, 513, 8192, 100000):
        assert bd.bi_gemm_bf16_host_batch_workspace_bytes([M], N, K) == \
            bd.bi_gemm_bf16_host_workspace_bytes(M, N, K)
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes([-1, 4], N, K) == 0
    # an explicit chunk: capped at the largest job; negative is refused (0)
    assert bd.bi_gemm_bf16_host_slot_bytes(sweep, N, K, 2304) == slot(2304, N, K)
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes(sweep, N, K, 2304) == 2 * slot(2304, N, K)
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes([3, 5], N, K, 1000) == 2 * slot(5, N, K)
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes([10], N, K, 1000) == slot(10, N, K)
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes([10], N, K, 3) == 2 * slot(3, N, K)
    assert bd.bi_gemm_bf16_host_batch_workspace_bytes([10], N, K, -1) == 0
    assert bd.bi_gemm_bf16_host_slot_bytes([10], N, K, 1 << 40) == 0


def test_host_batch_arguments_rejected_before_any_launch(bd):
    """Every argument of a job list is checked before anything is enqueued
    (so these calls need no GPU)."""
    lib = bd.load()
    J = bd.HostGemmJob

    def jobs(*rows):
        arr = (J * len(rows))()
        for j, (x, w, y, M) in enumerate(rows):
            arr[j].X_host, arr[j].W, arr[j].Y_host, arr[j].M = x, w, y, M
        return arr
    def call(arr, n, N, K, ws, ws_bytes, chunk_rows=0):
        return lib.bi_gemm_bf16_host_batch(arr, n, N, K, None, chunk_rows, ws, ws_bytes, None)
    assert call(None, 0, 128, 256, None, 0) == bd.BI_OK
    assert call(None, 1, 128, 256, None, 0) == bd.BI_ERR_INVALID_ARG
    assert call(None, -1, 128, 256, None, 0) == bd.BI_ERR_INVALID_ARG
    assert call(jobs((None, None, None, 0), (None, None, None, 0)), 2, 128, 256, None, 0) == bd.BI_OK
    assert call(jobs((16, 32, 48, 4), (None, None, None, -1)), 2, 128, 256, 256, 1 << 20) == \
        bd.BI_ERR_INVALID_ARG
    assert call(jobs((16, 32, 48, 4)), 1, 128, 250, 256, 1 << 20) == bd.BI_ERR_UNSUPPORTED_SHAPE
    assert call(jobs((16, 32, 48, 4)), 1, 128, 256, 256, 1 << 20, -1) == bd.BI_ERR_INVALID_ARG
    assert call(jobs((16, 32, 48, 4)), 1, 128, 256, 256, 1 << 20, 1 << 40) == bd.BI_ERR_UNSUPPORTED_SHAPE
    # the second job's null W or misaligned W is found before the first job runs
    assert call(jobs((16, 32, 48, 4), (16, None, 48, 4)), 2, 128, 256, 256, 1 << 20) == bd.BI_ERR_INVALID_ARG
    assert call(jobs((16, 32, 48, 4), (16, 40, 48, 4)), 2, 128, 256, 256, 1 << 20) == bd.BI_ERR_ALIGNMENT
    arr = jobs((16, 32, 48, 4), (16, 32, 48, 6))
    need = lib.bi_gemm_bf16_host_batch_workspace_bytes(arr, 2, 128, 256, 0)
    assert need == 2 * lib.bi_gemm_bf16_host_slot_bytes(arr, 2, 128, 256, 0)
    assert call(arr, 2, 128, 256, 256, need - 1) == bd.BI_ERR_WORKSPACE
    assert call(arr, 2, 128, 256, 512 + 16, need) == bd.BI_ERR_ALIGNMENT
    # 2-row chunks: five chunks, a larger slot count, a smaller slot
    need2 = lib.bi_gemm_bf16_host_batch_workspace_bytes(arr, 2, 128, 256, 2)
    assert need2 == 2 * lib.bi_gemm_bf16_host_slot_bytes(arr, 2, 128, 256, 2) and need2 < need
    assert call(arr, 2, 128, 256, 256, need2 - 1, 2) == bd.BI_ERR_WORKSPACE
    with pytest.raises(ValueError):
        bd.bi_gemm_bf16_host_batch([], [None])


def test_host_schedule_of_the_benchmark_sweep(bd):
    """The down_proj sweep as one list, 2304-row chunks: with a ring of two
    slots every job goes in whole chunks; with eight the last job's last rows
    go in halving chunks (multiples of 128, the last 256 whole), so that
    little is left after the last copy-in."""
    N, K = 4096, 14336
    sweep = [1 << i for i in range(14)]
    slot = bd.bi_gemm_bf16_host_slot_bytes(sweep, N, K, 2304)
    two = bd.bi_gemm_bf16_host_schedule(sweep, N, K, 2304)
    assert [c[3] for c in two if c[0] == 13] == [2304, 2304, 2304, 1280]
    assert [c[1] for c in two] == [i % 2 for i in range(len(two))]
    eight = bd.bi_gemm_bf16_host_schedule(sweep, N, K, 2304, 8 * slot)
    assert [c[3] for c in eight if c[0] == 13] == [2304, 2304, 1792, 896, 384, 256, 256]
    assert [c[3] for c in eight if c[0] == 12] == [2304, 1792]
    assert [c[1] for c in eight] == [i % 8 for i in range(len(eight))]
    # the default chunk (512 rows here) and three slots: the taper starts at 1024 rows left
    three = bd.bi_gemm_bf16_host_schedule([8192], N, K, 0, 3 * bd.bi_gemm_bf16_host_slot_bytes([8192], N, K))
    assert [c[3] for c in three][-4:] == [512, 512, 256, 256] and len(three) == 17
    assert bd.bi_gemm_bf16_host_schedule([0, 0], N, K) == []


def test_host_schedule_covers_every_row_once(bd):
    """On random lists: the chunks cover each job's rows once, in order, job
    after job; no chunk is above the chunk rows; the slots rotate through a
    ring of at most 8 slots and at most what the workspace holds; only the
    last job with rows is cut finer than the chunk rows, only with a ring of
    three slots or more, and then into multiples of 128 rows (its last piece
    aside)."""
    import numpy as np
    rng = np.random.default_rng(5)
    N, K = 1024, 4096
    for _ in range(300):
        ms = [int(rng.choice([0, rng.integers(1, 300), rng.integers(1, 6000)])) for _ in range(rng.integers(1, 7))]
        cr = int(rng.choice([0, 128, 300, 1000, 2304]))
        if sum(ms) == 0:
            assert bd.bi_gemm_bf16_host_schedule(ms, N, K, cr) == []
            continue
        slot = bd.bi_gemm_bf16_host_slot_bytes(ms, N, K, cr)
        ws = max(bd.bi_gemm_bf16_host_batch_workspace_bytes(ms, N, K, cr), int(rng.integers(1, 11)) * slot)
        sched = bd.bi_gemm_bf16_host_schedule(ms, N, K, cr, ws)
        if cr:
            assert max(c[3] for c in sched) <= min(cr, max(ms))
        pieces = {j: [] for j in range(len(ms))}
        prev = -1
        for j, _slot, r0, rows in sched:
            assert j >= prev and rows >= 1 and r0 == sum(pieces[j])
            prev = j
            pieces[j].append(rows)
        assert all(sum(pieces[j]) == M for j, M in enumerate(ms))
        slots = [c[1] for c in sched]
        depth = max(slots) + 1
        assert slots == [i % depth for i in range(len(sched))]
        assert depth <= min(8, ws // slot)
        last = max(j for j, M in enumerate(ms) if M > 0)
        for j, M in enumerate(ms):
            p = pieces[j]
            if M == 0:
                continue
            if j != last or depth < 3:
                # whole chunks of the chunk rows, the remainder last
                assert all(r == p[0] for r in p[:-1]) and p[-1] <= p[0], (ms, cr, j, p)
            else:
                assert all(r % 128 == 0 and r >= 128 for r in p[:-1] if r < p[0]), (ms, cr, p)


def test_host_schedule_arguments(bd):
    lib = bd.load()
    arr = bd._job_array([5, 9])
    n = ctypes.c_int64(0)
    call = lib.bi_gemm_bf16_host_schedule
    assert call(arr, 2, 128, 256, 0, 1 << 30, None, 0, None) == bd.BI_ERR_INVALID_ARG
    assert call(arr, 2, 128, 256, 0, 1 << 30, None, 1, ctypes.byref(n)) == bd.BI_ERR_INVALID_ARG
    assert call(arr, 2, 128, 256, 0, 1 << 30, None, -1, ctypes.byref(n)) == bd.BI_ERR_INVALID_ARG
    assert call(arr, 2, 128, 256, -1, 1 << 30, None, 0, ctypes.byref(n)) == bd.BI_ERR_INVALID_ARG
    assert call(arr, 2, 128, 250, 0, 1 << 30, None, 0, ctypes.byref(n)) == bd.BI_ERR_UNSUPPORTED_SHAPE
    need = lib.bi_gemm_bf16_host_batch_workspace_bytes(arr, 2, 128, 256, 0)
    assert call(arr, 2, 128, 256, 0, need - 1, None, 0, ctypes.byref(n)) == bd.BI_ERR_WORKSPACE
    assert call(arr, 2, 128, 256, 0, need, None, 0, ctypes.byref(n)) == bd.BI_OK and n.value == 2
    # fewer entries than chunks: the first ones are written, the count is whole
    out = (bd.HostChunk * 1)()
    assert call(arr, 2, 128, 256, 0, need, out, 1, ctypes.byref(n)) == bd.BI_OK and n.value == 2
    assert (out[0].job, out[0].slot, out[0].row0, out[0].rows) == (0, 0, 0, 5)


@pytest.mark.parametrize("N,K", TABLE_SHAPES + [(300, 200), (20000, 1000)])
def test_reduction_tree_never_depends_on_m(bd, N, K):
    """Detent Sec. 8.2: the batch reaches no GEMM selection point.  The plan's
    tree fields (K tile, split count and boundaries, MMA shape) are identical for
    every M, every SM count and every schedule; only the schedule fields move."""
    ref = None
    schedules = set()
    for M in ALL_M:
        for sm in (152, 148, 132, 7):
            plan = bd.bi_gemm_plan_describe(M, N, K, None, sm)
            if ref is None:
                ref = plan.tree()
            assert plan.tree() == ref, (M, sm)
            schedules.add(plan.schedule)
    pins = bd.bi_pins_default(N, K)
    for flags in (bd.BI_FLAG_SCHEDULE_LOCAL, bd.BI_FLAG_SCHEDULE_CLUSTER):
        if flags == bd.BI_FLAG_SCHEDULE_CLUSTER and pins.split_k > 8:
            continue
        for M in (1, 77, 8192):
            assert bd.bi_gemm_plan_describe(M, N, K, pins.replace(flags=flags)).tree() == ref


@pytest.mark.parametrize("N,K", TABLE_SHAPES)
@pytest.mark.parametrize("ctas", [1, 2])
def test_pinned_mma_layout_never_depends_on_m(bd, N, K, ctas):
    """With mma_ctas pinned, the MMA layout is fixed too (only the schedule moves)."""
    pins = bd.bi_pins_default(N, K).replace(mma_ctas=ctas)
    layouts = {bd.bi_gemm_plan_describe(M, N, K, pins, sm).layout() for M in ALL_M for sm in (152, 132)}
    assert len(layouts) == 1
    (T, c, mm, mn), = layouts
    assert c == ctas and mm == 128 * ctas and mn == T == pins.tok_tile


def test_open_grouping_follows_m(bd):
    """mma_ctas = 0 (the default): one CTA per MMA while the splits run as
    clusters or the token tile is short; CTA pairs with two-tile copies for
    persistent full-tile work."""
    assert bd.bi_pins_default(4096, 14336).mma_ctas == 0
    small = bd.bi_gemm_plan_describe(1, 4096, 14336)
    mid = bd.bi_gemm_plan_describe(512, 4096, 14336)
    big = bd.bi_gemm_plan_describe(8192, 4096, 14336)
    assert (small.mma_ctas, small.kps, small.schedule) == (1, 2, bd.BI_FLAG_SCHEDULE_CLUSTER)
    # M=512: 32 pair tiles, each a cluster of 2 pairs running 2 splits each (one wave)
    assert (mid.mma_ctas, mid.schedule, mid.units, mid.cluster_x) == (2, bd.BI_FLAG_SCHEDULE_CHAIN, 2, 4)
    assert mid.grid_x * mid.grid_y * mid.grid_z == 4 * 16 * 2
    assert (big.mma_ctas, big.kps, big.schedule, big.mma_m) == (2, 2, bd.BI_FLAG_SCHEDULE_LOCAL, 256)
    m256 = bd.bi_gemm_plan_describe(256, 4096, 14336)
    m1024 = bd.bi_gemm_plan_describe(1024, 4096, 14336)
    assert (m256.mma_ctas, m256.schedule) == (1, bd.BI_FLAG_SCHEDULE_CLUSTER)
    assert (m1024.mma_ctas, m1024.schedule) == (2, bd.BI_FLAG_SCHEDULE_LOCAL)
    assert small.tree() == mid.tree() == big.tree() == m256.tree() == m1024.tree()


@pytest.mark.parametrize("S", [3, 4, 5, 8])
@pytest.mark.parametrize("ctas", [1, 2])
def test_chain_schedule_plan(bd, S, ctas):
    """CHAIN: ceil(S/2) units per tile, each a CTA or a pair; the tree is unchanged."""
    pins = bd.bi_pins_default(4096, 14336).replace(split_k=S, mma_ctas=ctas, flags=bd.BI_FLAG_SCHEDULE_CHAIN)
    assert bd.bi_pins_validate(4096, 14336, pins) == bd.BI_OK
    plan = bd.bi_gemm_plan_describe(700, 4096, 14336, pins)
    u = (S + 1) // 2
    assert (plan.schedule, plan.units, plan.cluster_x, plan.grid_x) == (bd.BI_FLAG_SCHEDULE_CHAIN, u, u * ctas, u * ctas)
    assert plan.tree() == bd.bi_gemm_plan_describe(700, 4096, 14336, pins.replace(flags=0)).tree()


def test_split_boundaries_partition_k(bd):
    for N, K in TABLE_SHAPES:
        for S in range(1, 17):
            kt = -(-K // 64)
            if S > kt:
                continue
            p = bd.bi_pins_default(N, K).replace(split_k=S)
            plan = bd.bi_gemm_plan_describe(1, N, K, p)
            b = list(plan.split_begin[: S + 1])
            assert b[0] == 0 and b[-1] == kt
            assert all(b[i] < b[i + 1] for i in range(S))
            # boundaries are floor(s*KT/S): a fixed function of K and S
            assert b == [s * kt // S for s in range(S + 1)]


def test_plan_schedules(bd):
    # decode-sized down_proj runs as clusters of S CTAs; prefill-sized as persistent CTAs
    small = bd.bi_gemm_plan_describe(1, 4096, 14336)
    assert small.mma_ctas == 1 and small.mma_m == 128 and small.tok_tile == 64 and small.kps == 2
    assert small.schedule == bd.BI_FLAG_SCHEDULE_CLUSTER and small.cluster_x == small.split_k == 4
    assert small.grid_x * small.grid_y * small.grid_z == 32 * 4
    assert small.x_box_rows == 8 and small.w_stages > small.x_stages
    one = bd.bi_pins_default(4096, 14336).replace(mma_ctas=1)
    big = bd.bi_gemm_plan_describe(8192, 4096, 14336, one)
    assert big.schedule == bd.BI_FLAG_SCHEDULE_LOCAL and big.grid_x == 152 and big.cluster_x == 1
    assert big.x_box_rows == 256 and big.kps == 1
    pair = bd.bi_gemm_plan_describe(8192, 4096, 14336, one.replace(mma_ctas=2))
    assert pair.mma_m == 256 and pair.cluster_x == 2 and pair.grid_x == 152 and pair.x_box_rows == 128
    assert pair.kps == 2
    for plan in (small, big, pair):
        assert plan.smem_bytes <= 232448 and plan.block_threads == 32 * 19


def test_decode_plan_narrows_the_token_tile(bd):
    """A single short token tile on single-CTA MMAs, with the grouping and the
    W depth left open, runs at T = 64 (M <= 64) or 128 (M <= 128) with two K
    tiles per stage; the tree stays the pinned one."""
    for N, K in TABLE_SHAPES:
        ref = bd.bi_gemm_plan_describe(4096, N, K).tree()
        for M, T in ((1, 64), (8, 64), (33, 64), (64, 64), (65, 128), (128, 128)):
            plan = bd.bi_gemm_plan_describe(M, N, K)
            if plan.mma_ctas != 1:
                continue
            assert (plan.tok_tile, plan.mma_n, plan.kps, plan.m_tiles) == (T, T, 2, 1), (N, K, M)
            assert plan.x_stages >= 2 and plan.w_stages >= 4 and plan.smem_bytes <= 232448
            assert plan.tree() == ref
    pins = bd.bi_pins_default(4096, 14336)
    # pinned grouping, pinned W depth, or no two-tile flag: the pinned tile and one tile per stage
    for p in (pins.replace(mma_ctas=1), pins.replace(stages=4),
              pins.replace(flags=pins.flags & ~bd.BI_FLAG_KTILE_PAIRS)):
        plan = bd.bi_gemm_plan_describe(1, 4096, 14336, p)
        assert (plan.tok_tile, plan.kps) == (256, 1)
    # above 128 tokens the tile is the pinned one
    assert bd.bi_gemm_plan_describe(129, 4096, 14336).tok_tile == 256


def test_fp8_decode_plan_narrows_the_token_tile(bd):
    """The FP8 pins fix T = 256, but with the grouping left open a decode tile
    runs at T = 64 or 128 with two 128-value K tiles per stage; the tree (K
    tiles of 128 values, the splits) is the pinned one."""
    for N, K in ((4096, 14336), (6144, 4096)):
        ref = bd.bi_gemm_plan_describe_fp8(4096, N, K).tree()
        for M, T in ((1, 64), (64, 64), (65, 128), (128, 128)):
            plan = bd.bi_gemm_plan_describe_fp8(M, N, K)
            if plan.mma_ctas != 1:
                continue
            assert (plan.tok_tile, plan.kps, plan.bk) == (T, 2, 128), (N, K, M)
            assert plan.tree() == ref
        assert bd.bi_gemm_plan_describe_fp8(129, N, K).tok_tile == 256


def test_plan_ktile_pairs(bd):
    """Two K tiles per copy only with the flag, K % 64 == 0, T = 256 and full X boxes."""
    p = bd.bi_pins_default(4096, 14336).replace(mma_ctas=2, flags=bd.BI_FLAG_SCHEDULE_AUTO)
    pk = p.replace(flags=p.flags | bd.BI_FLAG_KTILE_PAIRS)
    big = bd.bi_gemm_plan_describe(8192, 4096, 14336, pk)
    assert big.kps == 2 and big.smem_bytes <= 232448
    assert bd.bi_gemm_plan_describe(8192, 4096, 14336, p).kps == 1
    assert big.tree() == bd.bi_gemm_plan_describe(8192, 4096, 14336, p).tree()
    assert bd.bi_gemm_plan_describe(8192, 4096, 14336, pk.replace(mma_ctas=1)).kps == 1  # one CTA
    assert bd.bi_gemm_plan_describe(1, 4096, 14336, pk).kps == 1          # short X box
    assert bd.bi_gemm_plan_describe(8192, 4096, 14336, pk.replace(tok_tile=128)).kps == 1
    q = bd.bi_pins_default(256, 200).replace(mma_ctas=2)
    assert bd.bi_gemm_plan_describe(512, 256, 200, q.replace(flags=q.flags | bd.BI_FLAG_KTILE_PAIRS)).kps == 1
    # a W depth legal with one-tile stages may be too deep for two-tile stages
    deep = p.replace(stages=6)
    assert bd.bi_pins_validate(4096, 14336, deep) == bd.BI_OK
    assert bd.bi_pins_validate(4096, 14336, deep.replace(flags=bd.BI_FLAG_KTILE_PAIRS)) == bd.BI_ERR_ILLEGAL_PINS


def test_global_schedule_plans_and_workspace_sizes(bd):
    """The fold workspace a GLOBAL plan needs (host only): the per-tile
    counters rounded up to 256 bytes, then one T x 128 fp32 partial per chain;
    nothing for plans the schedule does not apply to."""
    lib = bd.load()
    p = bd.bi_pins_default(6144, 4096).replace(split_k=3)
    pg = p.replace(flags=p.flags | bd.BI_FLAG_SCHEDULE_GLOBAL)
    need = bd.bi_gemm_bf16_workspace_bytes(32, 6144, 4096, pg)
    assert need == 256 + 48 * 3 * 64 * 128 * 4
    plan = bd.bi_gemm_plan_describe_ws(32, 6144, 4096, pg, 152, need)
    assert plan.schedule == bd.BI_FLAG_SCHEDULE_GLOBAL and plan.grid_x == 144 and plan.cluster_x == 1
    # the same tree as the other schedules
    other = bd.bi_gemm_plan_describe(32, 6144, 4096, p.replace(flags=p.flags | bd.BI_FLAG_SCHEDULE_LOCAL), 152)
    assert plan.tree() == other.tree()
    # too little workspace, several token tiles, paired MMAs, S = 1 or S > 8: no GLOBAL
    assert bd.bi_gemm_plan_describe_ws(32, 6144, 4096, pg, 152, need - 1).schedule != bd.BI_FLAG_SCHEDULE_GLOBAL
    assert bd.bi_gemm_bf16_workspace_bytes(300, 6144, 4096, pg) == 0
    assert bd.bi_gemm_bf16_workspace_bytes(32, 6144, 4096, pg.replace(mma_ctas=2)) == 0
    # a pinned single-CTA grouping keeps the pinned 256-token tile: larger partials
    assert bd.bi_gemm_bf16_workspace_bytes(32, 6144, 4096, pg.replace(mma_ctas=1)) == 256 + 48 * 3 * 256 * 128 * 4
    assert bd.bi_gemm_bf16_workspace_bytes(32, 6144, 4096, pg.replace(split_k=1)) == 0
    assert bd.bi_gemm_bf16_workspace_bytes(32, 6144, 4096, pg.replace(split_k=9)) == 0
    assert bd.bi_gemm_bf16_workspace_bytes(32, 6144, 4096, pg.replace(split_k=8)) == 256 + 48 * 8 * 64 * 128 * 4
    # schedule values past GLOBAL are illegal
    for sched in (5, 6, 7):
        assert lib.bi_pins_validate(6144, 4096, ctypes.byref(p.replace(flags=(p.flags & ~0x7) | sched))) == \
            bd.BI_ERR_ILLEGAL_PINS
    # the workspace entry point checks its alignment before anything else touches the GPU
    assert lib.bi_gemm_bf16_ws(16, 32, 48, 4, 6144, 4096, None, 264, 1 << 20, None) == bd.BI_ERR_ALIGNMENT
