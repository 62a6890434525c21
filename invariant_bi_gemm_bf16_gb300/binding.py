"""Thin Python binding of the C ABI in ``include/bi_gemm.h``.

Argument marshalling only: every function checks the tensors it is handed,
passes their device pointers, sizes and the current CUDA stream to the entry
point of the same name in ``libbi_gemm.so``, and raises ``BiError`` on a
non-OK status.  All arithmetic runs in the library's kernels.  There is no
fallback: if the library is missing or cannot be loaded, every call raises.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbi_gemm.so")
LIB_DEBUG_PATH = os.path.join(_PKG, "libbi_gemm_debug.so")  # the debug-bounds build

BI_OK = 0
BI_ERR_INVALID_ARG = 1
BI_ERR_ALIGNMENT = 2
BI_ERR_UNSUPPORTED_SHAPE = 3
BI_ERR_ILLEGAL_PINS = 4
BI_ERR_CUDA = 5
BI_ERR_DEVICE_TIMEOUT = 6
BI_ERR_WORKSPACE = 7
BI_ERR_DEBUG_BOUNDS = 8

BI_PINS_ABI_VERSION = 1
BI_BK = 64
BI_TILE_N = 128
BI_MAX_SPLIT_K = 16
BI_FLAG_SCHEDULE_AUTO = 0x0
BI_FLAG_SCHEDULE_LOCAL = 0x1
BI_FLAG_SCHEDULE_CLUSTER = 0x2
BI_FLAG_SCHEDULE_CHAIN = 0x3
BI_FLAG_SCHEDULE_GLOBAL = 0x4
BI_GLOBAL_MAX_SPLIT_K = 8
BI_FLAG_DEBUG_STALL_PRODUCER = 0x100
BI_FLAG_PREFETCH_W = 0x200
BI_FLAG_KTILE_PAIRS = 0x400
BI_FLAG_NORM_SMEM = 0x800
BI_FLAG_NORM_STAGED = 0x1000


class Pins(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_int32), ("bk", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("tok_tile", ctypes.c_int32), ("mma_ctas", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}

    def replace(self, **kw) -> "Pins":
        d = self.as_dict()
        d.update(kw)
        return Pins(**d)

    def __repr__(self):
        return "Pins(%s)" % ", ".join("%s=%s" % kv for kv in self.as_dict().items())


class Plan(ctypes.Structure):
    _fields_ = [("bk", ctypes.c_int32), ("split_k", ctypes.c_int32), ("tok_tile", ctypes.c_int32),
                ("mma_ctas", ctypes.c_int32), ("mma_m", ctypes.c_int32), ("mma_n", ctypes.c_int32),
                ("mma_k", ctypes.c_int32),
                ("k_tiles", ctypes.c_int64),
                ("split_begin", ctypes.c_int64 * (BI_MAX_SPLIT_K + 1)),
                ("schedule", ctypes.c_int32), ("units", ctypes.c_int32),
                ("w_stages", ctypes.c_int32), ("x_stages", ctypes.c_int32),
                ("x_box_rows", ctypes.c_int32), ("kps", ctypes.c_int32),
                ("n_tiles", ctypes.c_int64), ("m_tiles", ctypes.c_int64), ("group_n", ctypes.c_int32),
                ("grid_x", ctypes.c_int32), ("grid_y", ctypes.c_int32), ("grid_z", ctypes.c_int32),
                ("cluster_x", ctypes.c_int32), ("block_threads", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int64)]

    TREE_FIELDS = ("bk", "split_k", "mma_k", "k_tiles")
    LAYOUT_FIELDS = ("tok_tile", "mma_ctas", "mma_m", "mma_n")

    def tree(self) -> tuple:
        """The reduction-tree fields: a function of (N, K, pins) only."""
        return tuple(getattr(self, f) for f in self.TREE_FIELDS) + \
            tuple(self.split_begin[: self.split_k + 1])

    def layout(self) -> tuple:
        """The MMA layout: fixed by pins that fix mma_ctas, else chosen per
        launch; it changes no output bit."""
        return tuple(getattr(self, f) for f in self.LAYOUT_FIELDS)


class HostGemmJob(ctypes.Structure):
    """bi_host_gemm_job: one GEMM of bi_gemm_bf16_host_batch."""
    _fields_ = [("X_host", ctypes.c_void_p), ("W", ctypes.c_void_p), ("Y_host", ctypes.c_void_p),
                ("M", ctypes.c_int64)]


class HostChunk(ctypes.Structure):
    """bi_host_chunk: one chunk of bi_gemm_bf16_host_batch's schedule."""
    _fields_ = [("job", ctypes.c_int32), ("slot", ctypes.c_int32), ("row0", ctypes.c_int64),
                ("rows", ctypes.c_int64)]


class BiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64

# name -> (restype, argtypes); the C ABI of include/bi_gemm.h
_SIGNATURES = {
    "bi_abi_version": (ctypes.c_int32, []),
    "bi_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "bi_pins_default": (ctypes.c_int, [_i64, _i64, ctypes.POINTER(Pins)]),
    "bi_pins_validate": (ctypes.c_int, [_i64, _i64, ctypes.POINTER(Pins)]),
    "bi_gemm_plan_describe": (ctypes.c_int, [_i64, _i64, _i64, ctypes.POINTER(Pins), ctypes.c_int32,
                                             ctypes.POINTER(Plan)]),
    "bi_gemm_bf16": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.POINTER(Pins), _vp]),
    "bi_gemm_bf16_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64, ctypes.POINTER(Pins)]),
    "bi_gemm_bf16_ws": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.POINTER(Pins), _vp, ctypes.c_size_t,
                                       _vp]),
    "bi_gemm_plan_describe_ws": (ctypes.c_int, [_i64, _i64, _i64, ctypes.POINTER(Pins), ctypes.c_int32,
                                                ctypes.c_size_t, ctypes.POINTER(Plan)]),
    "bi_rmsnorm_bf16": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, ctypes.c_float, _vp]),
    "bi_rmsnorm_quantize_e4m3": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_float, _vp]),
    "bi_gemm_bf16_host_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64]),
    "bi_gemm_bf16_host": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.POINTER(Pins), _vp,
                                         ctypes.c_size_t, _vp]),
    "bi_gemm_bf16_host_batch_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(HostGemmJob), ctypes.c_int32,
                                                                  _i64, _i64, _i64]),
    "bi_gemm_bf16_host_slot_bytes": (ctypes.c_size_t, [ctypes.POINTER(HostGemmJob), ctypes.c_int32, _i64, _i64,
                                                       _i64]),
    "bi_gemm_bf16_host_batch": (ctypes.c_int, [ctypes.POINTER(HostGemmJob), ctypes.c_int32, _i64, _i64,
                                               ctypes.POINTER(Pins), _i64, _vp, ctypes.c_size_t, _vp]),
    "bi_gemm_bf16_host_schedule": (ctypes.c_int, [ctypes.POINTER(HostGemmJob), ctypes.c_int32, _i64, _i64, _i64,
                                                  ctypes.c_size_t, ctypes.POINTER(HostChunk), _i64,
                                                  ctypes.POINTER(_i64)]),
    "bi_rmsnorm_gemm_workspace_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "bi_rmsnorm_gemm_bf16": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_float,
                                            ctypes.POINTER(Pins), _vp, ctypes.c_size_t, _vp]),
    "bi_rmsnorm_gemm_bf16_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_float,
                                                    ctypes.POINTER(Pins), _vp]),
    "bi_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "bi_residual_add_bf16": (ctypes.c_int, [_vp, _vp, _vp, _i64, _vp]),
    "bi_silu_mul_bf16": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp]),
    "bi_attention_ctx1_bf16": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i64, _i64, _vp]),
    "bi_last_device_status": (ctypes.c_int, [_vp]),
    "bi_debug_bounds_enabled": (ctypes.c_int32, []),
    "bi_debug_bounds_detail": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint64), _vp]),
    "bi_log_softmax_bf16": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp]),
    "bi_quantize_rows_e4m3": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _vp]),
    "bi_pins_default_fp8": (ctypes.c_int, [_i64, _i64, ctypes.POINTER(Pins)]),
    "bi_pins_validate_fp8": (ctypes.c_int, [_i64, _i64, ctypes.POINTER(Pins)]),
    "bi_gemm_plan_describe_fp8": (ctypes.c_int, [_i64, _i64, _i64, ctypes.POINTER(Pins), ctypes.c_int32,
                                                 ctypes.POINTER(Plan)]),
    "bi_gemm_fp8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.POINTER(Pins), _vp]),
    "bi_token_logprobs_bf16": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _vp]),
    "bi_decode_attention_workspace_bytes": (ctypes.c_int, [_i64, _i64, _i64, _i64, _i64,
                                                           ctypes.POINTER(ctypes.c_size_t)]),
    "bi_decode_attention_bf16": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _vp, _vp, _i64, _i64, _i64, _i64,
                                                _i64, _i64, _i64, _i64, ctypes.c_float, _vp, ctypes.c_size_t,
                                                _vp]),
}


def load(path: str | None = None):
    """Loads libbi_gemm.so (built by ``__graft_entry__.build()``), or the
    library named by the BI_GEMM_LIB environment variable (the debug-bounds
    variant, for one); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or os.environ.get("BI_GEMM_LIB") or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError("libbi_gemm.so is not built (%s); run __graft_entry__.build()" % p)
            lib = ctypes.CDLL(p)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().bi_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != BI_OK:
        raise BiError(status, where)


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if isinstance(stream, torch.cuda.Stream) else int(stream)


def _on_current_device(t: torch.Tensor, name: str):
    # the library runs on the current device and reads every pointer there
    if t.device.index != torch.cuda.current_device():
        raise ValueError("%s is on %s, but the current CUDA device is cuda:%d" %
                         (name, t.device, torch.cuda.current_device()))


def _dev(t: torch.Tensor, name: str, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError("%s must be a contiguous bf16 CUDA tensor" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    _on_current_device(t, name)
    return t.data_ptr()


# ---------------------------------------------------------------------------
# pins and plans (host only)
# ---------------------------------------------------------------------------

def bi_pins_default(N: int, K: int) -> Pins:
    p = Pins()
    _check(load().bi_pins_default(N, K, ctypes.byref(p)), "bi_pins_default")
    return p


def bi_pins_validate(N: int, K: int, pins: Pins) -> int:
    return load().bi_pins_validate(N, K, ctypes.byref(pins))


def bi_gemm_plan_describe(M: int, N: int, K: int, pins: Pins | None = None, sm_count: int = 0) -> Plan:
    plan = Plan()
    _check(load().bi_gemm_plan_describe(M, N, K, ctypes.byref(pins) if pins is not None else None,
                                        sm_count, ctypes.byref(plan)), "bi_gemm_plan_describe")
    return plan


# ---------------------------------------------------------------------------
# the layer
# ---------------------------------------------------------------------------

# Observers of GEMM calls, fn(M, N, K): the pin tuner's workload recorder.
# They only count calls; nothing is computed here.
_call_hooks: list = []


def add_call_hook(fn):
    _call_hooks.append(fn)


def remove_call_hook(fn):
    _call_hooks.remove(fn)


def _report(M: int, N: int, K: int):
    for fn in list(_call_hooks):
        fn(M, N, K)


def _workspace(ws: torch.Tensor, name: str = "workspace") -> tuple:
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % name)
    _on_current_device(ws, name)
    return ws.data_ptr(), ws.numel() * ws.element_size()


def bi_gemm_plan_describe_ws(M: int, N: int, K: int, pins: Pins | None = None, sm_count: int = 0,
                             workspace_bytes: int = 0) -> Plan:
    plan = Plan()
    _check(load().bi_gemm_plan_describe_ws(M, N, K, ctypes.byref(pins) if pins is not None else None, sm_count,
                                           int(workspace_bytes), ctypes.byref(plan)), "bi_gemm_plan_describe_ws")
    return plan


def bi_gemm_bf16_workspace_bytes(M: int, N: int, K: int, pins: Pins | None = None) -> int:
    """Fold-workspace bytes the call can use (0: the GLOBAL schedule does not apply)."""
    return int(load().bi_gemm_bf16_workspace_bytes(M, N, K, ctypes.byref(pins) if pins is not None else None))


def bi_gemm_bf16(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None,
                 pins: Pins | None = None, stream=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Y = X . W^T (bf16, fp32 accumulation).  x [M,K], w [N,K] -> [M,N].
    With `workspace` (device memory whose counter part is zero, see
    bi_gemm_bf16_workspace_bytes) the call goes through bi_gemm_bf16_ws."""
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("expected x [M,K] and w [N,K]")
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if workspace is not None:
        ws_ptr, ws_bytes = _workspace(workspace)
        st = load().bi_gemm_bf16_ws(_dev(x, "x"), _dev(w, "w"), _dev(out, "out", (M, N)), M, N, K,
                                    ctypes.byref(pins) if pins is not None else None, ws_ptr, ws_bytes,
                                    _stream(stream))
        _check(st, "bi_gemm_bf16_ws")
    else:
        st = load().bi_gemm_bf16(_dev(x, "x"), _dev(w, "w"), _dev(out, "out", (M, N)), M, N, K,
                                 ctypes.byref(pins) if pins is not None else None, _stream(stream))
        _check(st, "bi_gemm_bf16")
    if _call_hooks:
        _report(M, N, K)
    return out


def _host(t: torch.Tensor, name: str, shape) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError("%s must be a contiguous bf16 host tensor" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    return t.data_ptr()


def bi_gemm_bf16_host_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().bi_gemm_bf16_host_workspace_bytes(M, N, K))


def bi_gemm_bf16_host(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None,
                      pins: Pins | None = None, workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """Y = X . W^T with x [M,K] and the result [M,N] in host memory (page-locked
    for overlapped copies) and w [N,K] on the device.  Asynchronous on
    `stream`: synchronize it before reading the result."""
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("expected x [M,K] and w [N,K]")
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True)
    need = bi_gemm_bf16_host_workspace_bytes(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=w.device)
    ws_ptr, ws_bytes = _workspace(workspace)
    st = load().bi_gemm_bf16_host(_host(x, "x", (M, K)), _dev(w, "w"), _host(out, "out", (M, N)), M, N, K,
                                  ctypes.byref(pins) if pins is not None else None, ws_ptr, ws_bytes,
                                  _stream(stream))
    _check(st, "bi_gemm_bf16_host")
    if _call_hooks:
        _report(M, N, K)
    return out


def _job_array(ms, xs=None, ws=None, outs=None):
    arr = (HostGemmJob * max(len(ms), 1))()
    for j, M in enumerate(ms):
        arr[j].M = int(M)
        if xs is not None:
            arr[j].X_host, arr[j].W, arr[j].Y_host = xs[j], ws[j], outs[j]
    return arr


def bi_gemm_bf16_host_batch_workspace_bytes(ms, N: int, K: int, chunk_rows: int = 0) -> int:
    """Workspace of bi_gemm_bf16_host_batch for jobs of ms[j] rows (a ring of
    two slots)."""
    return int(load().bi_gemm_bf16_host_batch_workspace_bytes(_job_array(ms), len(ms), N, K, chunk_rows))


def bi_gemm_bf16_host_slot_bytes(ms, N: int, K: int, chunk_rows: int = 0) -> int:
    """Bytes of one ring slot for jobs of ms[j] rows; d slots give a ring of
    depth d (at most 8)."""
    return int(load().bi_gemm_bf16_host_slot_bytes(_job_array(ms), len(ms), N, K, chunk_rows))


def bi_gemm_bf16_host_schedule(ms, N: int, K: int, chunk_rows: int = 0, workspace_bytes: int | None = None) -> list:
    """The chunks bi_gemm_bf16_host_batch would run for jobs of ms[j] rows, as
    (job, slot, row0, rows) tuples in order; workspace_bytes (the size of the
    workspace, which sets the ring depth) defaults to the workspace query's."""
    if workspace_bytes is None:
        workspace_bytes = bi_gemm_bf16_host_batch_workspace_bytes(ms, N, K, chunk_rows)
    arr = _job_array(ms)
    n = _i64(0)
    _check(load().bi_gemm_bf16_host_schedule(arr, len(ms), N, K, chunk_rows, int(workspace_bytes), None, 0,
                                             ctypes.byref(n)), "bi_gemm_bf16_host_schedule")
    out = (HostChunk * max(n.value, 1))()
    _check(load().bi_gemm_bf16_host_schedule(arr, len(ms), N, K, chunk_rows, int(workspace_bytes), out, n.value,
                                             ctypes.byref(n)), "bi_gemm_bf16_host_schedule")
    return [(c.job, c.slot, c.row0, c.rows) for c in out[:n.value]]


def bi_gemm_bf16_host_batch(xs, ws, outs=None, pins: Pins | None = None, workspace: torch.Tensor | None = None,
                            stream=None, chunk_rows: int = 0) -> list:
    """outs[j] = xs[j] . ws[j]^T for a list of jobs of one shape (N, K): x [M_j,K]
    and the results [M_j,N] in host memory, w [N,K] on the device (the jobs may
    share one).  One pipeline of chunks over all jobs (chunk_rows rows each, 0
    for the default of about 16 MB of X); each job gets the bits bi_gemm_bf16
    gives it alone.  Asynchronous on `stream`."""
    if len(xs) != len(ws) or (outs is not None and len(outs) != len(xs)):
        raise ValueError("xs, ws and outs must have one entry per job")
    if not xs:
        return []
    N, K = ws[0].shape
    ms = []
    for x, w in zip(xs, ws):
        if x.dim() != 2 or w.dim() != 2 or tuple(w.shape) != (N, K) or x.shape[1] != K:
            raise ValueError("expected x [M,K] and w [N,K] of one (N, K) for every job")
        ms.append(int(x.shape[0]))
    if outs is None:
        outs = [torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True) for M in ms]
    arr = _job_array(ms, [_host(x, "x", (M, K)) for x, M in zip(xs, ms)], [_dev(w, "w") for w in ws],
                     [_host(o, "out", (M, N)) for o, M in zip(outs, ms)])
    need = int(load().bi_gemm_bf16_host_batch_workspace_bytes(arr, len(ms), N, K, chunk_rows))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=ws[0].device)
    ws_ptr, ws_bytes = _workspace(workspace)
    st = load().bi_gemm_bf16_host_batch(arr, len(ms), N, K, ctypes.byref(pins) if pins is not None else None,
                                        chunk_rows, ws_ptr, ws_bytes, _stream(stream))
    _check(st, "bi_gemm_bf16_host_batch")
    if _call_hooks:
        for M in ms:
            _report(M, N, K)
    return outs


def bi_rmsnorm_bf16(x: torch.Tensor, g: torch.Tensor, eps: float = 1e-5, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """RMSNorm over the last dimension of x [M,H] with gain g [H]."""
    if x.dim() != 2:
        raise ValueError("expected x [M,H]")
    M, H = x.shape
    if out is None:
        out = torch.empty_like(x)
    st = load().bi_rmsnorm_bf16(_dev(x, "x"), _dev(g, "g", (H,)), _dev(out, "out", (M, H)), M, H,
                                float(eps), _stream(stream))
    _check(st, "bi_rmsnorm_bf16")
    return out


def bi_rmsnorm_gemm_workspace_bytes(M: int, K: int) -> int:
    return int(load().bi_rmsnorm_gemm_workspace_bytes(M, K))


def bi_rmsnorm_gemm_bf16(x: torch.Tensor, g: torch.Tensor, w: torch.Tensor, eps: float = 1e-5,
                         pins: Pins | None = None, out: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = RMSNorm(x; g) . W^T, equal bit for bit to the two calls in sequence."""
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("expected x [M,K] and w [N,K]")
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    need = bi_rmsnorm_gemm_workspace_bytes(M, K)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    ws_ptr, ws_bytes = _workspace(workspace)
    st = load().bi_rmsnorm_gemm_bf16(_dev(x, "x"), _dev(g, "g", (K,)), _dev(w, "w"),
                                     _dev(out, "out", (M, N)), M, N, K, float(eps),
                                     ctypes.byref(pins) if pins is not None else None,
                                     ws_ptr, ws_bytes, _stream(stream))
    _check(st, "bi_rmsnorm_gemm_bf16")
    if _call_hooks:
        _report(M, N, K)
    return out


def bi_noalloc_scratch_bytes() -> int:
    """Capacity of the library's static scratch array (BI_NOALLOC_SCRATCH_BYTES
    as compiled into the library)."""
    return int(load().bi_noalloc_scratch_bytes())


def bi_rmsnorm_gemm_bf16_noalloc(x: torch.Tensor, g: torch.Tensor, w: torch.Tensor, out: torch.Tensor,
                                 eps: float = 1e-5, pins: Pins | None = None, stream=None) -> torch.Tensor:
    """The fused layer for callers that cannot allocate device memory: the
    caller passes the output, and each row's RMSNorm scale (and the staged
    normalised rows, where they fit) is kept in the library's static device
    array (M * 4 <= bi_noalloc_scratch_bytes()).  Calls that overlap on the
    GPU race on that array."""
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("expected x [M,K] and w [N,K]")
    M, K = x.shape
    N = w.shape[0]
    st = load().bi_rmsnorm_gemm_bf16_noalloc(_dev(x, "x"), _dev(g, "g", (K,)), _dev(w, "w"),
                                             _dev(out, "out", (M, N)), M, N, K, float(eps),
                                             ctypes.byref(pins) if pins is not None else None,
                                             _stream(stream))
    _check(st, "bi_rmsnorm_gemm_bf16_noalloc")
    if _call_hooks:
        _report(M, N, K)
    return out


def bi_residual_add_bf16(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    if a.shape != b.shape:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty_like(a)
    st = load().bi_residual_add_bf16(_dev(a, "a"), _dev(b, "b"), _dev(out, "out", a.shape), a.numel(),
                                     _stream(stream))
    _check(st, "bi_residual_add_bf16")
    return out


def _dev_as(t: torch.Tensor, name: str, dtype, shape) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be a contiguous %s CUDA tensor" % (name, dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    _on_current_device(t, name)
    return t.data_ptr()


def bi_quantize_rows_e4m3(x: torch.Tensor, q: torch.Tensor | None = None, scale: torch.Tensor | None = None,
                          stream=None):
    """Per-row E4M3 codes (uint8 [M,K]) and scales (fp32 [M]) of x [M,K] bf16."""
    if x.dim() != 2:
        raise ValueError("expected x [M,K]")
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(M, dtype=torch.float32, device=x.device)
    st = load().bi_quantize_rows_e4m3(_dev(x, "x"), _dev_as(q, "q", torch.uint8, (M, K)),
                                      _dev_as(scale, "scale", torch.float32, (M,)), M, K, _stream(stream))
    _check(st, "bi_quantize_rows_e4m3")
    return q, scale


def bi_rmsnorm_quantize_e4m3(x: torch.Tensor, g: torch.Tensor, eps: float = 1e-5, q: torch.Tensor | None = None,
                             scale: torch.Tensor | None = None, stream=None):
    """E4M3 codes (uint8 [M,H]) and per-row scales (fp32 [M]) of RMSNorm(x; g),
    bit for bit those of bi_quantize_rows_e4m3(bi_rmsnorm_bf16(x, g, eps))."""
    if x.dim() != 2:
        raise ValueError("expected x [M,H]")
    M, H = x.shape
    if q is None:
        q = torch.empty((M, H), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(M, dtype=torch.float32, device=x.device)
    st = load().bi_rmsnorm_quantize_e4m3(_dev(x, "x"), _dev(g, "g", (H,)), _dev_as(q, "q", torch.uint8, (M, H)),
                                         _dev_as(scale, "scale", torch.float32, (M,)), M, H, float(eps),
                                         _stream(stream))
    _check(st, "bi_rmsnorm_quantize_e4m3")
    return q, scale


def bi_pins_default_fp8(N: int, K: int) -> Pins:
    p = Pins()
    _check(load().bi_pins_default_fp8(N, K, ctypes.byref(p)), "bi_pins_default_fp8")
    return p


def bi_pins_validate_fp8(N: int, K: int, pins: Pins) -> int:
    return load().bi_pins_validate_fp8(N, K, ctypes.byref(pins))


def bi_gemm_plan_describe_fp8(M: int, N: int, K: int, pins: Pins | None = None, sm_count: int = 0) -> Plan:
    plan = Plan()
    st = load().bi_gemm_plan_describe_fp8(M, N, K, ctypes.byref(pins) if pins is not None else None, sm_count,
                                          ctypes.byref(plan))
    _check(st, "bi_gemm_plan_describe_fp8")
    return plan


def bi_gemm_fp8(xq: torch.Tensor, sx: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor,
                out: torch.Tensor | None = None, pins: Pins | None = None, stream=None) -> torch.Tensor:
    """Y = bf16((Xq . Wq^T) * sx[m] * sw[n]); xq [M,K], wq [N,K] uint8 E4M3 codes."""
    if xq.dim() != 2 or wq.dim() != 2 or xq.shape[1] != wq.shape[1]:
        raise ValueError("expected xq [M,K] and wq [N,K]")
    M, K = xq.shape
    N = wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    st = load().bi_gemm_fp8(_dev_as(xq, "xq", torch.uint8, (M, K)), _dev_as(sx, "sx", torch.float32, (M,)),
                            _dev_as(wq, "wq", torch.uint8, (N, K)), _dev_as(sw, "sw", torch.float32, (N,)),
                            _dev(out, "out", (M, N)), M, N, K,
                            ctypes.byref(pins) if pins is not None else None, _stream(stream))
    _check(st, "bi_gemm_fp8")
    if _call_hooks:
        _report(M, N, K)
    return out


def bi_log_softmax_bf16(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Log-probabilities (fp32 [M,V]) of logits x [M,V] bf16."""
    if x.dim() != 2:
        raise ValueError("expected x [M,V]")
    M, V = x.shape
    if out is None:
        out = torch.empty((M, V), dtype=torch.float32, device=x.device)
    st = load().bi_log_softmax_bf16(_dev(x, "x"), _dev_as(out, "out", torch.float32, (M, V)), M, V,
                                    _stream(stream))
    _check(st, "bi_log_softmax_bf16")
    return out


def bi_token_logprobs_bf16(x: torch.Tensor, ids: torch.Tensor, out: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """out[m] = log-probability of token ids[m] in row m of x [M,V] (fp32 [M])."""
    if x.dim() != 2:
        raise ValueError("expected x [M,V]")
    M, V = x.shape
    if out is None:
        out = torch.empty(M, dtype=torch.float32, device=x.device)
    st = load().bi_token_logprobs_bf16(_dev(x, "x"), _dev_i32(ids, "ids", (M,)),
                                       _dev_as(out, "out", torch.float32, (M,)), M, V, _stream(stream))
    _check(st, "bi_token_logprobs_bf16")
    return out


def bi_silu_mul_bf16(gu: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    M, I2 = gu.shape
    I = I2 // 2
    if out is None:
        out = torch.empty((M, I), dtype=torch.bfloat16, device=gu.device)
    st = load().bi_silu_mul_bf16(_dev(gu, "gu"), _dev(out, "out", (M, I)), M, I, _stream(stream))
    _check(st, "bi_silu_mul_bf16")
    return out


def bi_attention_ctx1_bf16(qkv: torch.Tensor, nq: int, nkv: int, D: int, out: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    M = qkv.shape[0]
    if out is None:
        out = torch.empty((M, nq * D), dtype=torch.bfloat16, device=qkv.device)
    st = load().bi_attention_ctx1_bf16(_dev(qkv, "qkv", (M, (nq + 2 * nkv) * D)),
                                       _dev(out, "out", (M, nq * D)), M, nq, nkv, D, _stream(stream))
    _check(st, "bi_attention_ctx1_bf16")
    return out


def bi_last_device_status(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device's stall status."""
    return int(load().bi_last_device_status(_stream(stream)))


def bi_debug_bounds_enabled() -> bool:
    """True for the debug-bounds build of the library."""
    return bool(load().bi_debug_bounds_enabled())


def bi_debug_bounds_detail(stream=None) -> int:
    """The first failed index check since the last call, (check << 48) | value
    (0 if none), then cleared.  Synchronises the stream."""
    out = ctypes.c_uint64(0)
    _check(load().bi_debug_bounds_detail(ctypes.byref(out), _stream(stream)), "bi_debug_bounds_detail")
    return int(out.value)


# ---------------------------------------------------------------------------
# decode attention over a paged key/value cache
# ---------------------------------------------------------------------------

BI_ATTN_HEAD_DIM = 128
BI_ATTN_MAX_SPLIT = 4096
BI_ATTN_DEFAULT_SPLIT = 256


def bi_decode_attention_workspace_bytes(B: int, Hq: int, Hkv: int, max_seq_len: int, split_size: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(load().bi_decode_attention_workspace_bytes(B, Hq, Hkv, max_seq_len, split_size, ctypes.byref(n)),
           "bi_decode_attention_workspace_bytes")
    return int(n.value)


def _dev_i32(t: torch.Tensor, name: str, shape=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError("%s must be a contiguous int32 CUDA tensor" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    _on_current_device(t, name)
    return t.data_ptr()


def bi_decode_attention_bf16(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                             max_seq_len: int | None = None, split_size: int = 0,
                             out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """out [B,Hq,D] = softmax(scale * q . k) . v over each request's cached
    positions.  q [B,Hq,D]; caches [num_pages, page_size, Hkv, D];
    block_table [B,P] and seq_lens [B] int32 on the device.  max_seq_len
    (default P * page_size) bounds every length; split_size is the pin
    (0 = BI_ATTN_DEFAULT_SPLIT)."""
    if q.dim() != 3 or k_cache.dim() != 4 or block_table.dim() != 2:
        raise ValueError("expected q [B,Hq,D], caches [pages,page_size,Hkv,D], block_table [B,P]")
    B, Hq, D = q.shape
    num_pages, page_size, Hkv, Dk = k_cache.shape
    if Dk != D:
        raise ValueError("q and the caches disagree on the head dimension")
    if max_seq_len is None:
        max_seq_len = block_table.shape[1] * page_size
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    need = bi_decode_attention_workspace_bytes(B, Hq, Hkv, max_seq_len, split_size)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_ptr, ws_bytes = _workspace(workspace)
    st = load().bi_decode_attention_bf16(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache", tuple(k_cache.shape)),
        _dev_i32(block_table, "block_table", (B, block_table.shape[1])), block_table.shape[1],
        _dev_i32(seq_lens, "seq_lens", (B,)), _dev(out, "out", (B, Hq, D)), B, Hq, Hkv, D, num_pages,
        page_size, int(max_seq_len), int(split_size), float(scale), ws_ptr, ws_bytes, _stream(stream))
    _check(st, "bi_decode_attention_bf16")
    return out
