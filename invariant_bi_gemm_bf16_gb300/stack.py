"""A Llama-style decode-step linear stack built from the C ABI calls.

Per layer, on x [M, hidden]:
    qkv = RMSNorm(x; g_attn) . Wqkv^T              (bi_rmsnorm_gemm_bf16)
    a   = attention at a context of one token       (bi_attention_ctx1_bf16)
    h   = x + a . Wo^T                              (bi_gemm_bf16, bi_residual_add_bf16)
    gu  = RMSNorm(h; g_mlp) . Wgu^T                 (bi_rmsnorm_gemm_bf16)
    x'  = h + (silu(gate) * up) . Wd^T              (bi_silu_mul_bf16, bi_gemm_bf16, bi_residual_add_bf16)

Every step is row-local and runs in the library's kernels; this module only
sequences the calls and keeps the per-M activation buffers.  With a single
key, the softmax weight is exactly 1, so each query head returns its
key/value group's v vector (the attention stand-in for the linear stack of a
decode step; CoRun, Padding is Simple and Efficient for Deterministic LLM
Inference, Fig. 1(b) and Fig. 4, time such a decode forward).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as bd
from . import inputs


@dataclass
class StackShape:
    hidden: int = 8192
    n_q: int = 64
    n_kv: int = 8
    head_dim: int = 128
    inter: int = 28672
    layers: int = 4
    eps: float = 1e-5

    @property
    def qkv_width(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim


LLAMA31_70B = StackShape()


def random_layers(shape: StackShape, seed: int = 0, device="cuda") -> list:
    """Random-init weights (N(0, 0.02)) and gains (N(1, 0.1)) drawn on the device."""
    layers = []
    for l in range(shape.layers):
        base = 16 * (l + 1)
        layers.append({
            "g_attn": inputs.device_normal((shape.hidden,), std=0.1, mean=1.0, seed=seed, stream=base + 2, device=device),
            "Wqkv": inputs.device_normal((shape.qkv_width, shape.hidden), std=0.02, seed=seed, stream=base + 3,
                                         device=device),
            "Wo": inputs.device_normal((shape.hidden, shape.n_q * shape.head_dim), std=0.02, seed=seed,
                                       stream=base + 4, device=device),
            "g_mlp": inputs.device_normal((shape.hidden,), std=0.1, mean=1.0, seed=seed, stream=base + 5, device=device),
            "Wgu": inputs.device_normal((2 * shape.inter, shape.hidden), std=0.02, seed=seed, stream=base + 6,
                                        device=device),
            "Wd": inputs.device_normal((shape.hidden, shape.inter), std=0.02, seed=seed, stream=base + 7, device=device),
        })
    return layers


class DecodeStack:
    def __init__(self, shape: StackShape, layers: list, pins: dict | None = None,
                 pin_table: dict | None = None):
        """pins: {"qkv"|"o"|"gu"|"d": Pins} overrides; pin_table: {(N, K): Pins}
        (a tuned table, see tuner.load); both are fixed for every batch size."""
        self.shape = shape
        self.layers = layers
        s = shape
        # one pin set per (N, K), fixed for the deployment (never chosen from M)
        self.pins = {
            "qkv": bd.bi_pins_default(s.qkv_width, s.hidden),
            "o": bd.bi_pins_default(s.hidden, s.n_q * s.head_dim),
            "gu": bd.bi_pins_default(2 * s.inter, s.hidden),
            "d": bd.bi_pins_default(s.hidden, s.inter),
        }
        # The weights are written once, before serving: let each GEMM start
        # streaming its weights while the small kernels before it finish.
        for k in self.pins:
            self.pins[k] = self.pins[k].replace(flags=self.pins[k].flags | bd.BI_FLAG_PREFETCH_W)
        if pin_table:
            shapes = {"qkv": (s.qkv_width, s.hidden), "o": (s.hidden, s.n_q * s.head_dim),
                      "gu": (2 * s.inter, s.hidden), "d": (s.hidden, s.inter)}
            for name, nk in shapes.items():
                if nk in pin_table:
                    p = pin_table[nk]
                    self.pins[name] = p.replace(flags=p.flags | bd.BI_FLAG_PREFETCH_W)
        if pins:
            self.pins.update(pins)
        self._nk = {"qkv": (s.qkv_width, s.hidden), "o": (s.hidden, s.n_q * s.head_dim),
                    "gu": (2 * s.inter, s.hidden), "d": (s.hidden, s.inter)}
        self._bufs = {}
        self._fold = {}

    def _workspace(self, name: str, M: int, scratch: int, device) -> torch.Tensor:
        """The projection's workspace for M rows: room for the GEMM's fold in
        front (its counters at offset 0, zeroed once and left zero by every
        call, so one buffer serves every M) and `scratch` bytes at the end for
        the fused call's RMSNorm.  Grown, as a new zeroed buffer, when a call
        needs more."""
        N, K = self._nk[name]
        need = bd.bi_gemm_bf16_workspace_bytes(M, N, K, self.pins[name]) + scratch
        buf = self._fold.get(name)
        if buf is None or buf.numel() < need:
            buf = torch.zeros(max(need, 256), dtype=torch.uint8, device=device)
            self._fold[name] = buf
        return buf

    def _buffers(self, M: int, device):
        if M not in self._bufs:
            s = self.shape
            e = dict(dtype=torch.bfloat16, device=device)
            ws = bd.bi_rmsnorm_gemm_workspace_bytes(M, s.hidden)
            self._bufs[M] = {
                "ws_qkv": self._workspace("qkv", M, ws, device),
                "ws_o": self._workspace("o", M, 0, device),
                "ws_gu": self._workspace("gu", M, ws, device),
                "ws_d": self._workspace("d", M, 0, device),
                "qkv": torch.empty((M, s.qkv_width), **e),
                "att": torch.empty((M, s.n_q * s.head_dim), **e),
                "o": torch.empty((M, s.hidden), **e),
                "h": torch.empty((M, s.hidden), **e),
                "gu": torch.empty((M, 2 * s.inter), **e),
                "act": torch.empty((M, s.inter), **e),
                "d": torch.empty((M, s.hidden), **e),
                "x": [torch.empty((M, s.hidden), **e), torch.empty((M, s.hidden), **e)],
            }
        return self._bufs[M]

    def launches_per_step(self) -> int:
        return 10 * self.shape.layers   # the two fused calls launch two kernels each

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        """x [M, hidden] bf16 on the device -> [M, hidden] (a buffer owned by this object)."""
        s = self.shape
        M = x.shape[0]
        b = self._buffers(M, x.device)
        cur = x
        for i, L in enumerate(self.layers):
            bd.bi_rmsnorm_gemm_bf16(cur, L["g_attn"], L["Wqkv"], s.eps, pins=self.pins["qkv"], out=b["qkv"],
                                    workspace=b["ws_qkv"])
            bd.bi_attention_ctx1_bf16(b["qkv"], s.n_q, s.n_kv, s.head_dim, out=b["att"])
            bd.bi_gemm_bf16(b["att"], L["Wo"], out=b["o"], pins=self.pins["o"], workspace=b["ws_o"])
            bd.bi_residual_add_bf16(cur, b["o"], out=b["h"])
            bd.bi_rmsnorm_gemm_bf16(b["h"], L["g_mlp"], L["Wgu"], s.eps, pins=self.pins["gu"], out=b["gu"],
                                    workspace=b["ws_gu"])
            bd.bi_silu_mul_bf16(b["gu"], out=b["act"])
            bd.bi_gemm_bf16(b["act"], L["Wd"], out=b["d"], pins=self.pins["d"], workspace=b["ws_d"])
            nxt = b["x"][i % 2]
            bd.bi_residual_add_bf16(b["h"], b["d"], out=nxt)
            cur = nxt
        return cur
