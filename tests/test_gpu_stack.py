"""The decode-step linear stack (configuration 5 and a small variant).

Two kinds of parity, both against the CPU oracle:

1. Step by step (the tight check).  Each step of a layer is fed the GPU's own
   input to that step: GEMMs must meet the GEMM bar, RMSNorm and SiLU*up must be
   within one bf16 ulp, the attention copy and the residual adds bit-exact.

2. End to end (bounded drift).  When the oracle runs the whole stack from the
   same input, the two sides differ in fp32 summation order, so a few bf16-stored
   values differ by one rounding step; every GEMM then mixes its K inputs, so a
   fraction p of one-ulp flips at its input moves each output by about
   sqrt(p) * 2^-8 relative, and the flip fraction grows p -> sqrt(p) per GEMM
   until almost every stored value carries an independent rounding-size
   difference.  With n bf16 stores on the residual path (9 per layer: xn, qkv,
   o, h, hn, gate/up, act, d, out) the relative Frobenius error is then about
   2^-8 * sqrt(n / 3); the bar is 1.5 times that, and per element 8 times the
   Frobenius bar times the row's RMS plus half an ulp.  Bit-exact invariance is
   checked GPU against GPU (batch 1, 8, 32 and 256)."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, bits_to_f64, ulp_bf16
from invariant_bi_gemm_bf16_gb300 import inputs
from invariant_bi_gemm_bf16_gb300.stack import LLAMA31_70B, DecodeStack, StackShape, random_layers

pytestmark = pytest.mark.gpu


def host_layers(layers):
    return [{k: inputs.bits(v) for k, v in L.items()} for L in layers]


def drift_bar(layers: int) -> float:
    return 1.5 * 2.0 ** -8 * np.sqrt(9 * layers / 3.0)


def check_stack(got_bits, want_bits, layers, what):
    g = bits_to_f64(got_bits)
    w = bits_to_f64(want_bits)
    assert np.all(np.isfinite(g)), what
    bar = drift_bar(layers)
    rms = np.sqrt(np.mean(w * w, axis=1, keepdims=True))
    tol = 8 * bar * rms + 0.5 * ulp_bf16(np.maximum(np.abs(g), np.abs(w)))
    err = np.abs(g - w)
    rel = np.linalg.norm(g - w) / np.linalg.norm(w)
    same = float(np.mean(got_bits == want_bits))
    print("%s: rel Frobenius %.2e (bar %.2e), max err/tol %.3f, identical bits %.4f" % (
        what, rel, bar, float((err / tol).max()), same))
    assert rel <= bar, what
    assert np.all(err <= tol), what


def test_small_stack_parity(lib, oracle):
    shape = StackShape(hidden=512, n_q=8, n_kv=2, head_dim=64, inter=1024, layers=2)
    layers = random_layers(shape, seed=1)
    stack = DecodeStack(shape, layers)
    x = inputs.normal((7, shape.hidden), seed=1, stream=0).cuda()
    got = bf16_bits(stack.forward(x))
    want = oracle.stack(inputs.bits(x), host_layers(layers), shape.n_q, shape.n_kv, shape.head_dim, shape.eps)
    check_stack(got, want, shape.layers, "small stack")


@pytest.fixture(scope="module")
def big_stack(lib):
    layers = random_layers(LLAMA31_70B, seed=0)
    stack = DecodeStack(LLAMA31_70B, layers)
    x = inputs.device_normal((32, LLAMA31_70B.hidden), seed=0, stream=0)
    ref = stack.forward(x).clone()
    torch.cuda.synchronize()
    return stack, layers, x, ref


def test_70b_stack_rows_match_oracle(big_stack, oracle):
    """Every output row depends on its own input row only, so the oracle can
    compute two of the 32 rows through all four layers."""
    stack, layers, x, ref = big_stack
    rows = [0, 21]
    want = oracle.stack(inputs.bits(x[rows]), host_layers(layers), LLAMA31_70B.n_q, LLAMA31_70B.n_kv,
                        LLAMA31_70B.head_dim, LLAMA31_70B.eps)
    check_stack(bf16_bits(ref[rows]), want, LLAMA31_70B.layers, "70B stack rows %s" % rows)


def test_70b_stack_batch_invariance(lib, big_stack):
    """The same 32 rows at batch 1 (32 calls), batch 8 (4 calls) and embedded
    at random positions in a batch of 256 give identical bits."""
    stack, layers, x, ref = big_stack
    ref16 = ref.view(torch.int16)
    for i in range(32):
        assert torch.equal(stack.forward(x[i:i + 1]).view(torch.int16), ref16[i:i + 1]), i
    for i in range(0, 32, 8):
        assert torch.equal(stack.forward(x[i:i + 8]).view(torch.int16), ref16[i:i + 8]), i
    full, pos = inputs.scatter_rows(x.cpu(), 256, seed=5)
    out = stack.forward(full.cuda())
    assert torch.equal(out[torch.from_numpy(pos).cuda()].view(torch.int16), ref16)
    assert lib.bi_last_device_status() == lib.BI_OK


def test_70b_stack_steps(big_stack, oracle):
    """Every step of the first and the last layer, each fed the GPU's own input
    (two rows), against the oracle's step."""
    from helpers import check_gemm_parity, check_ulp
    from invariant_bi_gemm_bf16_gb300 import binding as bd
    stack, layers, x, ref = big_stack
    s = LLAMA31_70B
    cur = x[[0, 21]].contiguous()
    for l, L in enumerate(layers):
        H = host_layers([L])[0] if l in (0, len(layers) - 1) else None
        xn = bd.bi_rmsnorm_bf16(cur, L["g_attn"], s.eps)
        qkv = bd.bi_gemm_bf16(xn, L["Wqkv"])
        att = bd.bi_attention_ctx1_bf16(qkv, s.n_q, s.n_kv, s.head_dim)
        o = bd.bi_gemm_bf16(att, L["Wo"])
        h = bd.bi_residual_add_bf16(cur, o)
        hn = bd.bi_rmsnorm_bf16(h, L["g_mlp"], s.eps)
        gu = bd.bi_gemm_bf16(hn, L["Wgu"])
        act = bd.bi_silu_mul_bf16(gu)
        d = bd.bi_gemm_bf16(act, L["Wd"])
        out = bd.bi_residual_add_bf16(h, d)
        # the steps compose to exactly what the stack computes
        single = DecodeStack(StackShape(s.hidden, s.n_q, s.n_kv, s.head_dim, s.inter, 1, s.eps), [L])
        assert torch.equal(single.forward(cur).view(torch.int16), out.view(torch.int16))
        if H is not None:
            b = inputs.bits
            check_ulp(b(xn), oracle.rmsnorm(b(cur), H["g_attn"], s.eps), 1, "layer %d xn" % l)
            check_gemm_parity(b(qkv), oracle.gemm(b(xn), H["Wqkv"])[0], s.hidden, "layer %d qkv" % l)
            assert np.array_equal(b(att), oracle.attention_ctx1(b(qkv), s.n_q, s.n_kv, s.head_dim))
            check_gemm_parity(b(o), oracle.gemm(b(att), H["Wo"])[0], s.n_q * s.head_dim, "layer %d o" % l)
            assert np.array_equal(b(h), oracle.residual_add(b(cur), b(o)))
            check_ulp(b(hn), oracle.rmsnorm(b(h), H["g_mlp"], s.eps), 1, "layer %d hn" % l)
            check_gemm_parity(b(gu), oracle.gemm(b(hn), H["Wgu"])[0], s.hidden, "layer %d gate_up" % l)
            check_ulp(b(act), oracle.silu_mul(b(gu)), 1, "layer %d act" % l)
            check_gemm_parity(b(d), oracle.gemm(b(act), H["Wd"])[0], s.inter, "layer %d down" % l)
            assert np.array_equal(b(out), oracle.residual_add(b(h), b(d)))
        cur = out
