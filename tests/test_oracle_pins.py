"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test fixes the oracle to an independent fact -- a hand-derived bit
pattern, an exact integer result, a closed form, a textbook error bound against
an fp64 brute force, or a worked summation-order example -- chosen so that a
plausible mistake (a dropped term, a wrong sign or index, a transposed operand,
a different summation order, a wrong rounding mode, eps outside the sqrt)
fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from invariant_bi_gemm_bf16_gb300 import inputs

U = 2.0 ** -24  # unit roundoff of binary32


def f32_bits(x: float) -> int:
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0])


def bits_to_f32(b: int) -> float:
    return float(np.array([b], dtype=np.uint32).view(np.float32)[0])


def bf16_val(bits16) -> np.ndarray:
    b = np.asarray(bits16, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def gamma(n: int) -> float:
    return n * U / (1 - n * U)


def ordered(bits16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers ordered like the values (sign-magnitude)."""
    b = bits16.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_of_f64(x: np.ndarray) -> np.ndarray:
    """Exact round-to-nearest-even of float64 values to bf16, via Fractions
    (independent of the oracle's bit trick and of numpy's float32 cast)."""
    out = []
    for v in np.asarray(x, dtype=np.float64).ravel():
        if v == 0:
            out.append(0x8000 if math.copysign(1, v) < 0 else 0)
            continue
        s = 0x8000 if v < 0 else 0
        a = Fraction(abs(float(v)))
        e = math.floor(math.log2(a))
        while Fraction(2) ** e > a:
            e -= 1
        while Fraction(2) ** (e + 1) <= a:
            e += 1
        # 8 significant bits: quantum 2^(e-7)
        q = Fraction(2) ** (e - 7)
        n = a / q
        fl = math.floor(n)
        rem = n - fl
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
            fl += 1
        val = fl * q
        fbits = f32_bits(float(val))
        out.append(s | (fbits >> 16))
    return np.array(out, dtype=np.uint16).reshape(np.shape(x))


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("f32_in, bf16_out", [
    (0x3F800000, 0x3F80),   # 1.0
    (0x3F808000, 0x3F80),   # 1 + 2^-8: exact tie, kept part even -> down
    (0x3F818000, 0x3F82),   # 1 + 3*2^-8: exact tie, kept part odd -> up
    (0x3F808001, 0x3F81),   # just above the tie -> up
    (0x3F807FFF, 0x3F80),   # just below the tie -> down
    (0xBF808001, 0xBF81),   # sign is carried
    (0x80000000, 0x8000),   # -0
    (0x7F800000, 0x7F80),   # +inf
    (0xFF800000, 0xFF80),   # -inf
    (0x7F7FFFFF, 0x7F80),   # FLT_MAX rounds past the largest bf16 -> inf
    (0x7FC00000, 0x7FC0),   # quiet NaN
    (0x7F800001, 0x7FC0),   # signalling NaN whose payload would truncate to inf -> stays NaN
    (0x00010000, 0x0001),   # subnormal kept exactly
    (0x00008000, 0x0000),   # smallest subnormal tie -> even (0)
])
def test_bf16_rne_bits(oracle, f32_in, bf16_out):
    got = oracle.bf16_rne(np.array([bits_to_f32(f32_in)], dtype=np.float32))
    assert int(got[0]) == bf16_out


def test_bf16_rne_matches_exact_rounding(oracle):
    r = np.random.default_rng(123)
    x = (r.standard_normal(4000) * np.exp(r.uniform(-20, 20, 4000))).astype(np.float32)
    got = oracle.bf16_rne(x)
    want = bf16_of_f64(x.astype(np.float64))
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# GEMM
# ---------------------------------------------------------------------------

def test_gemm_integer_inputs_exact(oracle):
    """Integer inputs with small magnitudes: every partial sum is an integer below
    2^24, so every summation order gives the exact integer product."""
    X = inputs.integers((7, 300), -8, 8, seed=1, stream=0)
    W = inputs.integers((13, 300), -8, 8, seed=1, stream=1)
    Yf, Yb = oracle.gemm(inputs.bits(X), inputs.bits(W))
    exact = X.float().numpy().astype(np.int64) @ W.float().numpy().astype(np.int64).T
    assert np.array_equal(Yf.astype(np.int64), exact)
    assert np.array_equal(Yf, exact.astype(np.float32))


def test_gemm_summation_order_worked_example(oracle):
    """The order of the fp32 chain is the sequential a+b+c+d of CoRun Fig. 3.
    With x = [1, 2^-24, 2^-24, 2^-24] and w = 1:
      sequential ((1 + 2^-24) + 2^-24) + 2^-24: each step is a tie that rounds to
        the even value 1, so the result is exactly 1;
      the split-K tree (1 + 2^-24) + (2^-24 + 2^-24) gives 1 + 2^-23;
      the reversed chain gives 1 + 3*2^-24, a tie that rounds to 1 + 2^-22.
    Values derived by hand above; only the sequential order yields 1.0."""
    x = np.array([[1.0, 2.0 ** -24, 2.0 ** -24, 2.0 ** -24]], dtype=np.float32)
    w = np.ones((1, 4), dtype=np.float32)
    Yf, _ = oracle.gemm(inputs.bits(inputs.to_bf16(x)), inputs.bits(inputs.to_bf16(w)))
    assert Yf[0, 0] == np.float32(1.0)
    # and the other orders really do differ (so the example is discriminating)
    assert np.float32(1.0) + np.float32(2.0 ** -23) != np.float32(1.0)


def test_gemm_identity_weights(oracle):
    X = inputs.normal((9, 64), seed=2, stream=0)
    Wf = np.eye(64, dtype=np.float32)
    Yf, Yb = oracle.gemm(inputs.bits(X), inputs.bits(inputs.to_bf16(Wf)))
    assert np.array_equal(Yb, inputs.bits(X))


def test_gemm_permutation_weights(oracle):
    X = inputs.normal((5, 48), seed=3, stream=0)
    perm = np.random.default_rng(3).permutation(48)
    Wf = np.zeros((48, 48), dtype=np.float32)
    Wf[np.arange(48), perm] = 1.0  # y[n] = x[perm[n]]
    _, Yb = oracle.gemm(inputs.bits(X), inputs.bits(inputs.to_bf16(Wf)))
    assert np.array_equal(Yb, inputs.bits(X)[:, perm])


def test_gemm_one_hot_rows(oracle):
    """One non-zero per X row: y[m,n] = x[m,k_m] * w[n,k_m], a single exact product."""
    K, M, N = 40, 6, 11
    r = np.random.default_rng(4)
    W = inputs.normal((N, K), std=0.02, seed=4, stream=1)
    Xf = np.zeros((M, K), dtype=np.float32)
    ks = r.integers(0, K, size=M)
    Xf[np.arange(M), ks] = r.standard_normal(M).astype(np.float32)
    X = inputs.to_bf16(Xf)
    Yf, Yb = oracle.gemm(inputs.bits(X), inputs.bits(W))
    xv = X.double().numpy()
    wv = W.double().numpy()
    for m in range(M):
        exact = xv[m, ks[m]] * wv[:, ks[m]]
        assert np.array_equal(Yf[m].astype(np.float64), exact)
        assert np.array_equal(Yb[m], bf16_of_f64(exact))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 17), (4, 7, 256), (2, 3, 4096)])
def test_gemm_higham_bound(oracle, M, N, K):
    """Recursive summation of K exact products: |fl(sum) - sum| <= gamma_{K-1} sum|p_k|
    (Higham, Accuracy and Stability of Numerical Algorithms, Sec. 4.2)."""
    X = inputs.normal((M, K), seed=5, stream=0)
    W = inputs.normal((N, K), std=0.02, seed=5, stream=1)
    Yf, Yb = oracle.gemm(inputs.bits(X), inputs.bits(W))
    xv = X.double().numpy()
    wv = W.double().numpy()
    exact = xv @ wv.T                    # products exact in fp64; fp64 sum error ~1e-16 relative
    absdot = np.abs(xv) @ np.abs(wv).T
    bound = gamma(max(K - 1, 0)) * absdot + 1e-300
    assert np.all(np.abs(Yf.astype(np.float64) - exact) <= bound * (1 + 1e-9) + 1e-30)
    # the bf16 output is the round-to-nearest-even of the fp32 result
    assert np.array_equal(Yb, bf16_of_f64(Yf.astype(np.float64)))


def test_gemm_transposition_and_dropped_term(oracle):
    """A non-square case where X.W (instead of X.W^T) or a skipped last k fails."""
    X = inputs.integers((2, 3), -3, 3, seed=6, stream=0)
    W = inputs.integers((4, 3), -3, 3, seed=6, stream=1)
    Yf, _ = oracle.gemm(inputs.bits(X), inputs.bits(W))
    xv = X.float().numpy().astype(int)
    wv = W.float().numpy().astype(int)
    for m in range(2):
        for n in range(4):
            assert Yf[m, n] == sum(xv[m, k] * wv[n, k] for k in range(3))


def test_gemm_sampled_matches_full(oracle):
    X = inputs.normal((6, 96), seed=7, stream=0)
    W = inputs.normal((10, 96), std=0.02, seed=7, stream=1)
    Yf, _ = oracle.gemm(inputs.bits(X), inputs.bits(W))
    rows = np.array([0, 5, 3, 3])
    cols = np.array([9, 0, 4, 5])
    s = oracle.gemm_sampled(inputs.bits(X), inputs.bits(W), rows, cols)
    assert np.array_equal(s, Yf[rows, cols])


def test_gemm_thread_count_does_not_change_bits(oracle):
    X = inputs.normal((5, 512), seed=8, stream=0)
    W = inputs.normal((37, 512), std=0.02, seed=8, stream=1)
    a = oracle.gemm(inputs.bits(X), inputs.bits(W), nthreads=1)[0]
    b = oracle.gemm(inputs.bits(X), inputs.bits(W), nthreads=7)[0]
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_gemm_batch_invariance_by_construction(oracle):
    """Def. 1 of CoRun Sec. III-B on the oracle: a row's bits do not depend on
    the batch size, its position, or its co-runners (including inf/nan rows)."""
    K, N = 128, 24
    W = inputs.bits(inputs.normal((N, K), std=0.02, seed=9, stream=1))
    target = inputs.normal((3, K), seed=9, stream=0)
    ref = oracle.gemm(inputs.bits(target), W)[0]
    for batch, fill in [(3, None), (17, None), (64, float("nan")), (40, float("inf")), (33, 65504.0)]:
        full, pos = inputs.scatter_rows(target, batch, seed=batch, corunner_fill=fill)
        got = oracle.gemm(inputs.bits(full), W)[0]
        assert np.array_equal(got[pos].view(np.uint32), ref.view(np.uint32))


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

EPS = 1e-5


def test_rmsnorm_zero_row(oracle):
    X = np.zeros((2, 64), dtype=np.uint16)
    g = inputs.bits(inputs.normal((64,), std=0.1, mean=1.0, seed=10, stream=2))
    Y = oracle.rmsnorm(X, g, EPS)
    assert np.all(bf16_val(Y) == 0)


def test_rmsnorm_unit_rows_are_fixed_points(oracle):
    """Rows of +-1 with gain 1: mean(x^2) = 1 exactly, r = 1/sqrt(1 + 1e-5) =
    0.999995..., and bf16 rounds +-0.999995 to +-1 (the next bf16 below 1 is
    0.99609375).  So Y == X bit for bit."""
    r = np.random.default_rng(11)
    Xf = np.where(r.random((4, 256)) < 0.5, -1.0, 1.0).astype(np.float32)
    X = inputs.bits(inputs.to_bf16(Xf))
    g = inputs.bits(inputs.to_bf16(np.ones(256, dtype=np.float32)))
    assert np.array_equal(oracle.rmsnorm(X, g, EPS), X)


@pytest.mark.parametrize("c", [1.0, 4.0, 0.0625, 1024.0])
def test_rmsnorm_constant_magnitude_rows(oracle, c):
    """Rows of +-c with gain 0.5: y = +-0.5 * c / sqrt(c^2 + eps), which rounds
    to +-0.5 for these c (|c/sqrt(c^2+eps) - 1| < 2^-10)."""
    r = np.random.default_rng(12)
    sign = np.where(r.random((3, 128)) < 0.5, -1.0, 1.0)
    X = inputs.bits(inputs.to_bf16((sign * c).astype(np.float32)))
    g = inputs.bits(inputs.to_bf16(np.full(128, 0.5, dtype=np.float32)))
    Y = bf16_val(oracle.rmsnorm(X, g, EPS))
    assert np.array_equal(Y, (0.5 * sign).astype(np.float32))


def test_rmsnorm_eps_inside_sqrt(oracle):
    """Tiny rows where eps dominates: y = x / sqrt(x^2 + eps) * g.  With x = 2^-10:
    mean = 2^-20, r = 1/sqrt(2^-20 + 1e-5) ~ 302.5 (eps outside the sqrt, or added
    to the root, gives very different values)."""
    x = 2.0 ** -10
    X = inputs.bits(inputs.to_bf16(np.full((1, 64), x, dtype=np.float32)))
    g = inputs.bits(inputs.to_bf16(np.ones(64, dtype=np.float32)))
    Y = oracle.rmsnorm(X, g, EPS)
    want = bf16_of_f64(np.array([x / math.sqrt(x * x + float(np.float32(EPS)))]))
    diff = np.abs(ordered(Y[0]) - int(ordered(want)[0]))
    assert diff.max() <= 1


@pytest.mark.parametrize("H", [8, 256, 4096])
def test_rmsnorm_fp64_brute_force(oracle, H):
    """Against an fp64 evaluation of the same formula: within one bf16 ulp, and
    the inverse RMS within Higham's bound for the sum of squares plus the few
    roundings of the mean, sqrt and division."""
    X = inputs.rows_loguniform(16, H, seed=13, stream=0)
    g = inputs.normal((H,), std=0.1, mean=1.0, seed=13, stream=2)
    Y = oracle.rmsnorm(inputs.bits(X), inputs.bits(g), EPS)
    xv = X.double().numpy()
    gv = g.double().numpy()
    eps32 = float(np.float32(EPS))
    ss = (xv * xv).sum(axis=1)
    r_exact = 1.0 / np.sqrt(ss / H + eps32)
    want = bf16_of_f64((xv * r_exact[:, None]) * gv[None, :])
    assert np.abs(ordered(Y) - ordered(want)).max() <= 1
    for m in range(16):
        r_or = float(oracle.inv_rms(inputs.bits(X[m]), EPS))
        rel = abs(r_or - r_exact[m]) / r_exact[m]
        assert rel <= 0.5 * gamma(H - 1) + 4 * U


def test_rmsnorm_row_independence(oracle):
    H = 256
    g = inputs.bits(inputs.normal((H,), std=0.1, mean=1.0, seed=14, stream=2))
    target = inputs.rows_loguniform(2, H, seed=14, stream=0)
    ref = oracle.rmsnorm(inputs.bits(target), g, EPS)
    full, pos = inputs.scatter_rows(target, 37, seed=14, corunner_fill=float("nan"))
    got = oracle.rmsnorm(inputs.bits(full), g, EPS)
    assert np.array_equal(got[pos], ref)


def test_rmsnorm_gemm_is_the_composition(oracle):
    X = inputs.normal((5, 256), seed=15, stream=0)
    g = inputs.normal((256,), std=0.1, mean=1.0, seed=15, stream=2)
    W = inputs.normal((64, 256), std=0.02, seed=15, stream=1)
    Yf, Yb, Xh = oracle.rmsnorm_gemm(inputs.bits(X), inputs.bits(g), inputs.bits(W), EPS)
    Xh2 = oracle.rmsnorm(inputs.bits(X), inputs.bits(g), EPS)
    assert np.array_equal(Xh, Xh2)
    Yf2, Yb2 = oracle.gemm(Xh2, inputs.bits(W))
    assert np.array_equal(Yf.view(np.uint32), Yf2.view(np.uint32))
    assert np.array_equal(Yb, Yb2)


def test_rmsnorm_gemm_closed_form(oracle):
    """+-1 rows, gain 1 (normalisation is the identity, see above) into identity
    weights: the fused layer returns X."""
    r = np.random.default_rng(16)
    Xf = np.where(r.random((3, 64)) < 0.5, -1.0, 1.0).astype(np.float32)
    X = inputs.bits(inputs.to_bf16(Xf))
    g = inputs.bits(inputs.to_bf16(np.ones(64, dtype=np.float32)))
    W = inputs.bits(inputs.to_bf16(np.eye(64, dtype=np.float32)))
    _, Yb, _ = oracle.rmsnorm_gemm(X, g, W, EPS)
    assert np.array_equal(Yb, X)


# ---------------------------------------------------------------------------
# decode-layer glue
# ---------------------------------------------------------------------------

def test_silu_mul_closed_forms(oracle):
    gate = np.array([[0.0, 20.0, -20.0, 1.0, -1.0, 2.0]], dtype=np.float32)
    up = np.array([[3.0, 1.0, 1.0, 1.0, 1.0, -0.5]], dtype=np.float32)
    gu = inputs.bits(inputs.to_bf16(np.concatenate([gate, up], axis=1)))
    got = oracle.silu_mul(gu)
    g64 = gate.astype(np.float64)
    want = bf16_of_f64(g64 / (1 + np.exp(-g64)) * up.astype(np.float64))
    assert np.abs(ordered(got) - ordered(want)).max() <= 1
    assert bf16_val(got)[0, 0] == 0.0          # silu(0) = 0
    assert bf16_val(got)[0, 1] == 20.0         # silu(20) = 20 / (1 + 2e-9) rounds to 20


def test_residual_add_exact(oracle):
    a = inputs.integers((4, 32), -100, 100, seed=17, stream=0)
    b = inputs.integers((4, 32), -100, 100, seed=17, stream=1)
    got = bf16_val(oracle.residual_add(inputs.bits(a), inputs.bits(b)))
    assert np.array_equal(got, (a.float() + b.float()).numpy())


def test_attention_ctx1_routing(oracle):
    """nq=4 query heads, nkv=2 groups, D=2: heads 0,1 read v group 0 and heads 2,3
    read v group 1 (hand-written expectation)."""
    q = [1, 2, 3, 4, 5, 6, 7, 8]
    k = [9, 10, 11, 12]
    v = [13, 14, 15, 16]
    qkv = inputs.bits(inputs.to_bf16(np.array([q + k + v], dtype=np.float32)))
    got = bf16_val(oracle.attention_ctx1(qkv, 4, 2, 2))
    assert got.tolist() == [[13, 14, 13, 14, 15, 16, 15, 16]]


def _layer(Hd, nq, nkv, D, I, seed, zero=False):
    def w(shape, stream):
        if zero:
            return inputs.bits(inputs.to_bf16(np.zeros(shape, dtype=np.float32)))
        return inputs.bits(inputs.normal(shape, std=0.02, seed=seed, stream=stream))
    return {
        "g_attn": inputs.bits(inputs.normal((Hd,), std=0.1, mean=1.0, seed=seed, stream=2)),
        "g_mlp": inputs.bits(inputs.normal((Hd,), std=0.1, mean=1.0, seed=seed, stream=3)),
        "Wqkv": w(((nq + 2 * nkv) * D, Hd), 4),
        "Wo": w((Hd, nq * D), 5),
        "Wgu": w((2 * I, Hd), 6),
        "Wd": w((Hd, I), 7),
    }


def test_decode_layer_zero_weights_is_identity(oracle):
    x = inputs.bits(inputs.normal((3, 32), seed=18, stream=0))
    layer = _layer(32, 4, 2, 8, 48, seed=18, zero=True)
    assert np.array_equal(oracle.stack(x, [layer, layer], 4, 2, 8, EPS), x)


def test_decode_layer_attention_path_wiring(oracle):
    """Wgu = Wd = 0 and selector weights: Wqkv's v rows copy the normalised
    input, Wo sums head copies onto the hidden dims.  Then
    out = x + bf16(sum over heads of the routed v), checked against numpy."""
    Hd, nq, nkv, D, I = 8, 4, 2, 4, 16
    layer = _layer(Hd, nq, nkv, D, I, seed=19, zero=True)
    Wqkv = np.zeros(((nq + 2 * nkv) * D, Hd), dtype=np.float32)
    for j in range(nkv * D):                     # v rows: v = xn (hidden 8 = nkv*D)
        Wqkv[(nq + nkv) * D + j, j] = 1.0
    Wo = np.zeros((Hd, nq * D), dtype=np.float32)
    for j in range(nq):                          # o[d] = head j's v[d] for heads 0 and 2
        if j % 2 == 0:
            for d in range(D):
                Wo[(j // 2) * D + d, j * D + d] = 1.0
    layer["Wqkv"] = inputs.bits(inputs.to_bf16(Wqkv))
    layer["Wo"] = inputs.bits(inputs.to_bf16(Wo))
    x = inputs.bits(inputs.normal((2, Hd), seed=19, stream=0))
    out = oracle.decode_layer(x, layer, nq, nkv, D, EPS)
    xn = oracle.rmsnorm(x, layer["g_attn"], EPS)
    # head 0 reads group 0 = xn[:, 0:4]; head 2 reads group 1 = xn[:, 4:8]
    o = np.concatenate([xn[:, 0:4], xn[:, 4:8]], axis=1)
    want = bf16_of_f64(bf16_val(x).astype(np.float64) + bf16_val(o).astype(np.float64))
    assert np.array_equal(out, want)


def test_decode_layer_mlp_path_wiring(oracle):
    """The MLP half with non-zero weights, against a numpy closed form.

    Wo = 0 makes the attention half exact (h = x + 0 = x).  g_mlp is not
    g_attn.  Wgu's gate rows are selectors (gate_j = hn_j) and its up rows
    selectors of another column (up_j = hn_(j+5) mod 16); Wd is a permutation
    (d_i = s_(3i+1) mod 16).  Each selected value is one exact product plus
    zeros, so only RMSNorm_2, SiLU(gate) * up and the residual round.  hn is
    computed from the RMSNorm definition in numpy float32 (small-integer rows
    make the sum of squares and the mean exact), silu in fp64.  Wiring slips
    this catches: RMSNorm_2 skipped (gu = h . Wgu^T), RMSNorm_2 with g_attn,
    gate and up swapped, and d = gu . Wd^T in place of s . Wd^T."""
    Hd, nq, nkv, D, I = 16, 2, 1, 8, 16
    layer = _layer(Hd, nq, nkv, D, I, seed=20, zero=True)
    g_attn = np.ones(Hd, dtype=np.float32)
    g_mlp = (0.5 + np.arange(Hd) / 16.0).astype(np.float32)       # exact in bf16, far from 1
    layer["g_attn"] = inputs.bits(inputs.to_bf16(g_attn))
    layer["g_mlp"] = inputs.bits(inputs.to_bf16(g_mlp))
    layer["Wqkv"] = inputs.bits(inputs.to_bf16(np.full(((nq + 2 * nkv) * D, Hd), 0.25, dtype=np.float32)))
    up_src = [(j + 5) % Hd for j in range(I)]
    perm = [(3 * i + 1) % I for i in range(Hd)]
    Wgu = np.zeros((2 * I, Hd), dtype=np.float32)
    for j in range(I):
        Wgu[j, j] = 1.0
        Wgu[I + j, up_src[j]] = 1.0
    Wd = np.zeros((Hd, I), dtype=np.float32)
    for i in range(Hd):
        Wd[i, perm[i]] = 1.0
    layer["Wgu"] = inputs.bits(inputs.to_bf16(Wgu))
    layer["Wd"] = inputs.bits(inputs.to_bf16(Wd))
    # positive integer rows with an RMS far from 1 (so skipping the norm shows)
    x = np.array([[1 + (3 * k) % 7 for k in range(Hd)],
                  [8 - (5 * k) % 6 for k in range(Hd)]], dtype=np.float32)
    xb = inputs.bits(inputs.to_bf16(x))
    out = oracle.decode_layer(xb, layer, nq, nkv, D, EPS)

    want = []
    for row in x:
        ss = np.float32(0.0)
        for v in row:
            ss = np.float32(ss + np.float32(v * v))
        mean = np.float32(ss / np.float32(Hd))
        r = np.float32(np.float32(1.0) / np.sqrt(np.float32(mean + np.float32(EPS))))
        hn = bf16_val(bf16_of_f64(((row * r).astype(np.float32) * g_mlp).astype(np.float32).astype(np.float64)))
        gate = hn[:I].astype(np.float64)
        up = hn[up_src].astype(np.float64)
        s = bf16_val(bf16_of_f64(gate / (1.0 + np.exp(-gate)) * up)).astype(np.float64)
        d = s[perm]
        want.append(bf16_of_f64(row.astype(np.float64) + d))
    want = np.array(want, dtype=np.uint16)
    # silu goes through expf on one side and exp in fp64 on the other: one ulp
    assert np.abs(ordered(out) - ordered(want)).max() <= 1
    assert not np.array_equal(out, xb)   # the MLP half changed every row


# Three (acc, sx, sw) triples where the three orders of applying the scales
# give different bf16 results: bf16((acc*sx)*sw) differs from
# bf16(acc*(sx*sw)) and from bf16((acc*sw)*sx) in fp32.  Found by a search
# over random fp32 scales and confirmed below with exact rational arithmetic.
_SCALE_ORDER_CASES = [
    (3, 0.05462578684091568, 0.9683547019958496),
    (11, 0.023879144340753555, 1.3570051193237305),
    (19, 0.05306759104132652, 1.9913160800933838),
]


def _rne_frac(a: Fraction, bits: int) -> Fraction:
    """Exact round-to-nearest-even of a rational to `bits` significant bits
    (normal range only)."""
    if a == 0:
        return Fraction(0)
    sign = -1 if a < 0 else 1
    a = abs(a)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - bits + 1)
    n = a / q
    fl = math.floor(n)
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * q


def test_gemm_e4m3_scale_application_order(oracle):
    """y = bf16((acc * sx[m]) * sw[n]) with each product rounded to fp32, in
    that order.  The cases are chosen so that each other order changes the
    bf16 result; the expected value is derived with exact rationals."""
    f32 = lambda a: _rne_frac(a, 24)
    bf = lambda a: _rne_frac(a, 8)
    # acc as a sum of E4M3-exact integers, each times a weight code of 1
    parts = {3: [3], 11: [8, 3], 19: [16, 3]}
    for acc, sx, sw in _SCALE_ORDER_CASES:
        fsx, fsw = Fraction(float(np.float32(sx))), Fraction(float(np.float32(sw)))
        assert fsx == Fraction(sx) and fsw == Fraction(sw)   # the scales are fp32 values
        want = bf(f32(f32(acc * fsx) * fsw))
        assert want != bf(f32(acc * f32(fsx * fsw)))
        assert want != bf(f32(f32(acc * fsw) * fsx))
        vals = parts[acc]
        vx = np.zeros((1, 32), dtype=np.float32)
        vw = np.zeros((1, 32), dtype=np.float32)
        vx[0, :len(vals)] = vals
        vw[0, :len(vals)] = 1.0
        qx, qw = oracle.e4m3_encode(vx), oracle.e4m3_encode(vw)
        yf, yb = oracle.gemm_e4m3(qx, np.array([sx], np.float32), qw, np.array([sw], np.float32))
        assert yf[0, 0] == acc
        assert Fraction(float(bf16_val(yb)[0, 0])) == want


def test_rmsnorm_single_final_rounding(oracle):
    """The reading adopted for RMSNorm rounds once, after the gain: bf16((x*r)*g).
    The alternative (round x*r to bf16, then multiply by g and round again) gives
    a different value for some gains.  Rows of +-2^-6 make x*r = 1/sqrt(1 +
    eps/c^2) ~ 0.98013, visibly below 1; a gain is searched (in fp64, by exact
    rounding, independent of the oracle) for which the two readings differ with
    a wide margin, and the oracle must give the single-rounding value."""
    c = 2.0 ** -6
    eps32 = float(np.float32(EPS))
    xr = c / math.sqrt(c * c + eps32)            # ~0.98013, not near a bf16 midpoint
    xr_b = float(bf16_val(bf16_of_f64(np.array([xr])))[0])
    chosen = None
    for k in range(128):
        gv = 1.0 + k / 128.0                      # bf16 values in [1, 2)
        single = bf16_of_f64(np.array([xr * gv]))[0]
        double = bf16_of_f64(np.array([xr_b * gv]))[0]
        q = 2.0 ** -7                             # bf16 quantum in [1, 2)
        frac = (xr * gv / q) % 1.0
        if single != double and abs(frac - 0.5) > 0.01:
            chosen = (gv, single, double)
            break
    assert chosen is not None
    gv, single, double = chosen
    X = inputs.bits(inputs.to_bf16(np.full((1, 64), c, dtype=np.float32)))
    g = inputs.bits(inputs.to_bf16(np.full(64, gv, dtype=np.float32)))
    Y = oracle.rmsnorm(X, g, EPS)
    assert np.all(Y == single) and single != double


# --------------------------------------------------------------------------
# log-softmax (lm_head log-probabilities)
# --------------------------------------------------------------------------

def lsm_rows(values) -> np.ndarray:
    """Rows of exact bf16 values (given as floats) -> bf16 bits."""
    a = np.asarray(values, dtype=np.float32)
    bits = (a.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(bf16_val(bits), a, equal_nan=True), "values must be exact in bf16"
    return bits


@pytest.mark.parametrize("V", [1, 2, 8, 1000, 128256])
def test_log_softmax_uniform_row_is_minus_log_v(oracle, V):
    for c in (0.0, 3.5, -1024.0):
        out = oracle.log_softmax(lsm_rows(np.full((1, V), c)))
        assert np.allclose(out, -math.log(V), rtol=0, atol=1e-15 * (abs(c) + math.log(V) + 1))


def test_log_softmax_two_logits_softplus_form(oracle):
    # log p(a) = -log(1 + e^(b - a)), written with log1p of the smaller
    # exponential: independent of the max-shift formulation
    for a, b in [(0.0, 0.0), (1.0, 0.0), (0.0, -7.5), (96.0, 100.0), (-3.25, 2.5)]:
        out = oracle.log_softmax(lsm_rows([[a, b]]))[0]
        hi, lo = max(a, b), min(a, b)
        lse = hi + math.log1p(math.exp(lo - hi))
        assert abs(out[0] - (a - lse)) <= 1e-14 * (1 + abs(lse))
        assert abs(out[1] - (b - lse)) <= 1e-14 * (1 + abs(lse))


def test_log_softmax_large_logits_do_not_overflow(oracle):
    # exp(1000) overflows fp64: the max must be taken out before exp
    out = oracle.log_softmax(lsm_rows([[1000.0, 992.0, -1000.0]]))[0]
    lse = 1000.0 + math.log1p(math.exp(-8.0))
    assert np.all(np.isfinite(out[:2]))
    assert abs(out[0] + (lse - 1000.0)) < 1e-12 and abs(out[1] - (992.0 - lse)) < 1e-12


def test_log_softmax_normalised_and_shift_invariant(oracle):
    rng = np.random.default_rng(11)
    V = 4096
    base = np.clip(np.round(rng.normal(0, 6, size=(4, V))), -32, 31)   # integers: exact in bf16
    out = oracle.log_softmax(lsm_rows(base))
    assert np.all(np.abs(np.exp(out).sum(axis=1) - 1.0) < 1e-12)
    shifted = oracle.log_softmax(lsm_rows(base + 32.0))          # integers 0..63: still exact
    assert np.allclose(shifted, out, rtol=0, atol=1e-12)
    assert np.all(out <= 0)
    # monotone in the logit
    order = np.argsort(base[0], kind="stable")
    assert np.all(np.diff(out[0][order]) >= 0)


def test_log_softmax_infinities_and_nan(oracle):
    out = oracle.log_softmax(lsm_rows([[0.0, -np.inf, 0.0, -np.inf]]))[0]
    assert out[1] == -np.inf and out[3] == -np.inf
    assert abs(out[0] + math.log(2)) < 1e-15 and abs(out[2] + math.log(2)) < 1e-15
    for row in ([np.nan, 0.0, 1.0, 2.0], [np.inf, 0.0, 1.0, 2.0], [-np.inf] * 4):
        assert np.all(np.isnan(oracle.log_softmax(lsm_rows([row]))))


def test_token_logprobs_pick_the_row_value(oracle):
    rng = np.random.default_rng(12)
    x = lsm_rows(np.round(rng.normal(0, 2, size=(5, 300)) * 8) / 8)
    full = oracle.log_softmax(x)
    ids = np.array([0, 299, 17, 150, 3])
    assert np.array_equal(oracle.token_logprobs(x, ids), full[np.arange(5), ids])
    bad = oracle.token_logprobs(x, np.array([-1, 300, 0, 0, 0]))
    assert np.isnan(bad[0]) and np.isnan(bad[1]) and not np.isnan(bad[2])


def test_log_softmax_rows_are_independent(oracle):
    rng = np.random.default_rng(13)
    x = lsm_rows(np.round(rng.normal(0, 2, size=(7, 512)) * 16) / 16)
    full = oracle.log_softmax(x)
    for r in range(7):
        assert np.array_equal(oracle.log_softmax(x[r:r + 1])[0], full[r])


# --------------------------------------------------------------------------
# FP8 (E4M3) with per-row scales
# --------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    """Independent decoding from the format's fields (1 sign, 4 exponent bits
    with bias 7, 3 mantissa bits; S.1111.111 is NaN; exponent 0: subnormal)."""
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return math.nan
    v = m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if s else v


def test_e4m3_hand_derived_codes(oracle):
    # (value, code): 1.0 = 1.000 x 2^0 -> 0.0111.000; 448 = 1.110 x 2^8 -> 0.1111.110; ties go to
    # the even mantissa (1.0625 -> 1.000, 1.1875 -> 1.010); 2^-10 and 3 x 2^-10 are subnormal ties
    cases = [(1.0, 0x38), (448.0, 0x7E), (500.0, 0x7E), (-448.0, 0xFE), (1e30, 0x7E), (-np.inf, 0xFE),
             (0.5, 0x30), (2.0 ** -9, 0x01), (2.0 ** -6, 0x08), (1.0625, 0x38), (1.1875, 0x3A), (-0.0, 0x80),
             (0.0, 0x00), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (240.0, 0x77), (416.0, 0x7D)]
    got = oracle.e4m3_encode([v for v, _ in cases])
    assert [int(g) for g in got] == [c for _, c in cases]
    assert oracle.e4m3_encode([np.nan])[0] == 0x7F


def test_e4m3_decode_matches_the_fields_and_round_trips(oracle):
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.e4m3_decode(codes)
    for c in range(256):
        want = e4m3_value(c)
        if math.isnan(want):
            assert math.isnan(dec[c])
        else:
            assert dec[c] == want and math.copysign(1, dec[c]) == math.copysign(1, want)
    finite = [c for c in range(256) if not math.isnan(e4m3_value(c))]
    assert [int(v) for v in oracle.e4m3_encode(dec[finite])] == finite
    assert np.all(np.diff(dec[:0x7F]) > 0)          # codes 0..0x7E increase with their value
    assert dec[0x7E] == 448.0


def test_e4m3_rounding_is_nearest_even_by_brute_force(oracle):
    rng = np.random.default_rng(31)
    vals = np.concatenate([rng.uniform(-460, 460, 3000), rng.uniform(-0.05, 0.05, 2000)]).astype(np.float32)
    got = oracle.e4m3_encode(vals)
    table = [(c, e4m3_value(c)) for c in range(0x7F)]
    for v, g in zip(vals, got):
        a = abs(float(v))
        if a >= 448:
            want = 0x7E
        else:
            best = min(table, key=lambda cv: (abs(cv[1] - a), cv[0] & 1))
            want = best[0]
        if math.copysign(1, float(v)) < 0:
            want |= 0x80
        assert int(g) == want, (float(v), int(g), want)


def test_quantize_rows_exact_scales(oracle):
    # amax 448 -> scale 1; amax 224 -> scale 0.5 (x / 0.5 is exact); zero row -> scale 1
    rows = np.zeros((4, 16), dtype=np.float32)
    rows[0] = np.linspace(-448, 448, 16).round()
    rows[1] = np.linspace(-224, 224, 16).round()
    rows[3, 5] = np.inf
    bits = (rows.view(np.uint32) >> 16).astype(np.uint16)
    x = bf16_val(bits)
    q, s = oracle.quantize_rows_e4m3(bits)
    assert s[0] == 1.0 and s[1] == 0.5 and s[2] == 1.0 and np.isnan(s[3])
    assert np.array_equal(q[0], oracle.e4m3_encode(x[0]))
    assert np.array_equal(q[1], oracle.e4m3_encode(x[1] * 2))
    assert np.all(q[2] == 0) and np.all(q[3] == 0x7F)
    # the largest magnitude of a row lands on +-448
    rng = np.random.default_rng(32)
    X = inputs.normal((8, 300), std=3.0, seed=33, stream=0)
    q, s = oracle.quantize_rows_e4m3(inputs.bits(X))
    xv = X.float().numpy()
    for r in range(8):
        k = int(np.argmax(np.abs(xv[r])))
        assert q[r, k] & 0x7F == 0x7E
        assert s[r] == np.float32(np.float32(np.abs(xv[r]).max()) / np.float32(448.0))


def test_gemm_e4m3_integer_exact(oracle):
    # small-integer codes: every product and partial sum is an exact integer
    rng = np.random.default_rng(34)
    vx = rng.integers(-8, 9, size=(5, 96)).astype(np.float32)
    vw = rng.integers(-8, 9, size=(7, 96)).astype(np.float32)
    qx, qw = oracle.e4m3_encode(vx), oracle.e4m3_encode(vw)
    sx = np.array([1.0, 0.5, 2.0, 0.25, 4.0], dtype=np.float32)
    sw = np.array([1.0, 2.0, 0.5, 1.0, 0.125, 8.0, 1.0], dtype=np.float32)
    yf, yb = oracle.gemm_e4m3(qx, sx, qw, sw)
    exact = vx.astype(np.int64) @ vw.astype(np.int64).T
    assert np.array_equal(yf, exact.astype(np.float32))
    want = oracle.bf16_rne((exact * sx[:, None] * sw[None, :]).astype(np.float32))
    assert np.array_equal(yb, want)


# --------------------------------------------------------------------------- decode attention

def exact_bits(a) -> np.ndarray:
    """bf16 bit patterns of values that bf16 holds exactly (asserted)."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(bf16_val(bits), f), "value not exact in bf16"
    return bits


def bf16_round_vals(a) -> np.ndarray:
    """Values truncated to bf16 (exact by construction)."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return ((f.view(np.uint32) >> 16) << 16).view(np.float32)


def paged(kd, vd, page_size, order=None, pad_pages=0, fill=0.0):
    """Dense per-request K/V lists ([L_b, Hkv, D] each) -> (k_cache, v_cache,
    block_table, seq_lens) with the pages laid out in `order` (a permutation of
    the page slots; identity when None).  Rows past a request's length in its
    last page, and `pad_pages` unused pages, hold `fill`."""
    Hkv, D = kd[0].shape[1], kd[0].shape[2]
    need = [-(-k.shape[0] // page_size) for k in kd]
    total = sum(need) + pad_pages
    order = np.arange(total) if order is None else np.asarray(order)
    kc = np.full((total, page_size, Hkv, D), fill, dtype=np.float32)
    vc = np.full((total, page_size, Hkv, D), fill, dtype=np.float32)
    bt = np.full((len(kd), max(max(need), 1)), -1, dtype=np.int32)
    slot = 0
    for b, (k, v) in enumerate(zip(kd, vd)):
        for i in range(need[b]):
            pg = int(order[slot])
            slot += 1
            rows = slice(i * page_size, min((i + 1) * page_size, k.shape[0]))
            n = rows.stop - rows.start
            kc[pg, :n], vc[pg, :n] = k[rows], v[rows]
            bt[b, i] = pg
    lens = np.array([k.shape[0] for k in kd], dtype=np.int32)
    return kc, vc, bt, lens


def attn(oracle, q, kd, vd, scale, page_size=4, **kw):
    kc, vc, bt, lens = paged(kd, vd, page_size, **kw)
    finite = np.isfinite(kc) & np.isfinite(vc)
    exact_bits(np.where(finite, kc, 0.0))
    exact_bits(np.where(finite, vc, 0.0))
    kb = (kc.view(np.uint32) >> 16).astype(np.uint16)
    vb = (vc.view(np.uint32) >> 16).astype(np.uint16)
    return oracle.decode_attention(exact_bits(q), kb, vb, bt, lens, scale)


def rand_req(rng, L, Hkv, D, lo=-2.0, hi=2.0):
    return bf16_round_vals(rng.uniform(lo, hi, (L, Hkv, D))), bf16_round_vals(rng.uniform(lo, hi, (L, Hkv, D)))


def test_attention_one_position_gives_its_value_row(oracle):
    rng = np.random.default_rng(50)
    k, v = rand_req(rng, 1, 2, 16)
    q = bf16_round_vals(rng.uniform(-3, 3, (1, 4, 16)))
    out = attn(oracle, q, [k], [v], 0.25)
    for h in range(4):
        assert np.array_equal(out[0, h], v[0, h // 2].astype(np.float64))


def test_attention_equal_keys_or_zero_scale_give_the_mean(oracle):
    rng = np.random.default_rng(51)
    L, D = 7, 8
    v = np.asarray(rng.integers(-50, 51, (L, 1, D)), dtype=np.float32)
    krow = bf16_round_vals(rng.uniform(-1, 1, (1, 1, D)))
    q = bf16_round_vals(rng.uniform(-1, 1, (1, 1, D)))
    mean = np.array([float(sum(Fraction(int(x)) for x in v[:, 0, d]) / L) for d in range(D)])
    out = attn(oracle, q, [np.repeat(krow, L, axis=0)], [v], 0.7)
    assert np.allclose(out[0, 0], mean, rtol=0, atol=1e-12)
    k, _ = rand_req(rng, L, 1, D)
    out = attn(oracle, q, [k], [v], 0.0)
    assert np.allclose(out[0, 0], mean, rtol=0, atol=1e-12)


def test_attention_two_positions_follow_the_logistic_form(oracle):
    # integer q and k make q . k exact; with scale 1/8, s1 - s0 is exact too:
    # out = v0 + (v1 - v0) / (1 + exp(s0 - s1))
    rng = np.random.default_rng(52)
    D = 16
    for trial in range(6):
        q = rng.integers(-3, 4, (1, 1, D)).astype(np.float32)
        k = rng.integers(-3, 4, (2, 1, D)).astype(np.float32)
        v = bf16_round_vals(rng.uniform(-4, 4, (2, 1, D)))
        s = [float(q[0, 0] @ k[p, 0]) / 8 for p in range(2)]
        want = v[0, 0] + (v[1, 0].astype(np.float64) - v[0, 0]) / (1.0 + math.exp(s[0] - s[1]))
        out = attn(oracle, q, [k], [v], 0.125)
        assert np.allclose(out[0, 0], want, rtol=0, atol=1e-13), trial


def test_attention_a_dominant_key_selects_its_value(oracle):
    rng = np.random.default_rng(53)
    L, D = 40, 32
    k, v = rand_req(rng, L, 1, D, -0.5, 0.5)
    q = np.zeros((1, 1, D), dtype=np.float32)
    q[0, 0, 0] = 64.0
    k[:, 0, 0] = 0.0
    k[17, 0, 0] = 2.0                      # s_17 - s_p = 128 * scale = 64 for every other p
    out = attn(oracle, q, [k], [v], 0.5)
    assert np.allclose(out[0, 0], v[17, 0], rtol=0, atol=1e-20)


def test_attention_grouped_query_heads_read_their_group(oracle):
    # consecutive query heads share a key/value head: head h reads group h // (Hq / Hkv)
    rng = np.random.default_rng(54)
    D, L = 8, 5
    for Hq, Hkv in ((8, 2), (8, 4), (6, 3), (4, 1)):
        k, _ = rand_req(rng, L, Hkv, D)
        v = np.zeros((L, Hkv, D), dtype=np.float32)
        for j in range(Hkv):
            v[:, j] = j + 1
        q = bf16_round_vals(rng.uniform(-1, 1, (1, Hq, D)))
        out = attn(oracle, q, [k], [v], 0.3)
        G = Hq // Hkv
        for h in range(Hq):
            assert np.allclose(out[0, h], h // G + 1, rtol=0, atol=1e-14), (Hq, Hkv, h)


def test_attention_page_placement_and_position_order(oracle):
    rng = np.random.default_rng(55)
    D, Hkv, Hq = 16, 2, 4
    lens = [1, 9, 16, 23]
    kd, vd = zip(*[rand_req(rng, L, Hkv, D) for L in lens])
    q = bf16_round_vals(rng.uniform(-2, 2, (len(lens), Hq, D)))
    base = attn(oracle, q, kd, vd, 0.4, page_size=4)
    # the same rows in shuffled pages of another size: the same positions in the same order
    for ps in (1, 4, 8):
        n = sum(-(-L // ps) for L in lens) + 3
        got = attn(oracle, q, kd, vd, 0.4, page_size=ps, order=rng.permutation(n), pad_pages=3)
        assert np.array_equal(got, base), ps
    # permuting a request's positions changes only the rounding order of the sums
    perm = [rng.permutation(L) for L in lens]
    got = attn(oracle, q, [k[p] for k, p in zip(kd, perm)], [v[p] for v, p in zip(vd, perm)], 0.4)
    assert np.allclose(got, base, rtol=0, atol=1e-13)
    # each request is computed from its own rows: dropping the others changes nothing
    for b in range(len(lens)):
        alone = attn(oracle, q[b:b + 1], [kd[b]], [vd[b]], 0.4)
        assert np.array_equal(alone[0], base[b])


def test_attention_is_a_convex_combination(oracle):
    rng = np.random.default_rng(56)
    D, L = 32, 50
    k, v = rand_req(rng, L, 1, D, -3, 3)
    q = bf16_round_vals(rng.uniform(-3, 3, (1, 1, D)))
    out = attn(oracle, q, [k], [v], 1.0)[0, 0]
    assert np.all(out >= v[:, 0].min(axis=0) - 1e-12) and np.all(out <= v[:, 0].max(axis=0) + 1e-12)
    ones = attn(oracle, q, [k], [np.ones_like(v)], 1.0)[0, 0]   # the weights sum to one
    assert np.allclose(ones, 1.0, rtol=0, atol=1e-14)


def test_attention_ignores_cache_rows_past_the_length(oracle):
    rng = np.random.default_rng(57)
    D, Hkv, Hq = 8, 1, 2
    kd, vd = zip(*[rand_req(rng, L, Hkv, D) for L in (3, 6)])
    q = bf16_round_vals(rng.uniform(-2, 2, (2, Hq, D)))
    clean = attn(oracle, q, kd, vd, 0.5, page_size=4)
    for fill in (np.nan, np.inf, 2.0 ** 100):
        dirty = attn(oracle, q, kd, vd, 0.5, page_size=4, pad_pages=2, fill=fill)
        assert np.array_equal(dirty, clean), fill


def test_attention_empty_requests_and_nan_rows(oracle):
    rng = np.random.default_rng(58)
    D, Hkv, Hq = 8, 2, 4
    k, v = rand_req(rng, 5, Hkv, D)
    k[2, 1, 3] = np.nan                                   # a NaN key in group 1 only
    q = bf16_round_vals(rng.uniform(-2, 2, (2, Hq, D)))
    empty_k = np.zeros((0, Hkv, D), dtype=np.float32)
    out = attn(oracle, q, [k, empty_k], [v, empty_k], 0.5)
    assert np.all(np.isfinite(out[0, :2])) and np.all(np.isnan(out[0, 2:]))
    assert np.array_equal(out[1], np.zeros((Hq, D)))


def test_quantize_multiplies_by_the_reciprocal_scale(oracle):
    # amax = 0.8125 = 13/16 and x = -0.3046875 = -39/128: the exact quotient
    # x / (amax / 448) is -168, an E4M3 tie between 160 (mantissa 010) and 176
    # (011).  inv = fl(448 / 0.8125) lies above 551.3846..., so x * inv is just
    # past -168 and rounds to -176 (code 0xF3); fl(amax / 448) lies above
    # 13/7168, so x / scale is just short of -168 and would round to the even
    # -160 (0xF2).  The codes follow the product with the reciprocal.
    inv = np.float32(448.0) / np.float32(0.8125)
    assert float(inv) > 448.0 / 0.8125
    row = np.zeros((1, 16), dtype=np.float32)
    row[0, 0], row[0, 1] = 0.8125, -0.3046875
    bits = (row.view(np.uint32) >> 16).astype(np.uint16)
    q, s = oracle.quantize_rows_e4m3(bits)
    assert s[0] == np.float32(np.float32(0.8125) / np.float32(448.0))
    assert q[0, 0] == 0x7E and q[0, 1] == 0xF3


def test_quantize_subnormal_rows_keep_their_scale(oracle):
    # amax = 9.918e-39 (a subnormal binary32): scale = amax / 448 is the
    # subnormal 2.2139e-41, never 0; inv = 448 / amax overflows and is clamped
    # to the largest finite float, so amax * inv = 3.377... gives E4M3 3.5 (0x45).
    r = np.zeros((1, 16), dtype=np.float32)
    r[0, 0] = 1e-38
    bits = (r.view(np.uint32) >> 16).astype(np.uint16)
    amax = bf16_val(bits)[0, 0]
    q, s = oracle.quantize_rows_e4m3(bits)
    assert s[0] == np.float32(amax) / np.float32(448.0) and s[0] > 0
    assert q[0, 0] == 0x45 and np.all(q[0, 1:] == 0)
