"""Decode attention over a paged cache on the GPU: parity with the fp64 oracle
within a bound derived from the kernel's arithmetic, bitwise batch
invariance, the split-size pin, and the edge cases.

Tolerance (the pages give none; derived from the tree the kernel runs):
  * the weights p are rounded to bf16 (relative error <= 2^-9) and the same
    rounded values are summed into l, so out = sum w'_p v_p with w' a convex
    weight vector whose entries are off by a factor (1 + e_p), |e_p| <= eps_w;
    then |out' - out| <= 2 eps_w max_p |v_p - out| / (1 - eps_w);
  * eps_w also carries the score error: fp32 accumulation of q . k over D
    (at most (D + 3) 2^-24 sum_d |q_d k_d| after scaling by scale * log2 e)
    times ln 2, twice (the score and the maximum), and exp2f's 2 ulp;
  * the fp32 sums of o and l over n = L + 16 terms add 2 gamma_n max_p |v_p|;
  * the output rounding adds half a bf16 ulp.
The relative Frobenius error over a case must also stay below 2^-9 + 2^-10
(the output rounding alone reaches 2^-9 relative per element)."""
import math

import numpy as np
import pytest
import torch

from helpers import bf16_bits, bits_to_f64, ulp_bf16
from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu

D = 128
U = 2.0 ** -24


def dense(kc, vc, bt, lens, b):
    """Request b's keys and values [L, Hkv, D] gathered from its pages."""
    L = int(lens[b])
    P = kc.shape[1]
    pos = np.arange(L)
    pages = bt[b, pos // P].astype(np.int64)
    return kc[pages, pos % P], vc[pages, pos % P]


def head_tolerance(ref, got, q, k, v, scale):
    """Bound [D] for one query head: q [D], k and v [L, D] (fp64), L > 0."""
    L = k.shape[0]
    s_abs = scale * np.max(np.abs(k) @ np.abs(q))
    dt = (D + 3) * U * s_abs * math.log2(math.e)
    eps_w = 2.0 ** -9 + 2 * math.log(2) * dt + 2.0 ** -22
    n = L + 16
    gam = n * U / (1 - n * U)
    dev = np.max(np.abs(v - ref[None, :]), axis=0)
    big = np.maximum(np.abs(ref), np.abs(np.nan_to_num(got)))
    return (2 * eps_w / (1 - eps_w)) * dev + 2 * gam * np.max(np.abs(v), axis=0) + 0.5 * ulp_bf16(big)


def tolerance(ref, got, q, kc, vc, bt, lens, scale):
    """Per-element bound [B, Hq, D] (see the module docstring)."""
    B, Hq, _ = ref.shape
    G = Hq // kc.shape[2]
    tol = 0.5 * ulp_bf16(np.maximum(np.abs(ref), np.abs(np.nan_to_num(got))))
    for b in range(B):
        if int(lens[b]) == 0:
            continue
        k, v = dense(kc, vc, bt, lens, b)
        for h in range(Hq):
            tol[b, h] = head_tolerance(ref[b, h], got[b, h], q[b, h], k[:, h // G], v[:, h // G], scale)
    return tol


def f64(t):
    return bits_to_f64(bf16_bits(t))


def run(lib, q, kc, vc, bt, lens, scale, **kw):
    return lib.bi_decode_attention_bf16(q.cuda(), kc.cuda(), vc.cuda(), bt.cuda(), lens.cuda(), scale, **kw)


def check(lib, oracle, q, kc, vc, bt, lens, scale, what, **kw):
    got_t = run(lib, q, kc, vc, bt, lens, scale, **kw)
    assert lib.bi_last_device_status() == lib.BI_OK
    got = f64(got_t)
    ref = oracle.decode_attention(inputs.bits(q), inputs.bits(kc), inputs.bits(vc), bt.numpy(), lens.numpy(), scale)
    qf, kf, vf = f64(q), f64(kc), f64(vc)
    tol = tolerance(ref, got, qf, kf, vf, bt.numpy(), lens.numpy(), scale)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    assert not bad.any(), "%s: %d elements out of bound, worst %s" % (
        what, int(bad.sum()), np.unravel_index(np.argmax(np.where(bad, err - tol, -1)), err.shape))
    live = np.asarray(lens.numpy() > 0)
    if live.any():
        fro = np.linalg.norm((got - ref)[live]) / max(np.linalg.norm(ref[live]), 1e-30)
        assert fro <= 2.0 ** -9 + 2.0 ** -10, (what, fro)
    return got_t


CASES = [
    # (lens, Hq, Hkv, page_size, split_size, q_std)
    ([1, 17, 63, 64, 65, 300, 1000, 2049], 32, 8, 16, 256, 1.0),    # Llama-3.1-8B heads
    ([5, 640, 1500, 3000], 16, 2, 64, 128, 1.0),                      # groups of 8
    ([7, 129, 2500], 32, 2, 8, 64, 1.0),                              # groups of 16
    ([200, 1111], 4, 4, 128, 512, 1.0),                               # one head per group
    ([90, 700], 10, 2, 32, 192, 1.0),                                 # groups of 5
    ([33, 4097], 16, 2, 16, 4096, 1.0),                               # the largest split
    ([513, 2000], 16, 2, 16, 256, 6.0),                               # peaked softmax
    ([1, 2, 3], 16, 2, 256, 256, 1.0),                                # tiny contexts, big pages
    # more (request, head) pairs than SMs: the combine takes whole records
    ([(37 * i) % 401 for i in range(100)], 32, 2, 16, 64, 1.0),      # groups of 16, 100 requests
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_attention_parity(lib, oracle, case):
    lens, Hq, Hkv, P, S, q_std = CASES[case]
    kc, vc, bt, sl = inputs.paged_kv(lens, Hkv, D, P, seed=60 + case, spare_pages=3)
    q = inputs.normal((len(lens), Hq, D), std=q_std, seed=60 + case, stream=0)
    check(lib, oracle, q, kc, vc, bt, sl, 1 / math.sqrt(D), "case %d" % case, split_size=S)


def test_attention_single_position_returns_the_value_bits(lib):
    # one position: p = 1 exactly, o = 1 * v exactly, o / l = v
    kc, vc, bt, sl = inputs.paged_kv([1, 1, 1], 2, D, 16, seed=61)
    q = inputs.normal((3, 8, D), seed=61, stream=0)
    got = bf16_bits(run(lib, q, kc, vc, bt, sl, 0.3))
    vb = inputs.bits(vc)
    for b in range(3):
        for h in range(8):
            assert np.array_equal(got[b, h], vb[int(bt[b, 0]), 0, h // 4])


def test_attention_batch_invariance(lib):
    """A request's bits do not depend on the other requests, their number or
    lengths, its row in the batch, where its pages sit, or the call's length
    bound."""
    Hq, Hkv, P, S = 32, 8, 16, 256
    target = [777, 1, 2048, 300]
    rng = np.random.default_rng(62)
    kc, vc, bt, sl = inputs.paged_kv(target, Hkv, D, P, seed=62)
    q = inputs.normal((len(target), Hq, D), seed=62, stream=0)
    base = bf16_bits(run(lib, q, kc, vc, bt, sl, 0.0883, split_size=S))
    for r in range(len(target)):
        alone = bf16_bits(run(lib, q[r:r + 1], kc, vc, bt[r:r + 1], sl[r:r + 1], 0.0883, split_size=S))
        assert np.array_equal(alone[0], base[r])
    # a larger bound on the lengths (a larger grid) and a padded block table
    big_bt = torch.full((len(target), 400), -1, dtype=torch.int32)
    big_bt[:, :bt.shape[1]] = bt
    got = bf16_bits(run(lib, q, kc, vc, big_bt, sl, 0.0883, split_size=S, max_seq_len=6000))
    assert np.array_equal(got, base)
    # in batches of co-runners of other lengths, at random rows, with the
    # cache re-laid out in other pages
    for trial, batch in enumerate((8, 33, 128)):
        co = [int(x) for x in rng.integers(0, 5000, size=batch - len(target))]
        pos = np.sort(rng.choice(batch, size=len(target), replace=False))
        lens = list(co)
        for i, p in enumerate(pos):
            lens.insert(int(p), target[i])
        kc2, vc2, bt2, sl2 = inputs.paged_kv(lens, Hkv, D, P, seed=100 + trial, spare_pages=5)
        q2 = inputs.normal((batch, Hq, D), seed=100 + trial, stream=0)
        for i, p in enumerate(pos):
            # copy the target's data into its new pages and query row
            n = -(-target[i] // P)
            for j in range(n):
                kc2[int(bt2[p, j])] = kc[int(bt[i, j])]
                vc2[int(bt2[p, j])] = vc[int(bt[i, j])]
            q2[p] = q[i]
        got = bf16_bits(run(lib, q2, kc2, vc2, bt2, sl2, 0.0883, split_size=S))
        for i, p in enumerate(pos):
            assert np.array_equal(got[p], base[i]), (batch, i)


def test_attention_workspace_needs_no_initial_contents(lib):
    """Each call rewrites its control words, item list and records: a
    workspace full of garbage, or left over from another shape, gives the
    same bits."""
    kc, vc, bt, sl = inputs.paged_kv([300, 1, 700], 2, D, 16, seed=67)
    q = inputs.normal((3, 8, D), seed=67, stream=0)
    base = bf16_bits(run(lib, q, kc, vc, bt, sl, 0.0883, split_size=64))
    need = lib.bi_decode_attention_workspace_bytes(3, 8, 2, bt.shape[1] * 16, 64)
    for fill in (0xFF, 0x00, 0x7F):
        ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
        got = bf16_bits(run(lib, q, kc, vc, bt, sl, 0.0883, split_size=64, workspace=ws))
        assert np.array_equal(got, base), fill
        # the same workspace again, after a call of another shape
        run(lib, q[:1], kc, vc, bt[:1], sl[:1], 0.0883, split_size=64, workspace=ws)
        assert np.array_equal(bf16_bits(run(lib, q, kc, vc, bt, sl, 0.0883, split_size=64, workspace=ws)), base)


def test_attention_split_size_is_a_pin(lib, oracle):
    """Another split size is another tree: other bits, each within the bound."""
    lens = [3000, 1025]
    kc, vc, bt, sl = inputs.paged_kv(lens, 2, D, 16, seed=63)
    q = inputs.normal((2, 16, D), seed=63, stream=0)
    outs = {}
    for S in (64, 256, 1024):
        outs[S] = bf16_bits(check(lib, oracle, q, kc, vc, bt, sl, 0.0883, "split %d" % S, split_size=S))
    assert not np.array_equal(outs[64], outs[1024])


def test_attention_empty_and_nan(lib):
    kc, vc, bt, sl = inputs.paged_kv([0, 40, 0, 100], 2, D, 16, seed=64, stale=np.nan)
    # a NaN key inside request 1's context, in key/value head 1 only
    kc[int(bt[1, 1]), 3, 1, 7] = float("nan")
    q = inputs.normal((4, 8, D), seed=64, stream=0)
    got = run(lib, q, kc, vc, bt, sl, 0.0883).float().cpu().numpy()
    assert lib.bi_last_device_status() == lib.BI_OK
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert np.all(np.isfinite(got[1, :4])) and np.all(np.isnan(got[1, 4:]))
    assert np.all(np.isfinite(got[3]))


def test_attention_device_side_checks_report_and_recover(lib):
    kc, vc, bt, sl = inputs.paged_kv([50, 60], 2, D, 16, seed=65)
    q = inputs.normal((2, 8, D), seed=65, stream=0)
    assert lib.bi_last_device_status() == lib.BI_OK
    # a length above the call's bound: flagged, that request's output is NaN
    bad = sl.clone()
    bad[1] = 70
    out = run(lib, q, kc, vc, bt, bad, 0.0883, max_seq_len=64)
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_ERR_INVALID_ARG
    assert torch.isnan(out[1].float()).all()
    # a page id outside the cache: flagged (the page reads as zeros)
    bt2 = bt.clone()
    bt2[0, 1] = kc.shape[0] + 7
    run(lib, q, kc, vc, bt2, sl, 0.0883)
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_ERR_INVALID_ARG
    # the context is still usable, and a correct call reports OK again
    good = bf16_bits(run(lib, q, kc, vc, bt, sl, 0.0883))
    assert lib.bi_last_device_status() == lib.BI_OK
    assert np.array_equal(good, bf16_bits(run(lib, q, kc, vc, bt, sl, 0.0883)))


def test_attention_full_size_sampled(lib, oracle):
    """The benchmark's workload (Llama-3.1-70B heads: 64 query heads, 8
    key/value heads; 64 requests with lengths uniform on [512, 8192]; pages
    of 16 in shuffled order) in the benchmark's launch configuration, checked
    on sampled (request, head) rows against the oracle."""
    rng = np.random.default_rng(66)
    lens = [int(x) for x in rng.integers(512, 8193, size=64)]
    Hq, Hkv, P = 64, 8, 16
    kc, vc, bt, sl = inputs.device_paged_kv(lens, Hkv, D, P, seed=66)
    q = inputs.device_normal((64, Hq, D), seed=66, stream=0)
    out = lib.bi_decode_attention_bf16(q, kc, vc, bt, sl, 1 / math.sqrt(D))
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_OK
    pairs = np.stack([rng.integers(0, 64, size=48), rng.integers(0, Hq, size=48)], axis=1)
    pairs[0] = (int(np.argmax(lens)), 0)
    ref = oracle.decode_attention(inputs.bits(q.cpu()), inputs.bits(kc.cpu()), inputs.bits(vc.cpu()),
                                  bt.cpu().numpy(), sl.cpu().numpy(), 1 / math.sqrt(D), pairs=pairs)
    got = f64(out)[pairs[:, 0], pairs[:, 1]]
    qf = f64(q)
    for i, (b, h) in enumerate(pairs):
        L, kvh = lens[b], h // 8
        pos = torch.arange(L, device="cuda")
        pages = bt[b].long()[pos // P]
        k = f64(kc[pages, pos % P, kvh])
        v = f64(vc[pages, pos % P, kvh])
        tol = head_tolerance(ref[i], got[i], qf[b, h], k, v, 1 / math.sqrt(D))
        assert np.all(np.abs(got[i] - ref[i]) <= tol), (b, h)


def test_attention_one_long_request(lib, oracle):
    """The benchmark's long-context workload (one request of 32768 positions,
    Llama-3.1-70B heads, pages of 16 in shuffled order) at split 512: few
    requests take the static schedule, and their warps share the CTA's stage
    pool.  Sampled heads against the oracle; and the request's bits are those
    it gets at row 5 of 12 requests (ticket schedule, two stages per warp,
    its pages re-laid out)."""
    L, Hq, Hkv, P, S = 32768, 64, 8, 16, 512
    kc, vc, bt, sl = inputs.device_paged_kv([L], Hkv, D, P, seed=68)
    q = inputs.device_normal((1, Hq, D), seed=68, stream=0)
    alone = lib.bi_decode_attention_bf16(q, kc, vc, bt, sl, 1 / math.sqrt(D), split_size=S)
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_OK
    heads = [0, 7, 8, 31, 63]
    pairs = np.array([[0, h] for h in heads])
    ref = oracle.decode_attention(inputs.bits(q.cpu()), inputs.bits(kc.cpu()), inputs.bits(vc.cpu()),
                                  bt.cpu().numpy(), sl.cpu().numpy(), 1 / math.sqrt(D), pairs=pairs)
    got = f64(alone)[0, heads]
    qf = f64(q)
    pos = torch.arange(L, device="cuda")
    pages = bt[0].long()[pos // P]
    for i, h in enumerate(heads):
        k = f64(kc[pages, pos % P, h // 8])
        v = f64(vc[pages, pos % P, h // 8])
        tol = head_tolerance(ref[i], got[i], qf[0, h], k, v, 1 / math.sqrt(D))
        assert np.all(np.abs(got[i] - ref[i]) <= tol), h
    # the same request among eleven others
    lens = [300, 4000, 17, 900, 2500, L, 64, 1, 700, 5000, 128, 3333]
    kc2, vc2, bt2, sl2 = inputs.device_paged_kv(lens, Hkv, D, P, seed=69)
    n = L // P
    kc2[bt2[5, :n].long()] = kc[bt[0, :n].long()]
    vc2[bt2[5, :n].long()] = vc[bt[0, :n].long()]
    q2 = inputs.device_normal((len(lens), Hq, D), seed=69, stream=0)
    q2[5] = q[0]
    batch = lib.bi_decode_attention_bf16(q2, kc2, vc2, bt2, sl2, 1 / math.sqrt(D), split_size=S)
    torch.cuda.synchronize()
    assert lib.bi_last_device_status() == lib.BI_OK
    assert np.array_equal(bf16_bits(batch)[5], bf16_bits(alone)[0])
