"""The offline pin tuner's host logic (no GPU): grid legality, the additive
per-family cost (Detent, Eq. 3), the search, the delta bound, the recorder
and the JSON table."""
import json

import pytest

from invariant_bi_gemm_bf16_gb300 import binding as bd
from invariant_bi_gemm_bf16_gb300 import tuner


@pytest.fixture(scope="module")
def lib():
    bd.load()
    return bd


@pytest.mark.parametrize("N,K", [(4096, 14336), (6144, 4096), (256, 200), (128, 256)])
def test_legal_grid(lib, N, K):
    grid = tuner.legal_grid(N, K)
    assert grid, "empty grid"
    kt = -(-K // 64)
    for p in grid:
        assert bd.bi_pins_validate(N, K, p) == bd.BI_OK
        assert p.split_k <= kt
    keys = {tuner.key_of(p) for p in grid}
    assert len(keys) == len(grid)
    d = bd.bi_pins_default(N, K)
    assert (d.split_k, d.tok_tile, d.mma_ctas, d.stages, d.flags & bd.BI_FLAG_KTILE_PAIRS) in keys
    # the grid is a function of (N, K) alone: no axis is M
    assert [tuner.key_of(p) for p in tuner.legal_grid(N, K)] == [tuner.key_of(p) for p in grid]


def test_family_cost_is_the_weighted_sum():
    calls = [(1, 3), (32, 2), (512, 1)]
    t = {1: 10.0, 32: 12.0, 512: 40.0}
    assert tuner.family_cost(calls, t.__getitem__) == 3 * 10.0 + 2 * 12.0 + 40.0


def separable_cost(p):
    # a made-up cost, separable over the axes, with a unique optimum
    return ({1: 9, 2: 5, 3: 4, 4: 1, 5: 3, 6: 6, 7: 6.5, 8: 7, 12: 8, 16: 9}[p.split_k] + {128: 2, 256: 0}[p.tok_tile]
            + {0: 0, 1: 1, 2: 3}[p.mma_ctas] + (0 if p.flags & bd.BI_FLAG_KTILE_PAIRS else 0.5)
            + (0 if p.stages == 0 else 0.25))


def test_search_finds_the_optimum_of_a_separable_cost_with_few_measurements(lib):
    N, K = 4096, 14336
    grid = tuner.legal_grid(N, K)
    start = tuner.candidate(N, K, 1, 128, 2, 0, 0)
    best, c, measured = tuner.search(grid, start, separable_cost)
    ebest, ec, emeasured = tuner.exhaustive(grid, separable_cost)
    assert c == ec == separable_cost(ebest)
    assert tuner.key_of(best) == tuner.key_of(ebest)
    assert emeasured == len(grid) and measured < len(grid) // 2


def test_search_never_ends_worse_than_its_start(lib):
    N, K = 6144, 4096
    grid = tuner.legal_grid(N, K)
    start = tuner.candidate(N, K, 3, 256, 0, 0, bd.BI_FLAG_KTILE_PAIRS)

    def bumpy(p):   # not separable: an interaction between S and T
        return (p.split_k - 5) ** 2 * (1 if p.tok_tile == 256 else 3) + (p.mma_ctas == 1) + (p.flags & 1)
    best, c, _ = tuner.search(grid, start, bumpy)
    assert c <= bumpy(start)
    assert bd.bi_pins_validate(N, K, best) == bd.BI_OK


def test_delta_bound_matches_the_pages_example():
    # Detent, Sec. 6: a largest interaction of delta = 1.04% puts the per-family
    # choice within 2.1% of the best tuple.
    assert abs(tuner.delta_bound(0.0104) - 1.021) < 5e-4
    assert tuner.delta_bound(0.0) == 1.0
    with pytest.raises(ValueError):
        tuner.delta_bound(1.0)


def test_measured_delta():
    assert tuner.measured_delta(100.0, 20.0, [50.0, 30.0]) == 0.0
    assert abs(tuner.measured_delta(100.0, 20.0, [50.0, 35.0]) - 0.05) < 1e-12


def test_recorder_counts_calls_per_family(lib):
    rec = tuner.Recorder()
    with rec:
        bd._report(1, 4096, 14336)
        bd._report(1, 4096, 14336)
        bd._report(32, 6144, 4096)
    bd._report(7, 1, 1)   # after the context: not recorded
    assert rec.families() == {(4096, 14336): [(1, 2)], (6144, 4096): [(32, 1)]}


def test_json_round_trip_and_refusals(lib, tmp_path):
    p = bd.bi_pins_default(4096, 14336).replace(split_k=5, mma_ctas=2)
    entry = {"N": 4096, "K": 14336, "calls": [{"M": 1, "n": 1}], "pins": p.as_dict()}
    path = str(tmp_path / "t.json")
    tuner.dump([entry], path, workload="test")
    table = tuner.load(path)
    assert list(table) == [(4096, 14336)] and table[(4096, 14336)].as_dict() == p.as_dict()
    # an illegal tuple refuses the whole table
    bad = dict(entry, pins=p.replace(split_k=0).as_dict())
    tuner.dump([bad], path)
    with pytest.raises(ValueError):
        tuner.load(path)
    tuner.dump([entry, entry], path)
    with pytest.raises(ValueError):
        tuner.load(path)
    with open(path, "w") as f:
        json.dump({"format": "something else", "families": []}, f)
    with pytest.raises(ValueError):
        tuner.load(path)


def test_attention_split_grid_is_the_legal_sizes(lib):
    assert tuner.attn_legal_splits((32, 64, 100, 128, 4096, 8192)) == [64, 128, 4096]
    assert tuner.attn_legal_splits() == list(tuner.ATTN_SPLITS)


def test_tune_attention_takes_the_argmin_and_keeps_the_default_within_the_margin(lib):
    # Detent, Sec. 7: the split stride is tuned like a pin.  A made-up cost per split size.
    costs = {S: 11.0 for S in tuner.ATTN_SPLITS}
    costs.update({64: 10.0, 128: 8.0, 256: 9.0, 448: 5.5, 512: 5.0, 1024: 6.0, 2048: 7.0, 4096: 12.0})
    e = tuner.tune_attention(64, 8, 16, [([100, 200], 1)], timer=costs.__getitem__, repeats=1)
    att = e["attention"]
    assert att["split_size"] == 512 and att["T_us"] == 5.0 and att["T_default_us"] == 9.0
    assert sorted(int(k) for k in att["measured"]) == list(tuner.ATTN_SPLITS)
    near = {S: 10.0 for S in costs}
    near[256], near[512] = 9.0, 8.95   # the best beats the default by less than 1%
    e = tuner.tune_attention(64, 8, 16, [([100], 1)], timer=near.__getitem__, repeats=1)
    assert e["attention"]["split_size"] == bd.BI_ATTN_DEFAULT_SPLIT
    with pytest.raises(ValueError):
        tuner.tune_attention(64, 8, 16, [([100], 1)], splits=(100,), timer=costs.get)


def test_json_round_trip_with_an_attention_entry(lib, tmp_path):
    p = bd.bi_pins_default(4096, 14336)
    gemm = {"N": 4096, "K": 14336, "calls": [{"M": 1, "n": 1}], "pins": p.as_dict()}
    att = {"attention": {"Hq": 64, "Hkv": 8, "page_size": 16, "split_size": 512}}
    path = str(tmp_path / "t.json")
    tuner.dump([gemm, att], path)
    table = tuner.load(path)
    assert table[("attention", 64, 8, 16)] == 512 and table[(4096, 14336)].as_dict() == p.as_dict()
    for bad in (100, 8192, 0):
        tuner.dump([{"attention": dict(att["attention"], split_size=bad)}], path)
        with pytest.raises(ValueError):
            tuner.load(path)
    tuner.dump([att, att], path)
    with pytest.raises(ValueError):
        tuner.load(path)
