"""The pin tuner on the GPU: a small family tuned exhaustively gives a legal
tuple, no slower than the default beyond timing noise, and the tuned tuple is
as batch-invariant as any other (a row's bits do not depend on M)."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits
from invariant_bi_gemm_bf16_gb300 import binding as bd
from invariant_bi_gemm_bf16_gb300 import inputs, tuner

pytestmark = pytest.mark.gpu


def test_tune_small_family_exhaustive(lib, tmp_path):
    N, K = 512, 2048
    calls = [(1, 3), (40, 1), (300, 1)]
    e = tuner.tune_family(N, K, calls, mode="exhaustive", reps=3)
    assert e["measured"] == e["legal"] > 10
    pins = bd.Pins(**e["pins"])
    assert bd.bi_pins_validate(N, K, pins) == bd.BI_OK
    assert e["T_us"] <= e["T_default_us"] * 1.05
    path = str(tmp_path / "t.json")
    tuner.dump([e], path, workload="test")
    assert tuner.load(path)[(N, K)].as_dict() == pins.as_dict()
    # the tuned tuple's rows are the same alone and inside a batch
    X = inputs.normal((300, K), seed=4, stream=0).cuda()
    W = inputs.normal((N, K), std=0.02, seed=4, stream=1).cuda()
    full = bf16_bits(bd.bi_gemm_bf16(X, W, pins=pins))
    for r in (0, 41, 299):
        alone = bf16_bits(bd.bi_gemm_bf16(X[r:r + 1].contiguous(), W, pins=pins))
        assert np.array_equal(alone[0], full[r])


def test_search_measures_part_of_the_grid(lib):
    N, K = 1024, 4096
    e = tuner.tune_family(N, K, [(1, 1), (256, 1)], mode="search", reps=3)
    assert e["measured"] < e["legal"]
    assert e["T_us"] <= e["T_default_us"] * 1.05


def test_tune_attention_on_the_gpu(lib, tmp_path):
    """A small decode-attention family tuned on the GPU: every legal split
    size measured, a legal choice, and a table that loads."""
    from invariant_bi_gemm_bf16_gb300 import tuner
    calls = [([300, 1000, 77], 2), ([2000], 1)]
    e = tuner.tune_attention(16, 2, 16, calls, splits=(128, 256, 512))
    att = e["attention"]
    assert att["split_size"] in (128, 256, 512)
    assert set(att["measured"]) == {"128", "256", "512"} and all(v > 0 for v in att["measured"].values())
    path = str(tmp_path / "a.json")
    tuner.dump([e], path)
    assert tuner.load(path) == {("attention", 16, 2, 16): att["split_size"]}
