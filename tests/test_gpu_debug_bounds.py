"""The debug-bounds build (libbi_gemm_debug.so, compiled with -DBI_DEBUG_BOUNDS).

Its GEMM and decode-attention kernels check, before each access, the tile
coordinates of every copy (W and X rows, K tiles), the ring stage, the
tensor-memory columns of every accumulator, the fold workspace's partial and
counter indices, the CLUSTER fold's partial tile, and decode attention's
stages, items and split records.  A failed check skips the access and records
BI_ERR_DEBUG_BOUNDS (it never traps).

On the small invariance shapes (X [M, 256], W [128, 256], M in 1, 3, 7, 16,
33) and a few more that reach every schedule (LOCAL single CTAs and pairs,
CLUSTER, GLOBAL, several token tiles, both forms of the fused layer, FP8),
and on a small decode-attention batch, no check fails and every output has
the bits of the ordinary build."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# The same calls run in both builds; each returns a dict of named outputs.
CASES = r'''
import torch
from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs

def run_cases():
    out = {}
    dev = torch.device("cuda")
    for M in (1, 3, 7, 16, 33):          # the tiny invariance shapes
        x = inputs.normal((M, 256), seed=M, stream=0).cuda()
        w = inputs.normal((128, 256), std=0.02, seed=M, stream=1).cuda()
        out["tiny_M%d" % M] = bd.bi_gemm_bf16(x, w)
        g = inputs.normal((256,), std=0.1, mean=1.0, seed=M, stream=2).cuda()
        out["rms_M%d" % M] = bd.bi_rmsnorm_bf16(x, g, 1e-5)
    for (M, N, K, S, sched) in [(33, 640, 1024, 2, bd.BI_FLAG_SCHEDULE_CLUSTER),
                                (33, 640, 1024, 3, bd.BI_FLAG_SCHEDULE_GLOBAL),
                                (5, 640, 1024, 3, bd.BI_FLAG_SCHEDULE_LOCAL),
                                (300, 512, 2048, 2, 0),
                                (700, 384, 512, 1, 0)]:
        x = inputs.normal((M, K), seed=N + M, stream=0).cuda()
        w = inputs.normal((N, K), std=0.02, seed=N + M, stream=1).cuda()
        base = bd.bi_pins_default(N, K).replace(split_k=S)
        pins = base.replace(flags=base.flags | sched) if sched else base
        ws = torch.zeros(max(bd.bi_gemm_bf16_workspace_bytes(M, N, K, pins), 256), dtype=torch.uint8, device=dev)
        out["gemm_%d_%d_%d_S%d_%d" % (M, N, K, S, sched)] = bd.bi_gemm_bf16(x, w, pins=pins, workspace=ws)
    M, N, K = 5, 256, 512
    x = inputs.normal((M, K), seed=9, stream=0).cuda()
    w = inputs.normal((N, K), std=0.02, seed=9, stream=1).cuda()
    g = inputs.normal((K,), std=0.1, mean=1.0, seed=9, stream=2).cuda()
    p = bd.bi_pins_default(N, K)
    out["fused_staged"] = bd.bi_rmsnorm_gemm_bf16(x, g, w, 1e-5, pins=p)
    out["fused_smem"] = bd.bi_rmsnorm_gemm_bf16(x, g, w, 1e-5, pins=p.replace(flags=p.flags | bd.BI_FLAG_NORM_SMEM))
    xq = inputs.normal((40, 512), seed=10, stream=0).cuda()
    wq = inputs.normal((256, 512), std=0.02, seed=10, stream=1).cuda()
    q, sx = bd.bi_quantize_rows_e4m3(xq)
    qw, sw = bd.bi_quantize_rows_e4m3(wq)
    out["fp8"] = bd.bi_gemm_fp8(q, sx, qw, sw)
    lens = [1, 17, 300]
    kc, vc, bt, sl = inputs.paged_kv(lens, 2, 128, 16, seed=11)
    qa = inputs.normal((3, 16, 128), seed=11, stream=0)
    out["attn"] = bd.bi_decode_attention_bf16(qa.cuda(), kc.cuda(), vc.cuda(), bt.cuda(), sl.cuda(), 0.0883,
                                              split_size=64)
    torch.cuda.synchronize()
    return out
'''

CHILD = r'''
import json, sys, torch
sys.path.insert(0, sys.argv[1])
exec(open(sys.argv[2]).read())
from invariant_bi_gemm_bf16_gb300 import binding as bd
bd.load()
res = {"enabled": bd.bi_debug_bounds_enabled()}
out = run_cases()
res["status"] = bd.bi_last_device_status()
res["detail"] = bd.bi_debug_bounds_detail()
torch.save({k: v.cpu() for k, v in out.items()}, sys.argv[3])
print(json.dumps(res))
'''


def test_debug_bounds_build_runs_clean_with_the_same_bits(lib, tmp_path):
    from invariant_bi_gemm_bf16_gb300 import build
    dbg = build.build(debug=True)
    assert os.path.exists(dbg) and dbg != build.LIB
    cases = tmp_path / "cases.py"
    cases.write_text(CASES)
    child = tmp_path / "child.py"
    child.write_text(CHILD)
    got_path = tmp_path / "debug_out.pt"
    env = dict(os.environ, BI_GEMM_LIB=dbg)
    r = subprocess.run([sys.executable, str(child), ROOT, str(cases), str(got_path)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["enabled"] is True
    assert res["detail"] == 0, "check %d failed with value %d" % (res["detail"] >> 48, res["detail"] & (2**48 - 1))
    assert res["status"] == lib.BI_OK
    # the ordinary build, here
    assert not lib.bi_debug_bounds_enabled()
    scope = {}
    exec(CASES, scope)
    ref = scope["run_cases"]()
    got = torch.load(got_path)
    assert set(got) == set(ref)
    for k, v in ref.items():
        a, b = v.cpu(), got[k]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        elif a.dtype == torch.float32:
            a, b = a.view(torch.int32), b.view(torch.int32)
        assert torch.equal(a, b), k
    assert lib.bi_last_device_status() == lib.BI_OK


POKE_CHILD = r'''
import json, os, sys, torch
sys.path.insert(0, sys.argv[1])
from invariant_bi_gemm_bf16_gb300 import binding as bd, inputs
bd.load()
x = inputs.normal((3, 256), seed=3, stream=0).cuda()
w = inputs.normal((128, 256), std=0.02, seed=3, stream=1).cuda()
res = {}
os.environ["BI_DEBUG_POKE"] = "wrow"       # the first W copy of each CTA aimed past the tile grid
bd.bi_gemm_bf16(x, w)
res["poked_status"] = bd.bi_last_device_status()
res["poked_detail"] = bd.bi_debug_bounds_detail()
del os.environ["BI_DEBUG_POKE"]
y = bd.bi_gemm_bf16(x, w)
res["clean_status"] = bd.bi_last_device_status()
res["clean_detail"] = bd.bi_debug_bounds_detail()
torch.save(y.cpu(), sys.argv[2])
print(json.dumps(res))
'''


def test_debug_bounds_check_reports_and_recovers(lib, tmp_path):
    """Negative control: in the debug-bounds build, a W copy aimed past the tile
    grid (planted by the host of that build only) is caught by the kernel's
    own row check: the copy is skipped, the call reports BI_ERR_DEBUG_BOUNDS
    with the check number of the W row and the offending row, the kernel gives
    up through its bounded waits, and the next call runs clean with the
    ordinary bits."""
    from invariant_bi_gemm_bf16_gb300 import build, inputs
    dbg = build.build(debug=True)
    child = tmp_path / "poke.py"
    child.write_text(POKE_CHILD)
    out = tmp_path / "clean.pt"
    env = dict(os.environ, BI_GEMM_LIB=dbg)
    env.pop("BI_DEBUG_POKE", None)
    r = subprocess.run([sys.executable, str(child), ROOT, str(out)], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["poked_status"] == lib.BI_ERR_DEBUG_BOUNDS
    assert res["poked_detail"] >> 48 == 4                       # the W-row check
    assert res["poked_detail"] & (2 ** 48 - 1) >= 1 << 24       # the planted row
    assert res["clean_status"] == lib.BI_OK and res["clean_detail"] == 0
    x = inputs.normal((3, 256), seed=3, stream=0).cuda()
    w = inputs.normal((128, 256), std=0.02, seed=3, stream=1).cuda()
    ref = lib.bi_gemm_bf16(x, w).cpu()
    assert torch.equal(torch.load(out).view(torch.int16), ref.view(torch.int16))
