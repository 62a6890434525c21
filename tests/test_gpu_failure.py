"""Failure detection without a GPU fault.

Every wait in the GEMM kernel is bounded.  The diagnostic flag
BI_FLAG_DEBUG_STALL_PRODUCER makes the W producer withhold its first copy, so
the tensor-core warp's wait runs out (about 2 s); the kernel then records
BI_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees tensor memory and
returns.  The host reads the status; the context stays usable for the next call.
Illegal pins are refused on the host before any launch (Detent, Sec. 5: a
failed legality check stops execution before a kernel runs)."""
import pytest
import torch

from invariant_bi_gemm_bf16_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ctas", [1, 2])
@pytest.mark.parametrize("schedule", ["local", "cluster"])
def test_stalled_producer_reports_timeout_and_recovers(lib, ctas, schedule):
    M, N, K = 3, 128, 256
    x = inputs.normal((M, K), seed=0, stream=0).cuda()
    w = inputs.normal((N, K), std=0.02, seed=0, stream=1).cuda()
    flags = lib.BI_FLAG_SCHEDULE_LOCAL if schedule == "local" else lib.BI_FLAG_SCHEDULE_CLUSTER
    pins = lib.bi_pins_default(N, K).replace(split_k=2, tok_tile=128, mma_ctas=ctas, flags=flags)
    assert lib.bi_last_device_status() == lib.BI_OK           # clean start
    lib.bi_gemm_bf16(x, w, pins=pins.replace(flags=flags | lib.BI_FLAG_DEBUG_STALL_PRODUCER))
    assert lib.bi_last_device_status() == lib.BI_ERR_DEVICE_TIMEOUT
    # the status was cleared and the context still works
    assert lib.bi_last_device_status() == lib.BI_OK
    y = lib.bi_gemm_bf16(x, w, pins=pins)
    torch.cuda.synchronize()
    ref = lib.bi_gemm_bf16(x, w, pins=pins.replace(flags=0))
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    assert lib.bi_last_device_status() == lib.BI_OK


def test_illegal_pins_launch_nothing(lib):
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.full((4, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    for bad in (dict(split_k=0), dict(tok_tile=100), dict(mma_ctas=3), dict(bk=128), dict(flags=0x8000)):
        with pytest.raises(lib.BiError) as e:
            lib.bi_gemm_bf16(x, w, out=y, pins=lib.bi_pins_default(128, 256).replace(**bad))
        assert e.value.status == lib.BI_ERR_ILLEGAL_PINS
    torch.cuda.synchronize()
    assert torch.all(y.float() == 3.0)
    assert lib.bi_last_device_status() == lib.BI_OK
