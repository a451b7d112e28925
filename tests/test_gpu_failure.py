"""Failure detection on the GPU without a fault: a pipeline wait that runs out
gives up after its limit, reports MOE_DEV_TIMEOUT through the device status word,
and leaves the CUDA context usable for the next call."""

import time

import pytest
import torch

import ragged_grouped_gemm_topk_gb300 as moe_gpu
from _parity import need_gpu

pytestmark = pytest.mark.gpu

MOE_DEV_TIMEOUT = 4   # include/moe.h


@pytest.mark.parametrize("limit_us", [1000, 20000])
def test_bounded_wait_reports_timeout_and_context_survives(limit_us):
    need_gpu()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = moe_gpu.binding.moe_check_wait_timeout(limit_us)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) & MOE_DEV_TIMEOUT
    assert limit_us * 1e-6 <= dt < limit_us * 1e-6 + 5.0
    # the context still works: routing after the timeout is exact
    lg = torch.randn(64, 8, device="cuda")
    idx, w, counts = moe_gpu.moe_route_topk(lg, 2)
    assert int(counts.sum().item()) == 128
    assert torch.equal(idx[:, 0].long(), lg.argmax(dim=1))


def test_status_word_accumulates_flags():
    need_gpu()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe_gpu.binding.moe_check_wait_timeout(1000, dev_status=st)
    moe_gpu.binding.moe_check_wait_timeout(1000, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == MOE_DEV_TIMEOUT          # OR-ed, not added
