"""Failure detection on the GPU without faulting it: a bounded wait that
runs out reports MOE_ERR_TIMEOUT through the status word and leaves the
context usable; bad arguments are refused on the host."""
import time

import pytest
import torch

import routing_grouped_expert_gb300 as moe
from routing_grouped_expert_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    ws = moe.Workspace()
    ws.ensure(4096)
    t0 = time.perf_counter()
    moe.moe_diag_wait_timeout(ws, 20_000_000)          # 20 ms
    assert moe.moe_get_device_status(ws) == 3          # MOE_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    # the context still works and the next call clears the status
    wl = I.small("after_timeout", T=64, H=128, F=256, E=4, k=2)
    d = {n: t.cuda() for n, t in I.make_inputs(wl, "cpu").items()}
    out = moe.moe_forward(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], 2, ws=ws)
    assert moe.moe_get_device_status(ws) == 0
    assert torch.isfinite(out.float()).all()


def test_block_counter_wait_that_runs_out_reports_timeout():
    """The wait FC2 uses for a token block's FC1 tiles, on a counter nothing
    increments: MOE_ERR_TIMEOUT after the limit, and the context still works
    (the overlapped forward right after it is correct and reports OK)."""
    ws = moe.Workspace()
    ws.ensure(4096)
    t0 = time.perf_counter()
    moe.moe_diag_count_wait_timeout(ws, 20_000_000)    # 20 ms
    assert moe.moe_get_device_status(ws) == 3          # MOE_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    wl = I.small("after_count_timeout", T=600, H=256, F=512, E=2, k=2)
    d = {n: t.cuda() for n, t in I.make_inputs(wl, "cpu").items()}
    out = moe.moe_forward(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], 2, ws=ws)
    assert moe.moe_get_device_status(ws) == 0
    assert torch.isfinite(out.float()).all()


def test_bad_arguments_raise_on_the_host():
    ws = moe.Workspace()
    ws.ensure(4096)
    with pytest.raises(moe.MoeError):
        moe.moe_diag_wait_timeout(ws, 10)                          # limit below 1 ms
    x = torch.zeros(8, 100, dtype=torch.bfloat16, device="cuda")   # H not a multiple of 128
    W = torch.zeros(2, 100, 128, dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros(2, 128, 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_forward(x, torch.zeros(8, 2, device="cuda"), W, W, W2, 1)
