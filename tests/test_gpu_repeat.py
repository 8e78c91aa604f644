"""The layer run many times on one workspace gives the same bits every time
and a clean device status: exercises, under repetition, the cross-CTA
protocols of the fast paths -- the CTA pairs' cross-SM barriers and remote
arrivals (fine-grained FC1), the ticket counter of the one-launch small-batch
routing (tiny, decode), FC2's per-block waits on FC1 and the tile queue."""
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from routing_grouped_expert_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,n,every", [("fine_grained", 100, 10), ("tiny", 2000, 100),
                                          ("mixtral_decode", 200, 20)])
def test_repeated_forwards_are_bit_identical(name, n, every):
    wl = I.WORKLOADS[name]
    d = I.make_inputs(wl, "cuda")
    ws = moe.Workspace()
    args = (d["x"], d["logits"], d["W1"], d["W3"], d["W2"], wl.k)
    ref = moe.moe_forward(*args, ws=ws).clone()
    out = torch.empty_like(ref)
    for i in range(n):
        moe.moe_forward(*args, out=out, ws=ws)
        if (i + 1) % every == 0:
            assert torch.equal(out, ref), f"{name}: forward {i} differs"
            assert moe.moe_get_device_status(ws) == 0, f"{name}: status after forward {i}"
