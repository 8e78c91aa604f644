"""The layer's backward at the full sizes of the workloads of record, launched
exactly as the training benchmark launches it (moe_forward_train, then
moe_backward), against the oracle on samples it can afford:

  * dx and dlogits of a few tokens, from the oracle's backward of that
    sub-batch (a token's input and logit gradients depend on it alone);
  * dW1[:, :, J], dW3[:, :, J] and dW2[:, J, :] for a few features J, from
    the oracle's backward with F cut to J (SwiGLU acts feature by feature).

Both restrictions are pinned on the CPU against the uncut oracle.  The bound
is the one of the small-case backward test (tests.helpers.backward_mismatches:
elementwise 2^-8 |ref| + 6 eps mag, and normwise 2^-5, per expert for the
weight gradients)."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import backward_mismatches

pytestmark = pytest.mark.gpu

NAMES = ["mixtral_decode", "dbrx_prefill", "fine_grained", "skewed"]


def check(name, gpu, ref, key):
    msgs = backward_mismatches(name, gpu, ref, key)
    assert not msgs, "\n".join(msgs)


@pytest.mark.parametrize("name", NAMES)
def test_full_size_backward(name):
    wl = I.WORKLOADS[name]
    d = I.make_inputs(wl, "cuda")
    g = torch.Generator(device="cuda").manual_seed(7)
    dout = torch.randn(wl.T, wl.H, generator=g, device="cuda").to(torch.bfloat16)
    ws = moe.Workspace()
    moe.moe_forward_train(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], wl.k, ws)
    dx, dl, dW1, dW3, dW2 = moe.moe_backward(dout, d["logits"], d["W1"], d["W3"], d["W2"],
                                             wl.k, ws)
    assert moe.moe_get_device_status(ws) == 0
    logits = d["logits"].cpu().numpy()
    dout_c = dout.cpu()
    rng = np.random.default_rng(1)
    tok = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 3, replace=False)]))
    J = np.unique(np.concatenate([[0, wl.F - 1], rng.choice(wl.F, 4, replace=False)]))
    # sampled tokens: dx and dlogits
    sub = O.backward(d["x"][torch.from_numpy(tok).cuda()].cpu(), logits[tok], d["W1"], d["W3"],
                     d["W2"], wl.k, dout_c[torch.from_numpy(tok)], magnitudes=True)
    t_idx = torch.from_numpy(tok).cuda()
    check(name, dx[t_idx], sub, "dx")
    check(name, dl[t_idx], sub, "dlogits")
    # sampled features: the weight gradients
    Jt = torch.from_numpy(J).cuda()
    cut = O.backward(d["x"].cpu(), logits, d["W1"][:, :, Jt].cpu(), d["W3"][:, :, Jt].cpu(),
                     d["W2"][:, Jt, :].cpu(), wl.k, dout_c, magnitudes=True)
    check(name, dW1[:, :, Jt], cut, "dW1")
    check(name, dW3[:, :, Jt], cut, "dW3")
    check(name, dW2[:, Jt, :], cut, "dW2")
    # properties at any size: finite, and experts without tokens get zeros
    for t in (dx, dl, dW1, dW3, dW2):
        assert torch.isfinite(t.float()).all()
    counts = np.bincount(O.route_topk(logits, wl.k)[0].reshape(-1), minlength=wl.E)
    for e in np.nonzero(counts == 0)[0]:
        assert not dW1[e].any() and not dW3[e].any() and not dW2[e].any()
