"""The forward's one-launch routing for small batches (T*k <= 1024 and
E <= 256: 32 tokens routed per CTA, the last CTA to finish counts, scans and
scatters every assignment) against the oracle: top-k indices, counts,
offsets and the permutation bit-exact, weights within W_ATOL, the layer
output within the usual tolerance.  The shapes cover T not a multiple of
32, every lane width of the routing (E up to 32, 64, 128, 256), k up to 8,
the T*k = 1024 boundary and the first size past it (the chunked kernels),
and a non-finite logit."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import W_ATOL, assert_moe_close, to_np

pytestmark = pytest.mark.gpu

SHAPES = [  # (T, E, k)
    (1, 8, 1), (1, 8, 8), (31, 8, 2), (37, 129, 3), (33, 256, 8), (50, 100, 4),
    (100, 64, 5), (128, 200, 8), (1024, 16, 1), (205, 16, 5),
]


def run_forward(T, E, k, seed, nan_at=None):
    wl = I.small(f"smallroute_{T}_{E}_{k}_{seed}", T=T, H=128, F=128, E=E, k=k)
    d = I.make_inputs(wl, "cpu")
    if nan_at is not None:
        d["logits"][nan_at] = float("nan")
    dev = {n: t.cuda() for n, t in d.items()}
    ws = moe.Workspace()
    out = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], k, ws=ws)
    routing = moe.moe_forward_routing(ws, T, 128, 128, E, k)
    return d, out, routing, ws


@pytest.mark.parametrize("T,E,k", SHAPES)
def test_small_batch_routing_matches_oracle(T, E, k):
    d, out, (idx, w, counts, offsets, src, dest), ws = run_forward(T, E, k, seed=3)
    assert moe.moe_get_device_status(ws) == 0
    idx_ref, w_ref = O.route_topk(d["logits"].numpy(), k)
    np.testing.assert_array_equal(to_np(idx), idx_ref)
    np.testing.assert_allclose(to_np(w), w_ref, rtol=0, atol=W_ATOL)
    for got, ref in zip((counts, offsets, src, dest), O.permute(idx_ref, E)):
        np.testing.assert_array_equal(to_np(got), ref)
    ref = O.forward_perm(d["x"], d["logits"].numpy(), d["W1"], d["W3"], d["W2"], k)
    assert_moe_close(out, ref["out"], f"small routing T={T} E={E} k={k} out")


def test_small_batch_routing_twice_on_one_workspace():
    """The ticket counter the last CTA consumes is back at zero after a
    launch: a second forward on the same workspace routes the same way."""
    T, E, k = 300, 32, 3
    d, out, r1, ws = run_forward(T, E, k, seed=5)
    dev = {n: t.cuda() for n, t in d.items()}
    out2 = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], k, ws=ws)
    r2 = moe.moe_forward_routing(ws, T, 128, 128, E, k)
    assert torch.equal(out, out2)
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


def test_small_batch_nonfinite_logit_reported():
    T, E, k = 64, 16, 2
    _, _, (idx, _, counts, _, _, _), ws = run_forward(T, E, k, seed=7, nan_at=(5, 3))
    assert moe.moe_get_device_status(ws) == 2   # MOE_ERR_NONFINITE
    i = to_np(idx)
    assert i.min() >= 0 and i.max() < E
    assert to_np(counts).sum() == T * k
