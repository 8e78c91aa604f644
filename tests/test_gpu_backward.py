"""The layer's backward on the GPU against the oracle's fp64 gradients.

The GPU stores g, u, h, y, dY, dg, du, each assignment's dx row and the
outputs in bf16 (relative rounding eps = 2^-9 each) and accumulates in fp32.
Each gradient must meet both criteria of tests.helpers.backward_mismatches:
elementwise |gpu - ref| <= 2^-8 |ref| + 6 eps mag (mag: the oracle's
first-order worst case of those roundings) and normwise, per expert for the
weight gradients, ||gpu - ref|| <= 2^-5 ||ref||.  tests/test_backward_bound.py
pins mag against an independent first-order computation, shows an fp64 run
with the same bf16 roundings well inside both, and shows kernel-shaped
mistakes (a dropped 16-row K group, a missing block of dY, dg and du
exchanged) outside them."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import backward_mismatches

pytestmark = pytest.mark.gpu

CASES = {  # name: (T, H, F, E, k) -- block mode from the mean rows per expert
    "tiny_blocks": (64, 256, 384, 8, 2),
    "small_blocks": (200, 384, 512, 6, 3),
    "large_blocks_ragged": (300, 256, 256, 4, 2),      # paired dh and dx tiles
    "large_unpaired": (400, 384, 384, 4, 2),           # H, F not multiples of 256
    "large_pair_f_only": (400, 384, 512, 4, 2),
    "large_multi_block": (600, 256, 512, 2, 2),        # three blocks; 256 x 256 WGrad
    "deep_wgrad_f384": (600, 256, 384, 2, 2),          # dW2 128-wide, dW1/dW3 256 x 256
    "many_empty_experts": (20, 128, 256, 32, 1),
    "fine_grained_like": (150, 256, 128, 32, 6),
    "max_experts_topk": (64, 128, 128, 1024, 32),      # the header's limits
    "split_dx_tiny": (64, 2560, 256, 16, 2),          # 320 dx tiles: balanced K split
}


def mismatches(name, gpu, ref):
    return backward_mismatches("", gpu, ref, name)


@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(name):
    T, H, F, E, k = CASES[name]
    wl = I.small(name, T=T, H=H, F=F, E=E, k=k)
    d = I.make_inputs(wl, "cpu")
    dout = torch.randn(T, H, generator=torch.Generator().manual_seed(31)).to(torch.bfloat16)
    dev = {n: t.cuda() for n, t in d.items()}
    ws = moe.Workspace()
    out = moe.moe_forward_train(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], k, ws)
    plain = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], k)
    assert torch.equal(out, plain)                      # same forward, plus saved state
    dx, dl, dW1, dW3, dW2 = moe.moe_backward(dout.cuda(), dev["logits"], dev["W1"], dev["W3"],
                                             dev["W2"], k, ws)
    assert moe.moe_get_device_status(ws) == 0
    ref = O.backward(d["x"], d["logits"].numpy(), d["W1"], d["W3"], d["W2"], k, dout,
                     magnitudes=True)
    msgs = (mismatches("dx", dx, ref) + mismatches("dlogits", dl, ref) +
            mismatches("dW1", dW1, ref) + mismatches("dW3", dW3, ref) +
            mismatches("dW2", dW2, ref))
    assert not msgs, "\n".join(msgs)
    # experts that received no token get exactly zero gradients
    counts = np.bincount(O.route_topk(d["logits"].numpy(), k)[0].reshape(-1), minlength=E)
    for e in np.nonzero(counts == 0)[0]:
        assert not dW1[e].any() and not dW3[e].any() and not dW2[e].any()
    # deterministic: a second backward gives the same bits
    again = moe.moe_backward(dout.cuda(), dev["logits"], dev["W1"], dev["W3"], dev["W2"], k, ws)
    for a, b in zip((dx, dl, dW1, dW3, dW2), again):
        assert torch.equal(a, b)


# Rows per expert chosen so that the weight gradients' last K stage ends at
# every kind of place: inside the first 16-row group, on a 16-row boundary,
# one past it, at the end of a 64-row stage, one past it; plus an expert with
# no rows.  Each token goes to one expert (k = 1) through a logit margin.
TAIL_COUNTS = [1, 15, 16, 17, 31, 48, 63, 64, 65, 127, 128, 129, 0]


@pytest.mark.parametrize("H,F", [(256, 512), (384, 384)])
def test_backward_wgrad_tail_rows(H, F):
    E, k = len(TAIL_COUNTS), 1
    labels = np.repeat(np.arange(E), TAIL_COUNTS)
    rng = np.random.default_rng(5)
    rng.shuffle(labels)
    T = labels.size
    wl = I.small("tail_rows", T=T, H=H, F=F, E=E, k=k)
    d = I.make_inputs(wl, "cpu")
    logits = (0.1 * rng.standard_normal((T, E))).astype(np.float32)
    logits[np.arange(T), labels] += 5.0
    d["logits"] = torch.from_numpy(logits)
    assert np.array_equal(np.bincount(O.route_topk(logits, k)[0].reshape(-1), minlength=E),
                          TAIL_COUNTS)
    dout = torch.randn(T, H, generator=torch.Generator().manual_seed(32)).to(torch.bfloat16)
    dev = {n: t.cuda() for n, t in d.items()}
    ws = moe.Workspace()
    moe.moe_forward_train(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], k, ws)
    dx, dl, dW1, dW3, dW2 = moe.moe_backward(dout.cuda(), dev["logits"], dev["W1"], dev["W3"],
                                             dev["W2"], k, ws)
    assert moe.moe_get_device_status(ws) == 0
    ref = O.backward(d["x"], logits, d["W1"], d["W3"], d["W2"], k, dout, magnitudes=True)
    msgs = (mismatches("dx", dx, ref) + mismatches("dlogits", dl, ref) +
            mismatches("dW1", dW1, ref) + mismatches("dW3", dW3, ref) +
            mismatches("dW2", dW2, ref))
    assert not msgs, "\n".join(msgs)
    assert not dW1[E - 1].any() and not dW3[E - 1].any() and not dW2[E - 1].any()
