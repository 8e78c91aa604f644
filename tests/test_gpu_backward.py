"""The layer's backward on the GPU against the oracle's fp64 gradients.

The GPU stores g, u, h, y, dY, dg, du, dx_perm and the outputs in bf16
(relative rounding eps = 2^-9 each) and accumulates in fp32.  The oracle
returns, as "mag_<name>", the first-order size in units of eps of what those
roundings do to each gradient (the rounding of dY through dh, of u, of g
through the SwiGLU derivative -- whose factor crosses zero near g = -1.28 --
and of the stored results, each followed through the chain rule):
    |gpu - ref| <= 2^-8 |ref| + KAPPA * eps * mag,   KAPPA = 6.
An fp64 run that rounds the same intermediates to bf16 reaches at most 0.6
of this bound on these cases; a wrong index, transpose or missing term errs
by O(1) of the magnitude and fails it."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I

pytestmark = pytest.mark.gpu

KAPPA = 6
EPS = 2.0 ** -9

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
    g = gpu.double().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    r = np.asarray(ref[name], np.float64)
    bound = 2 * EPS * np.abs(r) + KAPPA * EPS * np.asarray(ref["mag_" + name]) + 1e-6
    err = np.abs(g - r)
    bad = err > bound
    if not bad.any():
        return []
    where = [tuple(int(v) for v in i) for i in np.argwhere(bad)[:6]]
    return [f"{name}: {bad.sum()}/{bad.size} out of bound, max err/bound "
            f"{(err / bound).max():.2f}; first at {where}: gpu "
            f"{[float(g[w]) for w in where]} ref {[float(r[w]) for w in where]}"]


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
