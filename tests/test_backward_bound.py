"""Pins the parity bound of the layer's backward, on the CPU.

The GPU check of the backward (tests/test_gpu_backward.py, with the criteria
of tests.helpers.backward_mismatches) accepts a gradient when
    |gpu - ref| <= 2 eps |ref| + KAPPA eps mag + 1e-6,   eps = 2^-9, KAPPA = 6,
elementwise, and ||gpu - ref|| <= 2^-5 ||ref|| normwise (per expert for the
weight gradients), where ref and mag come from the oracle's backward (mag =
the first-order size, in units of eps, of what rounding the stored bf16
operands does to each gradient).  A bound that leans on an oracle output
needs that output pinned from both sides:

  * from below -- mag is at least the largest first-order change that any
    signs of the roundings make, computed here independently by automatic
    differentiation of the chain with a relative perturbation on every
    stored operand;
  * from above -- the same automatic differentiation: mag equals that
    largest first-order change for dW1, dW3, dW2 and dlogits, and stays
    within a small factor of it for dx (where the oracle takes the triangle
    inequality inside the sum over features); and kernel-shaped mistakes (a
    16-row K group of one expert dropped from dW1, one 16-row block of dY
    left out, dg and du swapped) fail the criteria at the GPU cases' sizes,
    while an fp64 run that rounds the same operands to bf16 as the GPU stores
    them passes them with room to spare.
The elementwise bound is a worst case over the signs of the roundings, so
random roundings reach only a few percent (dx, dlogits) to about a tenth (the
weight gradients) of it; mistakes spread thinly over a large expert (a 16-row
K group out of 600 rows) stay under it too, and the normwise criterion is the
one that catches them.
The roundings are those of reading C15 of the design notes (which backward
intermediates the GPU keeps in bf16).
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import BWD_EPS as EPS, BWD_KAPPA as KAPPA, BWD_NORM_TOL, backward_mismatches

NAMES = ("dx", "dlogits", "dW1", "dW3", "dW2")

# the sizes of the GPU backward cases (block modes, paired tiles, empty
# experts, the header's limits)
GPU_CASES = {
    "tiny_blocks": (64, 256, 384, 8, 2),
    "small_blocks": (200, 384, 512, 6, 3),
    "large_blocks_ragged": (300, 256, 256, 4, 2),
    "large_unpaired": (400, 384, 384, 4, 2),
    "large_pair_f_only": (400, 384, 512, 4, 2),
    "large_multi_block": (600, 256, 512, 2, 2),
    "deep_wgrad_f384": (600, 256, 384, 2, 2),
    "many_empty_experts": (20, 128, 256, 32, 1),
    "fine_grained_like": (150, 256, 128, 32, 6),
    "max_experts_topk": (64, 128, 128, 1024, 32),
    "split_dx_tiny": (64, 2560, 256, 16, 2),
}


def bound(ref, name):
    return 2 * EPS * np.abs(ref[name]) + KAPPA * EPS * ref["mag_" + name] + 1e-6


def worst_ratio(got, ref, name):
    return float(np.max(np.abs(np.asarray(got[name]) - ref[name]) / bound(ref, name)))


# ------------------------------------------------------ the chain, perturbed
def perturbed_grads(x, logits, W1, W3, W2, k, dout, d):
    """The backward written as plain torch fp64 ops, with every operand the GPU
    stores in bf16 multiplied by (1 + d[name]) where it is stored: the forward's
    h and y, the saved g and u, dY, dg, du and the per-assignment dx rows.
    Returns the five gradients as one flat vector."""
    l = np.asarray(logits, np.float32)
    T, E = l.shape
    idx, w = O.route_topk(l, k)
    flat = idx.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")            # assignment of each sorted row
    tok, slot, exp = order // k, order % k, flat[order]
    X = torch.as_tensor(np.asarray(x, np.float64))[tok]
    W1t, W3t, W2t = (torch.as_tensor(np.asarray(W, np.float64))[exp] for W in (W1, W3, W2))
    Dt = torch.as_tensor(np.asarray(dout, np.float64))[tok]
    wt = torch.as_tensor(w.astype(np.float64))[tok, slot]
    g = torch.einsum("ph,phf->pf", X, W1t)
    u = torch.einsum("ph,phf->pf", X, W3t)
    h = (g * torch.sigmoid(g) * u) * (1 + d["h"])
    y = torch.einsum("pf,pfh->ph", h, W2t) * (1 + d["y"])
    dY = wt[:, None] * Dt * (1 + d["dY"])
    dw = (Dt * y).sum(1)
    gb, ub = g * (1 + d["g"]), u * (1 + d["u"])
    s = torch.sigmoid(gb)
    dh = torch.einsum("ph,pfh->pf", dY, W2t)
    dg = dh * ub * s * (1 + gb * (1 - s)) * (1 + d["dg"])
    du = dh * gb * s * (1 + d["du"])
    dxp = (torch.einsum("pf,phf->ph", dg, W1t) + torch.einsum("pf,phf->ph", du, W3t)) \
        * (1 + d["dxp"])
    H, F = X.shape[1], g.shape[1]
    tok_t = torch.as_tensor(tok)
    dx = torch.zeros(T, H, dtype=torch.float64).index_add(0, tok_t, dxp)
    key = torch.as_tensor(exp)
    dW1 = torch.zeros(E, H, F, dtype=torch.float64).index_add(
        0, key, X[:, :, None] * dg[:, None, :])
    dW3 = torch.zeros(E, H, F, dtype=torch.float64).index_add(
        0, key, X[:, :, None] * du[:, None, :])
    dW2 = torch.zeros(E, F, H, dtype=torch.float64).index_add(
        0, key, h[:, :, None] * dY[:, None, :])
    # exact softmax of the selected logits, and its Jacobian
    sel = np.take_along_axis(l.astype(np.float64), idx.astype(np.int64), axis=1)
    p = np.exp(sel - sel[:, :1])
    p = torch.as_tensor(p / p.sum(1, keepdims=True))
    dwm = torch.zeros(T, k, dtype=torch.float64).index_put((tok_t, torch.as_tensor(slot)), dw)
    dsel = p * (dwm - (p * dwm).sum(1, keepdim=True))
    dl = torch.zeros(T, E, dtype=torch.float64).scatter(1, torch.as_tensor(
        idx.astype(np.int64)), dsel)
    return torch.cat([v.reshape(-1) for v in (dx, dl, dW1, dW3, dW2)]), (T, H, F, E)


def first_order_max(x, logits, W1, W3, W2, k, dout):
    """The largest first-order change, over all signs of the roundings, of every
    gradient element: the sum of |d gradient / d perturbation| at zero."""
    P = np.asarray(logits).shape[0] * k
    H, F = np.asarray(W1).shape[1:]
    shapes = {"h": (P, F), "y": (P, H), "dY": (P, H), "g": (P, F), "u": (P, F),
              "dg": (P, F), "du": (P, F), "dxp": (P, H)}
    names = list(shapes)
    sizes = [int(np.prod(shapes[n])) for n in names]

    def fn(vec):
        parts = torch.split(vec, sizes)
        d = {n: v.reshape(shapes[n]) for n, v in zip(names, parts)}
        return perturbed_grads(x, logits, W1, W3, W2, k, dout, d)[0]

    zero = torch.zeros(sum(sizes), dtype=torch.float64)
    J = torch.autograd.functional.jacobian(fn, zero)
    m = J.abs().sum(1).numpy()
    T, E = np.asarray(logits).shape
    cuts = np.cumsum([T * H, T * E, E * H * F, E * H * F])
    parts = np.split(m, cuts)
    shp = {"dx": (T, H), "dlogits": (T, E), "dW1": (E, H, F), "dW3": (E, H, F),
           "dW2": (E, F, H)}
    return {n: v.reshape(shp[n]) for n, v in zip(NAMES, parts)}


def small_case(seed, T=9, H=4, F=6, E=5, k=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    W1, W3 = rng.standard_normal((E, H, F)) / 2, rng.standard_normal((E, H, F)) / 2
    W2 = rng.standard_normal((E, F, H)) / 2
    dout = rng.standard_normal((T, H))
    return x, logits, W1, W3, W2, k, dout


def test_perturbed_chain_is_the_oracle_backward():
    """With no perturbation the chain above gives the oracle's gradients (so
    the Jacobian below is taken of the right function)."""
    args = small_case(40)
    P = args[1].shape[0] * args[5]
    H, F = args[2].shape[1:]
    zero = {n: torch.zeros(P, F if n in ("h", "g", "u", "dg", "du") else H,
                           dtype=torch.float64)
            for n in ("h", "y", "dY", "g", "u", "dg", "du", "dxp")}
    vec, (T, H, F, E) = perturbed_grads(*args, zero)
    ref = O.backward(*args)
    want = np.concatenate([ref[n].reshape(-1) for n in NAMES])
    np.testing.assert_allclose(vec.numpy(), want, rtol=1e-10, atol=1e-12)


def check_magnitudes(seed, shape, backward=None):
    backward = backward or O.backward
    T, H, F, E, k = shape
    args = small_case(seed, T, H, F, E, k)
    ref = backward(*args, magnitudes=True)
    fo = first_order_max(*args)
    for n in ("dW1", "dW3", "dW2", "dlogits"):   # the oracle's sums are exact here
        np.testing.assert_allclose(ref["mag_" + n], fo[n], rtol=1e-9, atol=1e-12, err_msg=n)
    for n in ("dx",):                        # an upper bound, and not a loose one
        assert np.all(ref["mag_" + n] >= fo[n] * (1 - 1e-9) - 1e-12), n
        nz = fo[n] > 1e-9
        assert np.all(ref["mag_" + n][nz] <= 4.0 * fo[n][nz]), (n, (ref["mag_" + n][nz] /
                                                                   fo[n][nz]).max())


SMALL_SHAPES = [(41, (9, 4, 6, 5, 2)), (42, (12, 3, 8, 3, 3)), (43, (7, 5, 4, 6, 1))]


@pytest.mark.parametrize("seed,shape", SMALL_SHAPES)
def test_magnitudes_against_the_first_order_maximum(seed, shape):
    check_magnitudes(seed, shape)


def test_magnitude_pins_catch_planted_mistakes():
    """Magnitudes several times too large, or too small (as when a rounding
    term is left out), fail the first-order pin."""
    def scaled(f, only=None):
        def bwd(*a, **kw):
            r = O.backward(*a, **kw)
            for n in NAMES:
                if only is None or n == only:
                    r["mag_" + n] = r["mag_" + n] * f
            return r
        return bwd

    for bad in (scaled(10.0), scaled(0.5), scaled(10.0, "dx"), scaled(0.5, "dx"),
                scaled(0.5, "dW2"), scaled(2.0, "dlogits")):
        with pytest.raises(AssertionError):
            check_magnitudes(*SMALL_SHAPES[0], backward=bad)


# -------------------------------------- the GPU's roundings, emulated in fp64
def bf16(a):
    return torch.as_tensor(np.asarray(a, np.float64)).to(torch.bfloat16).double().numpy()


def emulate_gpu_backward(x, logits, W1, W3, W2, k, dout, plant=None):
    """The backward with the GPU's stores rounded to bf16 (fp64 arithmetic in
    between, standing in for fp32 accumulation): g, u, h and y of the forward,
    dY = bf16(w dout), dg, du, each assignment's dx row, and the results.
    `plant` names a kernel-shaped mistake to make on the way."""
    l = np.asarray(logits, np.float32)
    T, E = l.shape
    idx, w = O.route_topk(l, k)
    counts, offsets, src, dest = O.permute(idx, E)
    x64 = np.asarray(torch.as_tensor(x).double() if isinstance(x, torch.Tensor) else x,
                     np.float64)
    d64 = np.asarray(torch.as_tensor(dout).double() if isinstance(dout, torch.Tensor) else dout,
                     np.float64)
    Wd = [np.asarray(torch.as_tensor(W).double() if isinstance(W, torch.Tensor) else W,
                     np.float64) for W in (W1, W3, W2)]
    H, F = Wd[0].shape[1:]
    out = {"dx": np.zeros((T, H)), "dW1": np.zeros((E, H, F)), "dW3": np.zeros((E, H, F)),
           "dW2": np.zeros((E, F, H))}
    dw = np.zeros((T, k))
    dxp_all = np.zeros((T * k, H))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if lo == hi:
            continue
        a = src[lo:hi]
        t, j = a // k, a % k
        X = x64[t]
        g, u = X @ Wd[0][e], X @ Wd[1][e]
        h = bf16(g / (1 + np.exp(-g)) * u)
        y = bf16(h @ Wd[2][e])
        gb, ub = bf16(g), bf16(u)
        dY = bf16(w[t, j].astype(np.float64)[:, None] * d64[t])
        if plant == "omit_dY_block" and e == int(np.argmax(counts)):
            dY[:min(16, hi - lo)] = 0.0                 # one 16-row block of dY left out
        dw[t, j] = np.sum(d64[t] * y, axis=1)
        s = 1 / (1 + np.exp(-gb))
        dh = dY @ Wd[2][e].T
        dg = bf16(dh * ub * s * (1 + gb * (1 - s)))
        du = bf16(dh * gb * s)
        if plant == "swap_dg_du":
            dg, du = du, dg
        Xw = X
        if plant == "drop_k_group_dW1" and e == int(np.argmax(counts)) and hi - lo > 16:
            Xw = X.copy()
            Xw[16:32] = 0.0                             # rows 16..31 missing from dW1's K loop
        out["dW1"][e] = bf16(Xw.T @ dg)
        out["dW3"][e] = bf16(X.T @ du)
        out["dW2"][e] = bf16(h.T @ dY)
        dxp_all[a] = bf16(dg @ Wd[0][e].T + du @ Wd[1][e].T)
    for j in range(k):
        out["dx"] += dxp_all[np.arange(T) * k + j]
    out["dx"] = bf16(out["dx"])
    sel = np.take_along_axis(l.astype(np.float64), idx.astype(np.int64), axis=1)
    p = np.exp(sel - sel[:, :1])
    p = (p / p.sum(1, keepdims=True)).astype(np.float32).astype(np.float64)
    dl = np.zeros((T, E))
    np.put_along_axis(dl, idx.astype(np.int64), p * (dw - np.sum(p * dw, 1, keepdims=True)), 1)
    out["dlogits"] = dl.astype(np.float32).astype(np.float64)
    return out


def gpu_case(name):
    T, H, F, E, k = GPU_CASES[name]
    wl = I.small(name, T=T, H=H, F=F, E=E, k=k)
    d = I.make_inputs(wl, "cpu")
    dout = torch.randn(T, H, generator=torch.Generator().manual_seed(31)).to(torch.bfloat16)
    return (d["x"], d["logits"].numpy(), d["W1"], d["W3"], d["W2"], k, dout)


_REFS = {}


def ref_of(name):
    if name not in _REFS:
        args = gpu_case(name)
        _REFS[name] = (args, O.backward(*args, magnitudes=True))
    return _REFS[name]


def normwise_ratio(got, ref, n):
    """The largest normwise relative error (per expert for the weight gradients)
    as a fraction of the normwise tolerance."""
    g, r = np.asarray(got[n]), np.asarray(ref[n])
    groups = [(g[e], r[e]) for e in range(r.shape[0])] if n.startswith("dW") else [(g, r)]
    return max(float(np.linalg.norm(ge - re)) / (BWD_NORM_TOL * float(np.linalg.norm(re)) +
                                                 1e-6 * np.sqrt(re.size)) for ge, re in groups)


@pytest.mark.parametrize("name", list(GPU_CASES))
def test_bf16_rounding_stays_well_inside_the_bound(name):
    args, ref = ref_of(name)
    emu = emulate_gpu_backward(*args)
    for n in NAMES:
        assert not backward_mismatches(name, emu[n], ref, n)
        r = worst_ratio(emu, ref, n)
        assert r <= 0.6, (name, n, "elementwise", r)
        r = normwise_ratio(emu, ref, n)
        assert r <= 0.25, (name, n, "normwise", r)


@pytest.mark.parametrize("plant", ["drop_k_group_dW1", "omit_dY_block", "swap_dg_du"])
@pytest.mark.parametrize("name", ["tiny_blocks", "small_blocks", "large_multi_block",
                                  "fine_grained_like", "split_dx_tiny"])
def test_bound_rejects_kernel_shaped_mistakes(name, plant):
    args, ref = ref_of(name)
    bad = emulate_gpu_backward(*args, plant=plant)
    hit = {n: bool(backward_mismatches(name, bad[n], ref, n)) for n in NAMES}
    want = {"drop_k_group_dW1": ["dW1"], "omit_dY_block": ["dW2", "dW1", "dW3", "dx"],
            "swap_dg_du": ["dW1", "dW3", "dx"]}[plant]
    assert all(hit[n] for n in want), (name, plant, hit)
    # the gradients the mistake does not touch still pass
    assert not any(hit[n] for n in NAMES if n not in want), (name, plant, hit)
