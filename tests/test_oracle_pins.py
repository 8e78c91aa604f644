"""Pins the CPU oracle to facts that do not come from the oracle itself:
brute force on tiny inputs, closed forms, invariants, a reduction to a
library routine, and the pages' printed numbers (tests/golden).

The mutation tests at the bottom plant a plausible mistake in the oracle and
check that one of these pins fails, so the pins are known to have teeth.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import accounting as acc
from routing_grouped_expert_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def brute_topk(l, k):
    """Sort (−logit, expert) pairs; first k.  Python floats: -0.0 == 0.0."""
    T, E = l.shape
    return np.array([sorted(range(E), key=lambda e: (-float(l[t, e]), e))[:k]
                     for t in range(T)], dtype=np.int32).reshape(T, k)


def check_topk_brute(route=None, seed=0):
    route = route or O.route_topk
    rng = np.random.default_rng(seed)
    vals = np.array([-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 2.0], dtype=np.float32)
    for E in range(1, 7):
        for k in range(1, E + 1):
            for T in (1, 3, 8):
                l = rng.choice(vals, size=(T, E)).astype(np.float32)
                idx, _ = route(l, k)
                np.testing.assert_array_equal(idx, brute_topk(l, k))


def brute_ffn_row(x, W1e, W3e, W2e):
    """Pure-Python loops of (silu(x W1) * (x W3)) W2 for one row."""
    H, F = len(W1e), len(W1e[0])
    a = []
    for f in range(F):
        g = sum(float(x[h]) * float(W1e[h][f]) for h in range(H))
        u = sum(float(x[h]) * float(W3e[h][f]) for h in range(H))
        a.append(g / (1.0 + math.exp(-g)) * u)
    return [sum(a[f] * float(W2e[f][i]) for f in range(F)) for i in range(H)]


def check_ffn_brute(ffn=None, seed=1):
    ffn = ffn or O.expert_ffn
    rng = np.random.default_rng(seed)
    H, F, n = 3, 5, 4                          # non-square: a transpose cannot pass
    x = rng.standard_normal((n, H))
    W1, W3 = rng.standard_normal((H, F)), rng.standard_normal((H, F))
    W2 = rng.standard_normal((F, H))
    got = ffn(x, W1, W3, W2)
    want = np.array([brute_ffn_row(x[r], W1, W3, W2) for r in range(n)])
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def rand_layer(T, H, F, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(E, H, F, generator=g) / math.sqrt(H)).to(torch.bfloat16)
    W3 = (torch.randn(E, H, F, generator=g) / math.sqrt(H)).to(torch.bfloat16)
    W2 = (torch.randn(E, F, H, generator=g) / math.sqrt(F)).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g).numpy()
    return x, logits, W1, W3, W2


def check_permute(permute=None, seed=2):
    permute = permute or O.permute
    rng = np.random.default_rng(seed)
    for T, E, k in ((0, 4, 2), (1, 1, 1), (37, 8, 2), (200, 16, 4), (64, 256, 8)):
        idx, _ = O.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
        counts, offsets, src, dest = permute(idx, E)
        flat = idx.reshape(-1)
        assert counts.sum() == T * k                                 # sum c_e = T*k
        np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
        np.testing.assert_array_equal(offsets[1:], np.cumsum(counts))
        assert offsets[0] == 0
        np.testing.assert_array_equal(src, np.argsort(flat, kind="stable"))
        np.testing.assert_array_equal(np.sort(src), np.arange(T * k))  # bijection
        np.testing.assert_array_equal(dest[src], np.arange(T * k))
        np.testing.assert_array_equal(src[dest], np.arange(T * k))
        for e in range(E):                                          # by token, then slot
            seg = src[offsets[e]:offsets[e + 1]]
            assert np.all(np.diff(seg) > 0)
            assert np.all(flat[seg] == e)


# ------------------------------------------------------------------- top-k
def test_topk_brute_force_with_ties_and_signed_zeros():
    check_topk_brute()


def test_topk_slots_descending_and_distinct():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((100, 16)).astype(np.float32)
    idx, w = O.route_topk(l, 5)
    vals = np.take_along_axis(l, idx, 1)
    assert np.all(np.diff(vals, axis=1) <= 0)
    assert np.all(np.diff(w, axis=1) <= 0)
    assert all(len(set(r)) == 5 for r in idx.tolist())


def test_weights_closed_forms():
    rng = np.random.default_rng(4)
    l = rng.standard_normal((500, 8)).astype(np.float32)
    # k = 1: w = 1 exactly
    _, w1 = O.route_topk(l, 1)
    assert np.all(w1 == 1.0)
    # equal logits: w = 1/k exactly (after rounding to fp32)
    for k in (2, 3, 4, 8):
        _, we = O.route_topk(np.full((3, 8), 0.7, np.float32), k)
        assert np.all(we == np.float32(1.0 / k))
    # k = 2: w0 = logistic(l0 - l1)
    idx, w2 = O.route_topk(l, 2)
    v = np.take_along_axis(l.astype(np.float64), idx, 1)
    want = 1.0 / (1.0 + np.exp(v[:, 1] - v[:, 0]))
    np.testing.assert_allclose(w2[:, 0], want, rtol=2e-7)
    np.testing.assert_allclose(w2[:, 1], 1.0 - want, rtol=2e-7, atol=1e-7)
    # all k: weights sum to one
    for k in (1, 2, 3, 5, 8):
        _, w = O.route_topk(l, k)
        np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)


def test_weights_shift_invariance():
    rng = np.random.default_rng(5)
    l = rng.standard_normal((50, 12)).astype(np.float32)
    i0, w0 = O.route_topk(l, 4)
    i1, w1 = O.route_topk(l + np.float32(3.0), 4)
    np.testing.assert_array_equal(i0, i1)
    np.testing.assert_allclose(w0, w1, rtol=1e-5)


def test_nonfinite_and_bad_k_rejected():
    l = np.zeros((4, 8), np.float32)
    l[2, 3] = np.nan
    with pytest.raises(O.NonFiniteLogits):
        O.route_topk(l, 2)
    l[2, 3] = np.inf
    with pytest.raises(O.NonFiniteLogits):
        O.route_topk(l, 2)
    with pytest.raises(ValueError):
        O.route_topk(np.zeros((4, 8), np.float32), 9)
    with pytest.raises(ValueError):
        O.route_topk(np.zeros((4, 8), np.float32), 0)


# ---------------------------------------------------------------- permute
def test_permute_invariants_and_stable_order():
    check_permute()


def test_mean_count_closed_form():
    """E[s_e] = b*s*k/E: with every assignment kept the mean count is exact."""
    rng = np.random.default_rng(6)
    for T, E, k in ((256, 8, 2), (1000, 16, 4), (333, 256, 8)):
        idx, _ = O.route_topk(rng.standard_normal((T, E)).astype(np.float32), k)
        counts = O.permute(idx, E)[0]
        assert counts.sum() * 1.0 / E == T * k / E


# -------------------------------------------------------------------- FFN
def test_ffn_brute_force_loops():
    check_ffn_brute()


def test_dense_reduction_E1_k1_matches_library_swiglu():
    x, logits, W1, W3, W2 = rand_layer(40, 48, 80, 1, 1, seed=7)
    r = O.forward_perm(x, logits, W1, W3, W2, 1)
    xd, W1d, W3d, W2d = (t.double() for t in (x, W1[0], W3[0], W2[0]))
    want = (torch.nn.functional.silu(xd @ W1d) * (xd @ W3d)) @ W2d
    np.testing.assert_allclose(r["out"], want.numpy(), rtol=1e-12, atol=1e-12)


def test_identical_experts_reproduce_dense_ffn():
    x, logits, W1, W3, W2 = rand_layer(30, 32, 64, 1, 1, seed=8)
    E, k = 6, 3
    W1e, W3e, W2e = (W.expand(E, *W.shape[1:]).contiguous() for W in (W1, W3, W2))
    logits = np.random.default_rng(9).standard_normal((30, E)).astype(np.float32)
    r = O.forward_perm(x, logits, W1e, W3e, W2e, k)
    xd = x.double()
    dense = (torch.nn.functional.silu(xd @ W1[0].double()) * (xd @ W3[0].double())) \
        @ W2[0].double()
    np.testing.assert_allclose(r["out"], dense.numpy(), rtol=1e-6, atol=1e-9)


def test_direct_equals_permuted():
    x, logits, W1, W3, W2 = rand_layer(64, 32, 48, 8, 3, seed=10)
    r = O.forward_perm(x, logits, W1, W3, W2, 3)
    d = O.forward_direct(x, logits, W1, W3, W2, 3)
    np.testing.assert_allclose(d, r["out"], rtol=1e-12, atol=1e-13)
    tok = np.array([5, 0, 63, 17])
    np.testing.assert_allclose(O.forward_direct(x, logits, W1, W3, W2, 3, tokens=tok),
                               r["out"][tok], rtol=1e-12, atol=1e-13)


def test_expert_relabeling_equivariance():
    x, logits, W1, W3, W2 = rand_layer(50, 16, 24, 8, 2, seed=11)
    pi = np.random.default_rng(12).permutation(8)         # new expert i = old pi[i]
    r0 = O.forward_perm(x, logits, W1, W3, W2, 2)
    r1 = O.forward_perm(x, logits[:, pi], W1[pi], W3[pi], W2[pi], 2)
    np.testing.assert_array_equal(pi[r1["topk_idx"]], r0["topk_idx"])
    np.testing.assert_allclose(r1["out"], r0["out"], rtol=1e-12, atol=1e-13)


def test_token_permutation_and_batch_invariance():
    x, logits, W1, W3, W2 = rand_layer(60, 16, 32, 4, 2, seed=13)
    r0 = O.forward_perm(x, logits, W1, W3, W2, 2)
    sig = np.random.default_rng(14).permutation(60)
    r1 = O.forward_perm(x[sig], logits[sig], W1, W3, W2, 2)
    np.testing.assert_allclose(r1["out"], r0["out"][sig], rtol=1e-12, atol=1e-13)
    sub = np.arange(10, 25)
    r2 = O.forward_perm(x[sub], logits[sub], W1, W3, W2, 2)
    np.testing.assert_allclose(r2["out"], r0["out"][sub], rtol=1e-12, atol=1e-13)


def test_empty_batch():
    x, logits, W1, W3, W2 = rand_layer(0, 16, 32, 4, 2, seed=15)
    r = O.forward_perm(x, logits, W1, W3, W2, 2)
    assert r["out"].shape == (0, 16)
    assert r["counts"].sum() == 0 and np.all(r["offsets"] == 0)


# ------------------------------------------------ router and shared expert
def check_router_brute(router=None, seed=16):
    router = router or O.router_logits
    rng = np.random.default_rng(seed)
    T, H, E = 4, 5, 3                       # non-square: a transpose cannot pass
    x, Wg = rng.standard_normal((T, H)), rng.standard_normal((H, E))
    want = [[sum(float(x[t][h]) * float(Wg[h][e]) for h in range(H)) for e in range(E)]
            for t in range(T)]
    np.testing.assert_allclose(router(x, Wg), want, rtol=1e-12, atol=1e-12)


def test_router_logits_brute_force():
    check_router_brute()


def test_gated_layer_routes_on_fp32_router_output():
    x, _, W1, W3, W2 = rand_layer(40, 32, 48, 6, 2, seed=17)
    Wg = torch.randn(32, 6, generator=torch.Generator().manual_seed(18)).to(torch.bfloat16)
    r = O.forward_gated(x, Wg, W1, W3, W2, 2)
    l32 = (x.double() @ Wg.double()).numpy().astype(np.float32)
    np.testing.assert_array_equal(r["logits"], l32)
    np.testing.assert_allclose(r["out"], O.forward_perm(x, l32, W1, W3, W2, 2)["out"],
                               rtol=1e-12, atol=1e-13)


def test_shared_expert_adds_the_dense_ffn():
    # E = 1, k = 1 and a shared expert equal to the routed one: out = 2 * FFN(x)
    x, _, W1, W3, W2 = rand_layer(30, 32, 64, 1, 1, seed=19)
    Wg = torch.randn(32, 1, generator=torch.Generator().manual_seed(20)).to(torch.bfloat16)
    r = O.forward_gated(x, Wg, W1, W3, W2, 1, shared=(W1[0], W3[0], W2[0]))
    xd = x.double()
    dense = (torch.nn.functional.silu(xd @ W1[0].double()) * (xd @ W3[0].double())) \
        @ W2[0].double()
    np.testing.assert_allclose(r["out"], 2 * dense.numpy(), rtol=1e-12, atol=1e-12)
    # a zero shared expert changes nothing
    z = torch.zeros_like(W1[0]), torch.zeros_like(W3[0]), torch.zeros_like(W2[0])
    r0 = O.forward_gated(x, Wg, W1, W3, W2, 1, shared=z)
    np.testing.assert_allclose(r0["out"], dense.numpy(), rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------- backward
def autograd_grads(x, logits, W1, W3, W2, k, dout):
    """The same layer written as plain torch fp64 ops with the top-k picks
    held fixed, differentiated by torch.autograd."""
    idx, _ = O.route_topk(np.asarray(logits, np.float32), k)
    idx_t = torch.as_tensor(idx, dtype=torch.long)
    xt = torch.as_tensor(np.asarray(x, np.float64)).requires_grad_()
    lt = torch.as_tensor(np.asarray(logits, np.float32).astype(np.float64)).requires_grad_()
    Ws = [torch.as_tensor(np.asarray(W, np.float64)).requires_grad_() for W in (W1, W3, W2)]
    w = torch.softmax(torch.gather(lt, 1, idx_t), dim=1)
    # the layer uses fp32-rounded weights; the rounding passes gradients through
    w = w + (w.float().double() - w).detach()
    out = torch.zeros_like(xt)
    for j in range(k):
        e = idx_t[:, j]
        g = torch.einsum("th,thf->tf", xt, Ws[0][e])
        u = torch.einsum("th,thf->tf", xt, Ws[1][e])
        y = torch.einsum("tf,tfh->th", torch.nn.functional.silu(g) * u, Ws[2][e])
        out = out + w[:, j:j + 1] * y
    (out * torch.as_tensor(np.asarray(dout, np.float64))).sum().backward()
    return dict(dx=xt.grad.numpy(), dlogits=lt.grad.numpy(), dW1=Ws[0].grad.numpy(),
                dW3=Ws[1].grad.numpy(), dW2=Ws[2].grad.numpy())


def check_backward_autograd(backward=None, seed=21):
    backward = backward or O.backward
    rng = np.random.default_rng(seed)
    T, H, F, E, k = 9, 4, 6, 5, 2
    x = rng.standard_normal((T, H))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    W1, W3 = rng.standard_normal((E, H, F)) / 2, rng.standard_normal((E, H, F)) / 2
    W2 = rng.standard_normal((E, F, H)) / 2
    dout = rng.standard_normal((T, H))
    got = backward(x, logits, W1, W3, W2, k, dout)
    want = autograd_grads(x, logits, W1, W3, W2, k, dout)
    for name in ("dx", "dlogits", "dW1", "dW3", "dW2"):
        np.testing.assert_allclose(got[name], want[name], rtol=1e-10, atol=1e-12, err_msg=name)


def test_backward_matches_autograd():
    check_backward_autograd()


def test_backward_finite_differences():
    """Central differences of L = <dout, out> for a few entries of each input."""
    rng = np.random.default_rng(22)
    T, H, F, E, k = 6, 3, 5, 4, 2
    args = dict(x=rng.standard_normal((T, H)), logits=rng.standard_normal((T, E)),
                W1=rng.standard_normal((E, H, F)), W3=rng.standard_normal((E, H, F)),
                W2=rng.standard_normal((E, F, H)))
    dout = rng.standard_normal((T, H))

    def loss(a):
        return float(np.sum(dout * O.forward_perm(a["x"], a["logits"], a["W1"], a["W3"],
                                                  a["W2"], k)["out"]))

    g = O.backward(args["x"], args["logits"], args["W1"], args["W3"], args["W2"], k, dout)
    top = int(np.argmax(args["logits"][4]))
    # logits are ranked and weighted in fp32: a step well above fp32 resolution
    for name, key, pos, eps, tol in (("x", "dx", (2, 1), 1e-6, 1e-6),
                                     ("W1", "dW1", (1, 2, 3), 1e-6, 1e-6),
                                     ("W3", "dW3", (0, 1, 4), 1e-6, 1e-6),
                                     ("W2", "dW2", (3, 4, 0), 1e-6, 1e-6),
                                     ("logits", "dlogits", (4, top), 1e-3, 2e-3)):
        plus = {n: v.copy() for n, v in args.items()}
        minus = {n: v.copy() for n, v in args.items()}
        plus[name][pos] += eps
        minus[name][pos] -= eps
        fd = (loss(plus) - loss(minus)) / (2 * eps)
        assert abs(fd - g[key][pos]) <= tol * max(1.0, abs(fd)), (name, fd, g[key][pos])


def test_backward_magnitudes_bound_the_gradients():
    x, logits, W1, W3, W2 = rand_layer(30, 8, 12, 4, 2, seed=25)
    dout = np.random.default_rng(26).standard_normal((30, 8))
    g = O.backward(x, logits, W1, W3, W2, 2, dout, magnitudes=True)
    for n in ("dx", "dlogits", "dW1", "dW3", "dW2"):
        assert np.all(g["mag_" + n] >= np.abs(g[n]) - 1e-12), n   # triangle inequality
        assert np.all(g["mag_" + n] >= 0)


def test_backward_top1_has_no_logit_gradient():
    x, logits, W1, W3, W2 = rand_layer(20, 8, 12, 4, 1, seed=23)
    dout = np.random.default_rng(24).standard_normal((20, 8))
    g = O.backward(x, logits, W1, W3, W2, 1, dout)
    assert np.all(g["dlogits"] == 0)


def test_backward_restrictions_for_sampling():
    """The two restrictions a full-size check samples through: (a) a token's
    dx and dlogits depend on that token alone (routing and combine are per
    token), so the backward of a sub-batch gives the same rows; (b) SwiGLU
    acts feature by feature, so the backward with F cut to a feature subset J
    gives the dW1[:, :, J], dW3[:, :, J] and dW2[:, J, :] of the full one,
    magnitudes included."""
    T, H, F, E, k = 24, 6, 10, 5, 2
    x, logits, W1, W3, W2 = rand_layer(T, H, F, E, k, seed=27)
    dout = np.random.default_rng(28).standard_normal((T, H))
    full = O.backward(x, logits, W1, W3, W2, k, dout, magnitudes=True)
    tok = np.array([0, 5, 23])
    sub = O.backward(x[tok], logits[tok], W1, W3, W2, k, dout[tok], magnitudes=True)
    for n in ("dx", "dlogits", "mag_dx", "mag_dlogits"):
        np.testing.assert_allclose(sub[n], full[n][tok], rtol=1e-12, atol=1e-14, err_msg=n)
    J = np.array([0, 3, 9])
    cut = O.backward(x, logits, W1[:, :, J], W3[:, :, J], W2[:, J, :], k, dout,
                     magnitudes=True)
    for n, sl in (("dW1", np.s_[:, :, J]), ("dW3", np.s_[:, :, J]), ("dW2", np.s_[:, J, :])):
        for m in (n, "mag_" + n):
            np.testing.assert_allclose(cut[m], full[m][sl], rtol=1e-12, atol=1e-14, err_msg=m)


def test_layer_is_a_sum_over_ffn_feature_slices():
    """Expert-tensor sharding along F ("MegaScale-Infer", §3.4, tpe): the
    routing does not depend on the FFN width and SwiGLU acts feature by
    feature, so the layer over W1[:, :, S], W3[:, :, S], W2[:, S, :] summed
    over a partition of the features is the whole layer."""
    x, logits, W1, W3, W2 = rand_layer(40, 16, 24, 5, 2, seed=29)
    full = O.forward_perm(x, logits, W1, W3, W2, 2)["out"]
    for parts in (2, 3):
        S = np.array_split(np.arange(24), parts)
        tot = sum(O.forward_perm(x, logits, W1[:, :, s], W3[:, :, s], W2[:, s, :], 2)["out"]
                  for s in S)
        np.testing.assert_allclose(tot, full, rtol=1e-12, atol=1e-13)


# ------------------------------------------------- the pages' own numbers
def test_util_formula_a100_example():
    g = json.load(open(os.path.join(GOLDEN, "util_a100_example.json")))
    b_star = acc.ridge_tokens(g["peak_flops"], g["peak_bw_bytes_per_s"])
    assert b_star == pytest.approx(g["ridge_tokens"])
    assert b_star * g["topk"] / g["n_expert"] == pytest.approx(g["tokens_per_expert_at_ridge"])
    assert acc.util(g["topk"], g["n_expert"], g["peak_bw_bytes_per_s"], g["peak_flops"],
                    g["ridge_tokens"]) == pytest.approx(g["util_at_ridge_batch"])
    assert acc.util(1, 1, g["peak_bw_bytes_per_s"], g["peak_flops"], 1e6) == 1.0


def test_expert_weight_bytes_match_piper_table_iv():
    g = json.load(open(os.path.join(GOLDEN, "piper_table_iv.json")))
    for r in g["rows"]:
        b = acc.expert_weight_bytes(r["d_model"], r["d_ffn"], r["E"])
        assert abs(b / 2**30 - r["send_gb"]) <= 0.01, r
        assert abs(r["send_gb"] / g["bandwidth_gb_per_s"] * 1e3 - r["latency_ms"]) <= 0.05
    wl = I.WORKLOADS
    assert acc.expert_weight_bytes(wl["mixtral_decode"].H, wl["mixtral_decode"].F, 8) \
        == 4.5 * 2**30
    assert acc.expert_weight_bytes(wl["fine_grained"].H, wl["fine_grained"].F, 256) \
        == 21 * 2**30


def test_flop_count_closed_form():
    # one token, one expert: 3 matrices of H x F, 2 flops per multiply-add
    assert acc.ffn_flops(1, 7, 11, 1) == 2 * 3 * 7 * 11
    wl = I.WORKLOADS["fine_grained"]
    assert acc.ffn_flops(wl.T, wl.H, wl.F, wl.k) == 5_772_436_045_824


# ------------------------------------------------------ the workload recipe
def test_skewed_workloads_reach_their_skew():
    lit = I.WORKLOADS["skewed"]
    idx, _ = O.route_topk(I.make_logits(lit).numpy(), lit.k)
    c = O.permute(idx, lit.E)[0]
    assert c.max() == lit.T                     # alpha = 3: every token picks it
    cal = I.WORKLOADS["skewed_10x"]
    idx, _ = O.route_topk(I.make_logits(cal).numpy(), cal.k)
    c = O.permute(idx, cal.E)[0]
    ratio = c.max() / c.mean()
    assert 9.0 <= ratio <= 11.0, ratio
    assert (c > 0).sum() == cal.E


# --------------------------------------------- mutations the pins must catch
def test_pins_catch_planted_mistakes():
    # 1. ties to the higher expert index
    def route_hi(l, k):
        idx, w = O.route_topk(l[:, ::-1], k)
        return (l.shape[1] - 1 - idx).astype(np.int32), w
    with pytest.raises(AssertionError):
        check_topk_brute(route_hi)

    # 2. silu with the sign of the exponent flipped
    def ffn_bad_silu(x, W1e, W3e, W2e):
        g = O._f64(x) @ O._f64(W1e)
        u = O._f64(x) @ O._f64(W3e)
        return (g / (1 + np.exp(g)) * u) @ O._f64(W2e)
    with pytest.raises(AssertionError):
        check_ffn_brute(ffn_bad_silu)

    # 3. gate and up swapped
    with pytest.raises(AssertionError):
        check_ffn_brute(lambda x, a, b, c: O.expert_ffn(x, b, a, c))

    # 4. dropped up-projection term (silu(g) alone)
    def ffn_no_up(x, W1e, W3e, W2e):
        g = O._f64(x) @ O._f64(W1e)
        return O.silu(g) @ O._f64(W2e)
    with pytest.raises(AssertionError):
        check_ffn_brute(ffn_no_up)

    # 5. a transposed operand
    with pytest.raises((AssertionError, ValueError, RuntimeError)):
        check_ffn_brute(lambda x, a, b, c: O.expert_ffn(x, a, b, c.T))

    # 6. an unstable scatter (within an expert, last assignment first)
    def permute_rev(idx, E):
        counts, offsets, src, dest = O.permute(idx, E)
        src = src.copy()
        for e in range(E):
            src[offsets[e]:offsets[e + 1]] = src[offsets[e]:offsets[e + 1]][::-1]
        dest = np.empty_like(src)
        dest[src] = np.arange(len(src))
        return counts, offsets, src, dest
    with pytest.raises(AssertionError):
        check_permute(permute_rev)

    # 8. a weight gradient off by a tenth of a percent
    def backward_bad(x, logits, W1, W3, W2, k, dout):
        g = O.backward(x, logits, W1, W3, W2, k, dout)
        g["dW1"] = g["dW1"] * 1.001
        return g
    with pytest.raises(AssertionError):
        check_backward_autograd(backward_bad)

    # 9. the routing weights left out of dY (dY = dout)
    def backward_unweighted(x, logits, W1, W3, W2, k, dout):
        ones = np.zeros_like(np.asarray(logits, np.float32))
        return O.backward(x, ones, W1, W3, W2, k, dout)
    with pytest.raises(AssertionError):
        check_backward_autograd(backward_unweighted)

    # 7. router computed with the transposed product
    with pytest.raises((AssertionError, ValueError, RuntimeError)):
        check_router_brute(lambda x, Wg: O.router_logits(x, np.asarray(Wg).T))
