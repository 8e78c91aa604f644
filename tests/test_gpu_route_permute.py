"""Routing and permutation on the GPU against the oracle: bit-exact indices,
counts, offsets and permutation; weights within W_ATOL."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from tests.helpers import W_ATOL, to_np

pytestmark = pytest.mark.gpu

SHAPES = [  # (T, E, k)
    (1, 1, 1), (7, 4, 4), (33, 8, 1), (300, 8, 2), (1000, 16, 4), (129, 37, 5),
    (513, 256, 8), (200, 64, 32), (64, 1024, 8), (4097, 128, 6),
]


def logits_for(T, E, kind, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return torch.randn(T, E, generator=g)
    # many exact ties, signed zeros
    v = torch.tensor([-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 2.0])
    return v[torch.randint(0, len(v), (T, E), generator=g)]


@pytest.mark.parametrize("T,E,k", SHAPES)
@pytest.mark.parametrize("kind", ["normal", "ties"])
def test_route_and_permute_bit_exact(T, E, k, kind):
    l_cpu = logits_for(T, E, kind, seed=T * 1000 + E + k).float()
    idx_ref, w_ref = O.route_topk(l_cpu.numpy(), k)
    idx, w = moe.moe_route_topk(l_cpu.cuda(), k)
    np.testing.assert_array_equal(to_np(idx), idx_ref)
    np.testing.assert_allclose(to_np(w), w_ref, rtol=0, atol=W_ATOL)
    counts_ref, off_ref, src_ref, dest_ref = O.permute(idx_ref, E)
    counts, off, src, dest = moe.moe_permute(idx, E)
    np.testing.assert_array_equal(to_np(counts), counts_ref)
    np.testing.assert_array_equal(to_np(off), off_ref)
    np.testing.assert_array_equal(to_np(src), src_ref)
    np.testing.assert_array_equal(to_np(dest), dest_ref)


def test_permute_of_arbitrary_indices():
    """moe_permute takes any in-range index table, duplicates included."""
    g = torch.Generator().manual_seed(3)
    idx = torch.randint(0, 12, (777, 3), generator=g, dtype=torch.int32)
    ref = O.permute(idx.numpy(), 12)
    got = moe.moe_permute(idx.cuda(), 12)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(to_np(a), b)


def test_empty_batch():
    idx, w = moe.moe_route_topk(torch.empty(0, 8, device="cuda"), 2)
    assert idx.shape == (0, 2)
    counts, off, src, dest = moe.moe_permute(idx, 8)
    assert to_np(counts).sum() == 0 and np.all(to_np(off) == 0)
    assert src.numel() == 0 and dest.numel() == 0


def test_nonfinite_logit_reported_and_indices_stay_in_range():
    l = torch.randn(100, 16)
    l[5, 3] = float("nan")
    l[17, 0] = float("inf")
    l[40, 9] = float("-inf")
    ws = moe.Workspace()
    idx, _ = moe.moe_route_topk(l.cuda(), 4, ws=ws)
    assert moe.moe_get_device_status(ws) == 2   # MOE_ERR_NONFINITE
    i = to_np(idx)
    assert i.min() >= 0 and i.max() < 16
    # finite logits on the same workspace clear the status
    moe.moe_route_topk(torch.randn(100, 16).cuda(), 4, ws=ws)
    assert moe.moe_get_device_status(ws) == 0


def expected_with_bad_indices(idx, E):
    """What the permute must give when some expert indices are out of range:
    the valid assignments grouped exactly as the oracle groups them (the bad
    ones relabelled as an extra expert E, which sorts them last), and -1 for
    the bad ones' dest_of and for the tail of sorted_src."""
    flat = idx.reshape(-1).copy()
    bad = (flat < 0) | (flat >= E)
    flat[bad] = E
    counts, offsets, src, dest = O.permute(flat.reshape(idx.shape), E + 1)
    src = src.copy()
    dest = dest.copy()
    src[offsets[E]:] = -1
    dest[bad] = -1
    return counts[:E], offsets[:E + 1], src, dest


def test_out_of_range_expert_index_reported_and_marked():
    idx = torch.randint(0, 8, (700, 2), dtype=torch.int32, generator=torch.Generator().manual_seed(9))
    idx[10, 1] = 8
    idx[20, 0] = -1
    idx[650, 1] = 1 << 30
    ws = moe.Workspace()
    # outputs pre-filled with garbage: the marks must be written, not left over
    out = tuple(torch.full((n,), 12345, dtype=torch.int32, device="cuda")
                for n in (8, 9, 1400, 1400))
    counts, off, src, dest = moe.moe_permute(idx.cuda(), 8, ws=ws, out=out)
    assert moe.moe_get_device_status(ws) == 1   # MOE_ERR_INVALID_ARG
    want = expected_with_bad_indices(idx.numpy(), 8)
    for name, got, w in zip(("counts", "offsets", "sorted_src", "dest_of"),
                            (counts, off, src, dest), want):
        np.testing.assert_array_equal(to_np(got), w, err_msg=name)


def test_combine_skips_assignments_that_took_no_position():
    """A slot with dest_of = -1 adds nothing: out[t] sums its valid slots."""
    T, H, k = 50, 256, 3
    g = torch.Generator().manual_seed(3)
    y = torch.randn(T * k, H, generator=g).to(torch.bfloat16)
    dest = torch.randperm(T * k, generator=g).to(torch.int32)
    w = torch.rand(T, k, generator=g)
    dest[7] = -1
    dest[100] = -1
    out = moe.moe_combine(y.cuda(), dest.cuda(), w.cuda())
    d = dest.numpy().reshape(T, k)
    ref = np.zeros((T, H))
    for j in range(k):        # slot order, the oracle's combine on the valid slots
        ok = d[:, j] >= 0
        ref[ok] += w.numpy()[ok, j:j + 1].astype(np.float64) * \
            y.double().numpy()[d[ok, j]]
    np.testing.assert_allclose(to_np(out.double()), ref, rtol=2 ** -8, atol=1e-6)


def test_route_is_deterministic():
    l = torch.randn(5000, 256).cuda()
    a = moe.moe_route_topk(l, 8)
    b = moe.moe_route_topk(l, 8)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    pa = moe.moe_permute(a[0], 256)
    pb = moe.moe_permute(b[0], 256)
    for x, y in zip(pa, pb):
        assert torch.equal(x, y)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (96, 8, 2), (256, 8, 2), (2048, 8, 2),
                                   (512, 256, 8), (4096, 16, 1), (33, 37, 5), (4100, 16, 1),
                                   (600, 300, 4)])
def test_forward_routing_bit_exact(T, E, k):
    """The routing moe_forward itself computed, copied out of the workspace,
    against the oracle: bit-exact indices and permutation."""
    from routing_grouped_expert_gb300 import inputs as I
    wl = I.small("routing", T=T, H=128, F=128, E=E, k=k)
    d = {n: t.cuda() for n, t in I.make_inputs(wl, "cpu").items()}
    for kind in ("normal", "ties"):
        logits = logits_for(T, E, kind, seed=T + E + k).float()
        ws = moe.Workspace()
        moe.moe_forward(d["x"], logits.cuda(), d["W1"], d["W3"], d["W2"], k, ws=ws)
        assert moe.moe_get_device_status(ws) == 0
        idx, w, counts, off, src, dest = moe.moe_forward_routing(ws, T, 128, 128, E, k)
        idx_ref, w_ref = O.route_topk(logits.numpy(), k)
        np.testing.assert_array_equal(to_np(idx), idx_ref)
        np.testing.assert_allclose(to_np(w), w_ref, rtol=0, atol=W_ATOL)
        for name, got, ref in zip(("counts", "offsets", "sorted_src", "dest_of"),
                                  (counts, off, src, dest), O.permute(idx_ref, E)):
            np.testing.assert_array_equal(to_np(got), ref, err_msg=f"{name} {kind}")

