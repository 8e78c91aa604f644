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


def test_out_of_range_expert_index_reported():
    idx = torch.randint(0, 8, (64, 2), dtype=torch.int32)
    idx[10, 1] = 8
    idx[20, 0] = -1
    ws = moe.Workspace()
    moe.moe_permute(idx.cuda(), 8, ws=ws)
    assert moe.moe_get_device_status(ws) == 1   # MOE_ERR_INVALID_ARG


def test_route_is_deterministic():
    l = torch.randn(5000, 256).cuda()
    a = moe.moe_route_topk(l, 8)
    b = moe.moe_route_topk(l, 8)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    pa = moe.moe_permute(a[0], 256)
    pb = moe.moe_permute(b[0], 256)
    for x, y in zip(pa, pb):
        assert torch.equal(x, y)
