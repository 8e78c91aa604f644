"""moe_permute_noalloc, the permute entry point for callers that cannot
allocate device memory (its scratch is a fixed array inside the library):
called through the C ABI and compared bit for bit with the oracle's
permutation and with moe_permute, which takes a caller-allocated workspace.
The permutation is integer work, so all three must agree exactly.  This file
is collected last on purpose, and each case also runs on its own."""
import ctypes

import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import binding

pytestmark = pytest.mark.gpu


def permute_noalloc(topk_idx: torch.Tensor, E: int, stream=None, fill=None):
    lib = binding.load_library()
    T, k = topk_idx.shape
    dev = topk_idx.device
    outs = [torch.empty(n, dtype=torch.int32, device=dev) for n in (E, E + 1, T * k, T * k)]
    if fill is not None:
        for t in outs:
            t.fill_(fill)
    counts, offsets, sorted_src, dest_of = outs
    s = stream if stream is not None else torch.cuda.current_stream()
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())   # inputs and fills are ready
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.moe_permute_noalloc(p(topk_idx), T, E, k, p(counts), p(offsets), p(sorted_src),
                                 p(dest_of), ctypes.c_void_p(s.cuda_stream))
    assert rc == 0, binding.moe_status_string(rc)
    s.synchronize()
    return counts, offsets, sorted_src, dest_of


def routed(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    return O.route_topk(logits.numpy(), k)[0]


def check_against_oracle(got, idx, E, what):
    want = O.permute(idx, E)
    for name, g, w in zip(("counts", "offsets", "sorted_src", "dest_of"), got, want):
        np.testing.assert_array_equal(g.cpu().numpy(), w, err_msg=f"{name} {what}")


def test_noalloc_permute_matches_oracle_and_workspace_permute_on_consecutive_calls():
    # Calls in a row with different sizes: each runs on the scratch the one
    # before it left behind.
    for T, E, k, seed in ((1000, 64, 6, 1), (300, 8, 2, 2), (8192, 256, 8, 3), (5, 1024, 32, 4)):
        idx = routed(T, E, k, seed)
        idx_d = torch.from_numpy(idx).cuda()
        got = permute_noalloc(idx_d, E, fill=-7)
        check_against_oracle(got, idx, E, f"T={T} E={E} k={k}")
        want = moe.moe_permute(idx_d, E)
        torch.cuda.synchronize()
        for name, g, w in zip(("counts", "offsets", "sorted_src", "dest_of"), got, want):
            assert torch.equal(g, w), f"{name} differs from moe_permute at T={T} E={E} k={k}"


def test_noalloc_permute_on_a_side_stream():
    idx = routed(4000, 128, 4, 5)
    side = torch.cuda.Stream()
    got = permute_noalloc(torch.from_numpy(idx).cuda(), 128, stream=side, fill=99)
    check_against_oracle(got, idx, 128, "side stream")


def test_noalloc_empty_batch_zeroes_counts_and_offsets():
    idx = torch.empty(0, 4, dtype=torch.int32, device="cuda")
    counts, offsets, _, _ = permute_noalloc(idx, 16, fill=5)
    assert not counts.any() and not offsets.any()


def test_noalloc_marks_out_of_range_indices():
    idx = routed(600, 8, 2, 6)
    idx[3, 1] = 8
    idx[500, 0] = -2
    got = permute_noalloc(torch.from_numpy(idx).cuda(), 8, fill=777)
    flat = idx.reshape(-1).copy()
    bad = (flat < 0) | (flat >= 8)
    flat[bad] = 8                                   # an extra expert sorts them last
    counts, offsets, src, dest = O.permute(flat.reshape(idx.shape), 9)
    src, dest = src.copy(), dest.copy()
    src[offsets[8]:] = -1
    dest[bad] = -1
    for name, g, w in zip(("counts", "offsets", "sorted_src", "dest_of"), got,
                          (counts[:8], offsets[:9], src, dest)):
        np.testing.assert_array_equal(g.cpu().numpy(), w, err_msg=name)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = binding.load_library()
    fake = ctypes.c_void_p(4096)      # never dereferenced: rejected on the host
    # T=100000, k=8, E=1024 needs ~6.4 MB of scratch, more than the array holds.
    rc = lib.moe_permute_noalloc(fake, 100000, 1024, 8, fake, fake, fake, fake, None)
    assert rc == 4, binding.moe_status_string(rc)      # MOE_ERR_WORKSPACE
    assert lib.moe_permute_noalloc(fake, 10, 8, 9, fake, fake, fake, fake, None) == 1
