"""moe_permute_noalloc, the permute entry point for callers that cannot
allocate device memory (its scratch is a fixed array inside the library),
called through the C ABI and compared with moe_permute, which takes a
caller-allocated workspace.  The permutation is integer work, so the two
must agree bit for bit.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

import routing_grouped_expert_gb300 as moe
from routing_grouped_expert_gb300 import binding

pytestmark = pytest.mark.gpu


def permute_noalloc(topk_idx: torch.Tensor, E: int):
    lib = binding.load_library()
    T, k = topk_idx.shape
    dev = topk_idx.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_src = torch.empty(T * k, dtype=torch.int32, device=dev)
    dest_of = torch.empty(T * k, dtype=torch.int32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.moe_permute_noalloc(p(topk_idx), T, E, k, p(counts), p(offsets), p(sorted_src),
                                 p(dest_of),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, binding.moe_status_string(rc)
    return counts, offsets, sorted_src, dest_of


def routed(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g).cuda()
    return moe.moe_route_topk(logits, k)[0]


def test_noalloc_permute_matches_workspace_permute_on_consecutive_calls():
    # Two calls in a row with different sizes: the second runs on the scratch
    # the first one left behind.
    for T, E, k, seed in ((1000, 64, 6, 1), (300, 8, 2, 2), (8192, 256, 8, 3)):
        idx = routed(T, E, k, seed)
        got = permute_noalloc(idx, E)
        want = moe.moe_permute(idx, E)
        torch.cuda.synchronize()
        for name, g, w in zip(("counts", "offsets", "sorted_src", "dest_of"), got, want):
            assert torch.equal(g, w), f"{name} differs at T={T} E={E} k={k}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = binding.load_library()
    fake = ctypes.c_void_p(4096)      # never dereferenced: rejected on the host
    # T=100000, k=8, E=1024 needs ~6.4 MB of scratch, more than the array holds.
    rc = lib.moe_permute_noalloc(fake, 100000, 1024, 8, fake, fake, fake, fake, None)
    assert rc == 4, binding.moe_status_string(rc)      # MOE_ERR_WORKSPACE
    assert lib.moe_permute_noalloc(fake, 10, 8, 9, fake, fake, fake, fake, None) == 1
