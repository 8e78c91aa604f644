"""The five workloads of record at full size, through moe_forward exactly as
the benchmark launches it.  Routing and the permutation are compared in full
(bit-exact); the layer output is compared on sampled tokens that the oracle
computes one by one from the per-token definition."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import W_ATOL, assert_moe_close, to_np

pytestmark = pytest.mark.gpu

NAMES = ["mixtral_decode", "dbrx_prefill", "fine_grained", "skewed", "skewed_10x"]


@pytest.mark.parametrize("name", NAMES)
def test_full_size_workload(name):
    wl = I.WORKLOADS[name]
    d = I.make_inputs(wl, "cuda")
    logits_cpu = d["logits"].cpu()
    # routing and permutation: full arrays, bit-exact
    idx_ref, w_ref = O.route_topk(logits_cpu.numpy(), wl.k)
    idx, w = moe.moe_route_topk(d["logits"], wl.k)
    np.testing.assert_array_equal(to_np(idx), idx_ref)
    np.testing.assert_allclose(to_np(w), w_ref, rtol=0, atol=W_ATOL)
    perm_ref = O.permute(idx_ref, wl.E)
    for got, ref in zip(moe.moe_permute(idx, wl.E), perm_ref):
        np.testing.assert_array_equal(to_np(got), ref)
    # the fused layer, twice: bit-reproducible
    ws = moe.Workspace()
    out = moe.moe_forward(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], wl.k, ws=ws)
    out2 = moe.moe_forward(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], wl.k, ws=ws)
    assert moe.moe_get_device_status(ws) == 0
    assert torch.equal(out, out2)
    # sampled tokens against the per-token definition
    rng = np.random.default_rng(0)
    tokens = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 4, replace=False)]))
    ref = O.forward_direct(d["x"], logits_cpu.numpy(), d["W1"], d["W3"], d["W2"], wl.k,
                           tokens=tokens)
    assert_moe_close(out[torch.from_numpy(tokens).cuda()], ref, f"{name} sampled out")
    # properties that hold at any size
    counts = to_np(moe.moe_permute(idx, wl.E)[0])
    assert counts.sum() == wl.T * wl.k
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name", ["mixtral_decode", "dbrx_prefill", "fine_grained"])
def test_full_size_host_buffers(name):
    """moe_forward_host with pinned host buffers gives moe_forward's bits: x and
    the logits are read and the result written in place across the host link
    (117 MB of x at the fine-grained size, each row read once by the gather)."""
    wl = I.WORKLOADS[name]
    d = I.make_inputs(wl, "cuda")
    out = moe.moe_forward(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], wl.k)
    xh, lh = d["x"].cpu().pin_memory(), d["logits"].cpu().pin_memory()
    out_h = moe.moe_forward_host(xh, lh, d["W1"], d["W3"], d["W2"], wl.k)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out_h, out.cpu())


def chosen_experts(counts, E, beta_rows):
    """Experts whose every row is compared: the hottest, one cut into several
    token blocks, the last expert (its tiles end the tile list, where the
    balanced K split cuts them), the coldest non-empty one and the first."""
    nz = np.nonzero(counts)[0]
    pick = [int(np.argmax(counts)), int(nz[-1]), int(nz[np.argmin(counts[nz])]), int(nz[0])]
    multi = np.nonzero(counts > beta_rows)[0]
    if multi.size:
        pick.append(int(multi[len(multi) // 2]))
    return list(dict.fromkeys(pick))


@pytest.mark.parametrize("name", NAMES)
def test_full_size_whole_experts(name):
    """Every row of a few chosen experts at full size: the grouped FFN run on the
    full batch's permutation (the same GEMM launches as the layer's) against the
    oracle's FFN of those experts, element by element."""
    wl = I.WORKLOADS[name]
    d = I.make_inputs(wl, "cuda")
    idx, _ = moe.moe_route_topk(d["logits"], wl.k)
    counts, offsets, sorted_src, _ = moe.moe_permute(idx, wl.E)
    y = moe.moe_grouped_ffn(d["x"], sorted_src, offsets, d["W1"], d["W3"], d["W2"], wl.k)
    torch.cuda.synchronize()
    c, off, src = to_np(counts), to_np(offsets), to_np(sorted_src)
    mean = wl.T * wl.k / wl.E
    beta = 64 if mean <= 40 else 128 if mean <= 80 else 256
    x_cpu = d["x"].cpu()
    for e in chosen_experts(c, wl.E, beta):
        lo, hi = int(off[e]), int(off[e + 1])
        ref = O.expert_ffn(x_cpu[torch.from_numpy(src[lo:hi] // wl.k)], d["W1"][e].cpu(),
                           d["W3"][e].cpu(), d["W2"][e].cpu())
        assert_moe_close(y[lo:hi], ref, f"{name} expert {e} ({hi - lo} rows)")
