"""Grouped FFN, combine and the fused forward on the GPU against the oracle,
at sizes the oracle finishes in seconds that still span several tiles and
ragged tails (token blocks of 128 rows, feature tiles of 128, K stages of
64)."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import assert_moe_close, to_np

pytestmark = pytest.mark.gpu

CASES = {  # name: (T, H, F, E, k, skew_alpha)
    "dense_E1_k1": (200, 256, 384, 1, 1, 0.0),
    "ragged_small": (300, 256, 384, 4, 2, 0.0),
    "tiny_config": (256, 512, 1024, 8, 2, 0.0),
    "decode_like": (64, 1024, 2048, 8, 2, 0.0),
    "many_experts": (777, 384, 256, 64, 6, 0.0),
    "skewed": (600, 256, 512, 32, 4, 3.0),
    "single_token": (1, 128, 128, 4, 2, 0.0),
    "k_equals_E": (50, 128, 256, 3, 3, 0.0),
    # > 128 rows per expert: 256-row blocks; F >= 4096 pairs two W2 tiles in FC2
    "large_blocks_paired_fc2": (600, 512, 4096, 2, 2, 0.0),
    # decode-like (64-row blocks) with a long FC2 K range
    "decode_long_k": (48, 256, 1024, 8, 2, 0.0),
    # more tokens than a grid's y dimension holds (65535)
    "many_tokens": (70000, 128, 128, 4, 1, 0.0),
    # the header's limits: 1024 experts, top-32 (most experts get 0-4 rows)
    "max_experts_topk": (64, 128, 128, 1024, 32, 0.0),
    # FC2 tiles (320) not a multiple of the SMs: a balanced K split cuts some
    # tiles between two CTAs (64- and 128-row blocks)
    "split_fc2_tiny": (64, 2560, 1024, 16, 2, 0.0),
    "split_fc2_small": (400, 2560, 512, 16, 2, 0.0),
}


def make(name):
    T, H, F, E, k, a = CASES[name]
    wl = I.small(name, T=T, H=H, F=F, E=E, k=k, skew_alpha=a)
    d = I.make_inputs(wl, "cpu")
    return wl, d


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    wl, d = make(request.param)
    ref = O.forward_perm(d["x"], d["logits"].numpy(), d["W1"], d["W3"], d["W2"], wl.k)
    dev = {n: t.cuda() for n, t in d.items()}
    return wl, d, dev, ref


def test_grouped_ffn_matches_oracle(case):
    wl, d, dev, ref = case
    src = torch.from_numpy(ref["sorted_src"]).cuda()
    off = torch.from_numpy(ref["offsets"]).cuda()
    y = moe.moe_grouped_ffn(dev["x"], src, off, dev["W1"], dev["W3"], dev["W2"], wl.k)
    assert_moe_close(y, ref["y_sorted"], "y_sorted")


def test_combine_matches_oracle(case):
    wl, d, dev, ref = case
    # feed the oracle's own y (rounded to bf16) so only the combine is tested
    y = torch.from_numpy(ref["y_sorted"]).to(torch.bfloat16).cuda()
    dest = torch.from_numpy(ref["dest_of"]).cuda()
    w = torch.from_numpy(ref["topk_w"]).cuda()
    out = moe.moe_combine(y, dest, w)
    want = O.combine(y.double().cpu().numpy(), ref["dest_of"], ref["topk_w"])
    np.testing.assert_allclose(out.double().cpu().numpy(), want, rtol=2 ** -8, atol=1e-6)


def test_forward_matches_oracle(case):
    wl, d, dev, ref = case
    out = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], wl.k)
    assert_moe_close(out, ref["out"], "out")
    direct = O.forward_direct(d["x"], d["logits"].numpy(), d["W1"], d["W3"], d["W2"], wl.k)
    assert_moe_close(out, direct, "out vs per-token definition")


def test_forward_is_bit_reproducible(case):
    wl, d, dev, ref = case
    a = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], wl.k)
    b = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], wl.k)
    assert torch.equal(a, b)


def test_forward_host_matches_device(case):
    wl, d, dev, ref = case
    out_d = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], wl.k)
    xh = d["x"].pin_memory()
    lh = d["logits"].pin_memory()
    out_h = moe.moe_forward_host(xh, lh, dev["W1"], dev["W3"], dev["W2"], wl.k)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out_h, out_d.cpu())
    # pageable buffers take the staging copies: same bits
    out_p = torch.empty_like(out_h, device="cpu")
    moe.moe_forward_host(d["x"].clone(), d["logits"].clone(), dev["W1"], dev["W3"], dev["W2"],
                         wl.k, out_host=out_p)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out_p, out_d.cpu())


def test_status_ok_after_forward(case):
    wl, d, dev, ref = case
    ws = moe.Workspace()
    moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], wl.k, ws=ws)
    assert moe.moe_get_device_status(ws) == 0


def test_identical_experts_give_dense_ffn():
    wl = I.small("ident", T=160, H=256, F=256, E=6, k=3)
    d = I.make_inputs(wl.with_(E=1), "cpu")
    W1, W3, W2 = (d[n].expand(6, *d[n].shape[1:]).contiguous() for n in ("W1", "W3", "W2"))
    logits = torch.randn(160, 6, generator=torch.Generator().manual_seed(9))
    out = moe.moe_forward(d["x"].cuda(), logits.cuda(), W1.cuda(), W3.cuda(), W2.cuda(), 3)
    dense = O.expert_ffn(d["x"], d["W1"][0], d["W3"][0], d["W2"][0])
    assert_moe_close(out, dense, "identical experts vs dense FFN")


def test_empty_batch_forward():
    wl = I.small("empty", T=0, H=128, F=128, E=4, k=2)
    W1, W3, W2 = (t.cuda() for t in I.make_weights(wl, "cpu"))
    out = moe.moe_forward(torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"),
                          torch.empty(0, 4, device="cuda"), W1, W3, W2, 2)
    assert out.shape == (0, 128)


def test_fused_and_stepwise_paths_agree_bit_for_bit(case):
    wl, d, dev, ref = case
    out = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], wl.k)
    idx, w = moe.moe_route_topk(dev["logits"], wl.k)
    counts, off, src, dest = moe.moe_permute(idx, wl.E)
    y = moe.moe_grouped_ffn(dev["x"], src, off, dev["W1"], dev["W3"], dev["W2"], wl.k)
    assert torch.equal(moe.moe_combine(y, dest, w), out)
