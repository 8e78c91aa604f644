"""The steps either side of the routed path on the GPU: the router projection
logits = x @ Wg and the layer from hidden states with an optional shared
expert, against the oracle.  The logits are compared with the oracle's fp64
product.  Routing is an integer decision taken on fp32 logits: the GPU's
top-k on its own logits must equal the oracle's top-k on the oracle's logits
(rounded to fp32) for every token whose decision is not within the logit
tolerance of a tie; the few that are are counted and reported.  The layer's
output is then compared with the oracle ranked on the GPU's router output, so
that such near-ties do not make the comparison of the FFN arithmetic moot."""
import math

import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import assert_moe_close

pytestmark = pytest.mark.gpu

# fp32 accumulation of H bf16 products (exact in fp32): a few 1e-6 for
# O(1) logits; the bound below leaves room for H up to 7168.
LOGIT_ATOL = 1e-4
LOGIT_RTOL = 1e-4

CASES = {  # name: (T, H, F, E, k, Fs)
    "simt_router_E8_shared": (96, 256, 384, 8, 2, 256),
    "simt_router_E16": (300, 512, 256, 16, 4, 0),
    "simt_router_E4": (40, 128, 128, 4, 2, 128),
    "tc_router_E64_shared": (200, 256, 256, 64, 6, 384),
    "tc_router_E128_large": (1000, 256, 256, 128, 4, 0),
    "tc_router_E256_shared": (520, 384, 512, 256, 8, 256),
}


def near_tie_tokens(ref_logits32, k, err):
    """Tokens whose top-k decision (the set and the slot order) could differ
    between the oracle's fp32 logits and logits within `err` of the exact
    product: two neighbours in the descending order of the first k+1 logits
    closer than 2 (err + one fp32 rounding)."""
    l = np.sort(np.asarray(ref_logits32, np.float64), axis=1)[:, ::-1]
    top = l[:, :min(k + 1, l.shape[1])]
    gaps = top[:, :-1] - top[:, 1:]
    band = 2 * (err + 2.0 ** -24 * np.abs(top[:, :-1]))
    return np.nonzero((gaps <= band).any(axis=1))[0] if gaps.size else np.zeros(0, int)


def check_routing_against_oracle(name, gpu_logits, ref_logits, k):
    """GPU top-k on the GPU's logits vs oracle top-k on the oracle's fp32
    logits: equal on every token that is not near a tie, given the largest
    logit error seen."""
    ref32 = np.asarray(ref_logits, np.float32)
    err = float(np.abs(gpu_logits.double().cpu().numpy() - ref_logits).max())
    got = moe.moe_route_topk(gpu_logits, k)[0].cpu().numpy()
    want = O.route_topk(ref32, k)[0]
    near = set(near_tie_tokens(ref32, k, err).tolist())
    diff = np.nonzero((got != want).any(axis=1))[0]
    unexplained = [int(t) for t in diff if t not in near]
    assert not unexplained, (f"{name}: routing differs from the oracle's on tokens "
                             f"{unexplained[:8]} that are not near a tie")
    print(f"{name}: max logit error {err:.2e}; {len(near)} of {len(got)} tokens near a tie, "
          f"{len(diff)} routed differently")
    assert len(near) <= 2 + len(got) // 100, (name, len(near))


def make(name):
    T, H, F, E, k, Fs = CASES[name]
    wl = I.small(name, T=T, H=H, F=F, E=E, k=k)
    d = I.make_inputs(wl, "cpu")
    g = torch.Generator().manual_seed(7)
    d["Wg"] = (torch.randn(H, E, generator=g) / math.sqrt(H)).to(torch.bfloat16)
    if Fs:
        d["Ws1"] = (torch.randn(H, Fs, generator=g) / math.sqrt(H)).to(torch.bfloat16)
        d["Ws3"] = (torch.randn(H, Fs, generator=g) / math.sqrt(H)).to(torch.bfloat16)
        d["Ws2"] = (torch.randn(Fs, H, generator=g) / math.sqrt(Fs)).to(torch.bfloat16)
    return wl, d


@pytest.mark.parametrize("name", list(CASES))
def test_gated_layer_matches_oracle(name):
    wl, d = make(name)
    dev = {n: t.cuda() for n, t in d.items()}
    shared = (dev["Ws1"], dev["Ws3"], dev["Ws2"]) if "Ws1" in dev else None
    logits = moe.moe_router_logits(dev["x"], dev["Wg"])
    ref_l = O.router_logits(d["x"], d["Wg"])
    err = np.abs(logits.double().cpu().numpy() - ref_l)
    assert np.all(err <= LOGIT_ATOL + LOGIT_RTOL * np.abs(ref_l)), err.max()
    check_routing_against_oracle(name, logits, ref_l, wl.k)
    ws = moe.Workspace()
    out = moe.moe_forward_gated(dev["x"], dev["Wg"], dev["W1"], dev["W3"], dev["W2"], wl.k,
                                shared=shared, ws=ws)
    assert moe.moe_get_device_status(ws) == 0
    ref = O.forward_gated(d["x"], d["Wg"], d["W1"], d["W3"], d["W2"], wl.k,
                          shared=None if shared is None else (d["Ws1"], d["Ws3"], d["Ws2"]),
                          logits=logits.cpu().numpy())
    assert_moe_close(out, ref["out"], f"{name} out")
    # without a shared expert the gated layer is moe_forward on its own logits
    plain = moe.moe_forward_gated(dev["x"], dev["Wg"], dev["W1"], dev["W3"], dev["W2"], wl.k)
    again = moe.moe_forward(dev["x"], logits, dev["W1"], dev["W3"], dev["W2"], wl.k)
    assert torch.equal(plain, again)


FULL = {  # workload of record, shared-expert width (0 = none)
    "mixtral_decode": 0,        # E = 8: the SIMT router
    "dbrx_prefill": 0,          # E = 16
    "fine_grained": 2048,       # E = 256: the tensor-core router, plus a shared expert
}


@pytest.mark.parametrize("name", list(FULL))
def test_gated_layer_full_size(name):
    """Full sizes, launched as the gated benchmark launches them: every logit
    against the fp64 product; the output on sampled tokens against the routed
    per-token definition (ranked on the GPU's own fp32 logits) plus the shared
    expert of those tokens."""
    wl, Fs = I.WORKLOADS[name], FULL[name]
    d = I.make_inputs(wl, "cuda")
    g = torch.Generator(device="cuda").manual_seed(6)
    Wg = (torch.randn(wl.H, wl.E, generator=g, device="cuda") / math.sqrt(wl.H)).to(
        torch.bfloat16)
    shared = None
    if Fs:
        shared = tuple((torch.randn(r, c, generator=g, device="cuda") / math.sqrt(r)).to(
            torch.bfloat16) for r, c in ((wl.H, Fs), (wl.H, Fs), (Fs, wl.H)))
    ws = moe.Workspace()
    out = moe.moe_forward_gated(d["x"], Wg, d["W1"], d["W3"], d["W2"], wl.k, shared=shared,
                                ws=ws)
    assert moe.moe_get_device_status(ws) == 0
    logits = moe.moe_router_logits(d["x"], Wg)
    ref_l = O.router_logits(d["x"].cpu(), Wg.cpu())
    err = np.abs(logits.double().cpu().numpy() - ref_l)
    assert np.all(err <= LOGIT_ATOL + LOGIT_RTOL * np.abs(ref_l)), err.max()
    check_routing_against_oracle(name, logits, ref_l, wl.k)
    rng = np.random.default_rng(2)
    tok = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 4, replace=False)]))
    ref = O.forward_direct(d["x"], logits.cpu().numpy(), d["W1"], d["W3"], d["W2"], wl.k,
                           tokens=tok)
    if shared is not None:
        ref = ref + O.expert_ffn(d["x"][torch.from_numpy(tok).cuda()], *shared)
    assert_moe_close(out[torch.from_numpy(tok).cuda()], ref, f"{name} gated out")
