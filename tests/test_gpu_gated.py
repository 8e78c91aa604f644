"""The steps either side of the routed path on the GPU: the router projection
logits = x @ Wg and the layer from hidden states with an optional shared
expert, against the oracle.  Routing is an integer decision taken on fp32
logits, so the oracle ranks on the GPU's own router output; the logits
themselves are compared with the oracle's fp64 product."""
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
    rng = np.random.default_rng(2)
    tok = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, 4, replace=False)]))
    ref = O.forward_direct(d["x"], logits.cpu().numpy(), d["W1"], d["W3"], d["W2"], wl.k,
                           tokens=tok)
    if shared is not None:
        ref = ref + O.expert_ffn(d["x"][torch.from_numpy(tok).cuda()], *shared)
    assert_moe_close(out[torch.from_numpy(tok).cuda()], ref, f"{name} gated out")
