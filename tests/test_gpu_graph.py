"""moe_forward captured in a CUDA graph (moe_forward_graph_create /
moe_graph_launch): every launch gives moe_forward's bits for the inputs in
the buffers at launch time, on a small-batch layer (one-launch routing,
64-row blocks), a 128-row-block layer and a layer whose FC1 runs on CTA
pairs; and the arguments the capture refuses."""
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import assert_moe_close

pytestmark = pytest.mark.gpu

CASES = {  # name: (T, H, F, E, k)
    "tiny_blocks": (96, 256, 384, 8, 2),
    "small_blocks": (256, 512, 1024, 8, 2),
    "pair_fc1": (700, 512, 512, 4, 2),
}


@pytest.mark.parametrize("name", list(CASES))
def test_graph_launches_match_eager_forward(name):
    T, H, F, E, k = CASES[name]
    wl = I.small(f"graph_{name}", T=T, H=H, F=F, E=E, k=k)
    d = I.make_inputs(wl, "cuda")
    x = d["x"].clone()
    logits = d["logits"].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = moe.ForwardGraph(x, logits, d["W1"], d["W3"], d["W2"], k)
        outs = []
        for r in range(3):   # new inputs in the same buffers before each launch
            xr = I.make_inputs(wl.with_(realization=r), "cuda") if r else d
            x.copy_(xr["x"])
            logits.copy_(xr["logits"])
            out = g.launch().clone()
            ref = moe.moe_forward(x, logits, d["W1"], d["W3"], d["W2"], k)
            assert torch.equal(out, ref), f"launch {r}"
            outs.append((out, x.cpu(), logits.cpu()))
        s.synchronize()
        g.close()
    torch.cuda.current_stream().wait_stream(s)
    out, xc, lc = outs[-1]
    ref = O.forward_perm(xc, lc.numpy(), d["W1"].cpu(), d["W3"].cpu(), d["W2"].cpu(), k)
    assert_moe_close(out, ref["out"], f"{name} graph out")


def test_graph_refuses_the_legacy_stream_and_empty_batches():
    wl = I.small("graph_bad", T=32, H=128, F=128, E=4, k=2)
    d = I.make_inputs(wl, "cuda")
    with pytest.raises(moe.MoeError):   # the legacy default stream cannot be captured
        with torch.cuda.stream(torch.cuda.default_stream()):
            moe.ForwardGraph(d["x"], d["logits"], d["W1"], d["W3"], d["W2"], 2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with pytest.raises(moe.MoeError):
            moe.ForwardGraph(d["x"][:0], d["logits"][:0], d["W1"], d["W3"], d["W2"], 2)
