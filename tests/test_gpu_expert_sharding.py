"""Expert-tensor sharding along the FFN features ("MegaScale-Infer", §3.4, tpe),
emulated on one GPU: the layer run on G feature slices of every expert (what G
GPUs would each hold) and summed equals the whole layer.  Routing does not
depend on F, so each slice routes identically; the sum is the one exchange
step a multi-GPU run would do with an all-reduce."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import assert_moe_close

pytestmark = pytest.mark.gpu

CASES = {  # name: (T, H, F, E, k, slices)
    "decode_like_2": (64, 512, 1024, 8, 2, 2),
    "large_blocks_4": (600, 256, 512, 2, 2, 4),
    "many_experts_2": (300, 256, 256, 32, 4, 2),
    "fine_grained_like_2": (512, 512, 512, 16, 8, 2),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fp32_partials_sum_to_the_layer(name):
    """The feature-sharded runner's arithmetic on one GPU: moe_forward_f32 on
    each slice (unrounded fp32 partials), summed in fp32 as the all-reduce
    would, rounded to bf16 once by moe_cast_bf16."""
    from routing_grouped_expert_gb300 import sharded
    T, H, F, E, k, G = CASES[name]
    wl = I.small(name, T=T, H=H, F=F, E=E, k=k)
    d = I.make_inputs(wl, "cpu")
    dev = {n: t.cuda() for n, t in d.items()}
    acc = torch.zeros(T, H, dtype=torch.float32, device="cuda")
    for r in range(G):
        W1s, W3s, W2s = sharded.shard_weights(dev["W1"], dev["W3"], dev["W2"], G, r)
        acc += moe.moe_forward_f32(dev["x"], dev["logits"], W1s, W3s, W2s, k)
    out = moe.moe_cast_bf16(acc)
    ref = O.forward_perm(d["x"], d["logits"].numpy(), d["W1"], d["W3"], d["W2"], k)["out"]
    assert_moe_close(out, ref, f"{name}: fp32 partials of {G} feature slices")
    # the unsharded fp32 output rounds to the plain layer's bits
    whole = moe.moe_forward_f32(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], k)
    plain = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], k)
    assert torch.equal(moe.moe_cast_bf16(whole), plain)
    assert torch.equal(whole.to(torch.bfloat16), plain)


@pytest.mark.parametrize("name", list(CASES))
def test_feature_slices_sum_to_the_layer(name):
    T, H, F, E, k, G = CASES[name]
    wl = I.small(name, T=T, H=H, F=F, E=E, k=k)
    d = I.make_inputs(wl, "cpu")
    dev = {n: t.cuda() for n, t in d.items()}
    full = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], k)
    acc = torch.zeros(T, H, dtype=torch.float32, device="cuda")
    for s in np.split(np.arange(F), G):
        s = torch.from_numpy(s).cuda()
        part = moe.moe_forward(dev["x"], dev["logits"], dev["W1"][:, :, s].contiguous(),
                               dev["W3"][:, :, s].contiguous(), dev["W2"][:, s, :].contiguous(),
                               k)
        acc += part.float()
    ref = O.forward_perm(d["x"], d["logits"].numpy(), d["W1"], d["W3"], d["W2"], k)["out"]
    assert_moe_close(acc, ref, f"{name}: sum over {G} feature slices")
    assert_moe_close(full, ref, f"{name}: whole layer")
