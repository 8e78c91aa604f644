"""The layer split over GPUs along the FFN features (expert tensor
parallelism: "MegaScale-Infer", §3.4 Performance Simulation Model, where an
expert GEMM (b_e, h) x (h, h'/tpe) runs on tpe GPUs).

Each of the G ranks holds, for every expert, the slice Fg of its FFN
features: W1[:, :, Fg], W3[:, :, Fg] and W2[:, Fg, :].  Routing does not
depend on the features, so every rank routes all tokens identically and no
token moves between GPUs; each computes its partial output in fp32
(moe_forward_f32), one all-reduce sums the partials, and the sum is rounded
to bf16 once (moe_cast_bf16).  SwiGLU acts feature by feature and the
weighted combine is linear, so the sum over the slices is the layer.

Every rank reads only its own memory: there is no multicast or peer load,
the exchange is the collective.
"""
from __future__ import annotations

import torch

from . import binding

SLICE_ALIGN = 128   # the library's feature granularity


def feature_slice(F: int, world: int, rank: int) -> tuple[int, int]:
    """[lo, hi) of rank's FFN features: contiguous, equal, multiples of 128."""
    if F % (SLICE_ALIGN * world) != 0:
        raise ValueError(f"F={F} does not split into {world} slices of a multiple of "
                         f"{SLICE_ALIGN} features")
    w = F // world
    return rank * w, (rank + 1) * w


def shard_weights(W1: torch.Tensor, W3: torch.Tensor, W2: torch.Tensor, world: int, rank: int):
    """This rank's slices of the expert weights, as contiguous tensors."""
    lo, hi = feature_slice(W1.shape[2], world, rank)
    return (W1[:, :, lo:hi].contiguous(), W3[:, :, lo:hi].contiguous(),
            W2[:, lo:hi, :].contiguous())


def sharded_forward(x, logits, W1s, W3s, W2s, k: int, group=None, partial=None, cast=None,
                    ws=None):
    """The layer from this rank's feature slices: partial (fp32), one
    all-reduce over `group` (skipped when the process group is absent or has
    one rank), then one rounding to bf16.  `partial` and `cast` default to the
    library's moe_forward_f32 and moe_cast_bf16."""
    import torch.distributed as dist
    if partial is None:
        part = binding.moe_forward_f32(x, logits, W1s, W3s, W2s, k, ws=ws)
    else:
        part = partial(x, logits, W1s, W3s, W2s, k)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(part, op=dist.ReduceOp.SUM, group=group)
    return binding.moe_cast_bf16(part) if cast is None else cast(part)
