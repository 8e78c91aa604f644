"""Shared test helpers: the output tolerance and GPU input placement."""
import numpy as np
import torch

# |gpu - oracle| <= ATOL + RTOL * |oracle|, elementwise (bf16 GPU output,
# fp64 oracle).  The GPU rounds h = silu(g)*u and the expert outputs to bf16
# (relative 2^-9 each) and accumulates in fp32; values are O(1).
ATOL = 1e-2
RTOL = 1e-2
# Routing weights: fp32 softmax on the GPU vs fp64 rounded once on the CPU.
W_ATOL = 2e-6


def assert_moe_close(gpu, ref, what="out"):
    g = gpu.detach().to("cpu", torch.float64).numpy() if isinstance(gpu, torch.Tensor) \
        else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    bad = np.abs(g - r) > ATOL + RTOL * np.abs(r)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first at "
            f"{tuple(i)}: gpu={g[tuple(i)]!r} oracle={r[tuple(i)]!r}; "
            f"max |err| = {np.abs(g - r).max():.3e}")


def to_np(t):
    return t.detach().cpu().numpy()


def gpu_inputs(wl, device="cuda"):
    """Inputs of a workload on the GPU (x and weights drawn there, logits on
    the CPU) plus CPU copies of the small tensors."""
    from routing_grouped_expert_gb300 import inputs as I
    d = I.make_inputs(wl, device)
    return d
