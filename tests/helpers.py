"""Shared test helpers: the output tolerance and GPU input placement."""
import math

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


# ------------------------------------------------------------ the backward
# The GPU keeps g, u, h, y, dY, dg, du, each assignment's dx row and the
# results in bf16 (relative rounding eps = 2^-9) and accumulates in fp32.
# A gradient passes when both hold:
#   elementwise  |gpu - ref| <= 2 eps |ref| + KAPPA eps mag + 1e-6, with mag the
#                oracle's first-order worst case of those roundings (a sum of
#                absolute values, so it admits every sign pattern of them);
#   normwise     ||gpu - ref|| <= NORM_TOL ||ref|| (+ 1e-6 per element), per
#                expert for the weight gradients: random bf16 roundings give
#                about sqrt(r / 3) eps for r roundings in a chain (0.2-0.6% at
#                the test sizes), and 2^-5 leaves more than 5x of that, while a
#                mistake spread over a whole expert (a dropped 16-row K group,
#                a missing block of dY, dg and du exchanged) moves the norm by
#                10% or more -- sums of random-signed terms that the
#                elementwise worst case alone would let through.
BWD_EPS = 2.0 ** -9
BWD_KAPPA = 6
BWD_NORM_TOL = 2.0 ** -5


def backward_mismatches(name, gpu, ref, key):
    """Messages for every way `gpu` misses ref[key] (empty when it passes)."""
    g = gpu.detach().to("cpu", torch.float64).numpy() if isinstance(gpu, torch.Tensor) \
        else np.asarray(gpu, np.float64)
    r = np.asarray(ref[key], np.float64)
    assert g.shape == r.shape, (name, key, g.shape, r.shape)
    msgs = []
    bound = 2 * BWD_EPS * np.abs(r) + BWD_KAPPA * BWD_EPS * np.asarray(ref["mag_" + key]) + 1e-6
    err = np.abs(g - r)
    bad = err > bound
    if bad.any():
        where = [tuple(int(v) for v in i) for i in np.argwhere(bad)[:4]]
        msgs.append(f"{name} {key}: {bad.sum()}/{bad.size} out of the elementwise bound, "
                    f"max err/bound {(err / bound).max():.2f}; first at {where}: gpu "
                    f"{[float(g[w]) for w in where]} ref {[float(r[w]) for w in where]}")
    groups = [(g[e], r[e]) for e in range(r.shape[0])] if key.startswith("dW") else [(g, r)]
    for i, (ge, re) in enumerate(groups):
        dn = float(np.linalg.norm(ge - re))
        lim = BWD_NORM_TOL * float(np.linalg.norm(re)) + 1e-6 * math.sqrt(re.size)
        if dn > lim:
            msgs.append(f"{name} {key}{f'[{i}]' if len(groups) > 1 else ''}: normwise error "
                        f"{dn:.3e} above {lim:.3e} (relative {dn / max(np.linalg.norm(re), 1e-300):.3e})")
            break
    return msgs
