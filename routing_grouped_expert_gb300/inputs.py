"""Seeded synthetic workloads for the MoE expert-layer forward.

This module only draws random inputs; it holds none of the layer's arithmetic
(no routing, no permutation, no FFN).  Both the CUDA path and the CPU oracle
are fed from here, so they always see identical values.

Shapes follow the model families the pages measure on: Mixtral-8x22B and
DBRX ("MegaScale-Infer: Serving Mixture-of-Experts at Scale with Disaggregated
Expert Parallelism", evaluation models; "Piper", Table I) and DeepSeek-V3-style
fine-grained experts ("Piper", Table I and Table IV).  The pages measure on
production traces and checkpoints, which are not available; seeded Gaussian
inputs of the same shapes stand in for them, and a Zipf-shaped per-expert
logit bias stands in for the trace-derived skewed routes ("MegaFlux", §B.1).

Recipe (every workload):
  router logits  fp32 [T, E] ~ N(0, 1), drawn on the CPU with seed 0,
                 plus bias_e for the skewed workloads;
  x              bf16 [T, H] ~ N(0, 1), seed 1;
  W1 (gate)      bf16 [E, H, F] ~ N(0, 1/H), seed 2;
  W3 (up)        bf16 [E, H, F] ~ N(0, 1/H), seed 3;
  W2 (down)      bf16 [E, F, H] ~ N(0, 1/F), seed 4;
  expert ranking for the skew bias: a random permutation, seed 5.
Weights are drawn one expert at a time in fp32 and rounded to bf16, so the
transient fp32 buffer is one expert's matrix.  Further realizations of a
workload (the benchmark's median over several) shift every seed by 1000 r.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    F: int
    E: int
    k: int
    skew_alpha: float = 0.0   # 0 = uniform routing
    zipf_s: float = 1.2
    note: str = ""
    realization: int = 0      # r > 0: every seed below shifted by 1000 r

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five workloads of record.  `skewed` takes the bias literally
# (alpha = 3 on the natural log of the Zipf weight); under it every token
# picks the hottest expert.  `skewed_10x` uses the smaller alpha that gives
# the hottest expert about ten times the mean count, which is the skew the
# workload description aims at.
WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=512, F=1024, E=8, k=2,
                     note="tiny MoE layer, uniform routing"),
    "mixtral_decode": Workload("mixtral_decode", T=128, H=6144, F=16384, E=8, k=2,
                               note="Mixtral-8x22B-shaped layer, decode batch"),
    "dbrx_prefill": Workload("dbrx_prefill", T=4096, H=6144, F=10752, E=16, k=4,
                             note="DBRX-shaped layer, prefill chunk"),
    "fine_grained": Workload("fine_grained", T=8192, H=7168, F=2048, E=256, k=8,
                             note="DeepSeek-style fine-grained experts"),
    "skewed": Workload("skewed", T=8192, H=7168, F=2048, E=256, k=8, skew_alpha=3.0,
                       note="fine-grained shapes, Zipf(1.2) logit bias, alpha=3 (literal)"),
    "skewed_10x": Workload("skewed_10x", T=8192, H=7168, F=2048, E=256, k=8,
                           skew_alpha=0.27,
                           note="fine-grained shapes, Zipf(1.2) logit bias, alpha=0.27 "
                                "(hottest expert ~10x the mean count)"),
}

SEED_LOGITS, SEED_X, SEED_W1, SEED_W3, SEED_W2, SEED_PERM = 0, 1, 2, 3, 4, 5


def zipf_bias(E: int, alpha: float, s: float = 1.2, seed: int = SEED_PERM) -> torch.Tensor:
    """bias_e = alpha * ln(w_rank(e)), w_r = r^-s / sum_r' r'^-s, ranks 1..E
    assigned to experts by a seeded random permutation.  fp64, CPU."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(E, generator=g)                 # rank-1 of expert e
    r = torch.arange(1, E + 1, dtype=torch.float64)
    w = r.pow(-s)
    w = w / w.sum()
    return alpha * torch.log(w[perm])


def _seed(wl: Workload, base: int) -> int:
    return base + 1000 * wl.realization


def make_logits(wl: Workload) -> torch.Tensor:
    """fp32 [T, E] router logits, always drawn on the CPU."""
    g = torch.Generator().manual_seed(_seed(wl, SEED_LOGITS))
    logits = torch.randn(wl.T, wl.E, generator=g, dtype=torch.float32)
    if wl.skew_alpha != 0.0:
        logits = logits + zipf_bias(wl.E, wl.skew_alpha, wl.zipf_s,
                                    seed=_seed(wl, SEED_PERM)).to(torch.float32)
    return logits


def _randn_bf16(shape, std: float, gen: torch.Generator, device) -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def make_x(wl: Workload, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device).manual_seed(_seed(wl, SEED_X))
    return _randn_bf16((wl.T, wl.H), 1.0, g, device)


def make_weights(wl: Workload, device="cpu"):
    """(W1, W3, W2) bf16: W1, W3 [E, H, F] ~ N(0, 1/H); W2 [E, F, H] ~ N(0, 1/F)."""
    out = []
    for seed, (r, c), std in ((SEED_W1, (wl.H, wl.F), 1.0 / math.sqrt(wl.H)),
                              (SEED_W3, (wl.H, wl.F), 1.0 / math.sqrt(wl.H)),
                              (SEED_W2, (wl.F, wl.H), 1.0 / math.sqrt(wl.F))):
        g = torch.Generator(device=device).manual_seed(_seed(wl, seed))
        W = torch.empty(wl.E, r, c, dtype=torch.bfloat16, device=device)
        for e in range(wl.E):
            W[e] = _randn_bf16((r, c), std, g, device)
        out.append(W)
    return tuple(out)


def make_inputs(wl: Workload, device="cpu"):
    """All inputs of one forward: dict with x, logits, W1, W3, W2 on `device`."""
    W1, W3, W2 = make_weights(wl, device)
    return dict(x=make_x(wl, device), logits=make_logits(wl).to(device),
                W1=W1, W3=W3, W2=W2)


def small(name: str, **kw) -> Workload:
    """A named ad-hoc workload (for parity tests at sizes the oracle finishes
    in seconds)."""
    return Workload(name, **kw)
