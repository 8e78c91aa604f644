"""The expert-replica planner on the GPU against the oracle's plan, bit for
bit: random instances (the CPU pins' families), the backward plan with the
reduction penalty, and the per-expert counts of the full-size workloads'
routings fed straight from moe_permute on the device."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import replica_planner as RP
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import to_np

pytestmark = pytest.mark.gpu


def compare(counts, G, beta, budget, lam=None, rounds=None, counts_dev=None):
    ref = RP.plan_replicas(list(counts), G, beta, budget, lam=lam, rounds=rounds)
    c = counts_dev if counts_dev is not None else torch.tensor(counts, dtype=torch.int32).cuda()
    n, rows, load, info = moe.moe_plan_replicas(c, G, beta, budget,
                                                -1 if rounds is None else rounds,
                                                -1 if lam is None else lam)
    torch.cuda.synchronize()
    what = f"G={G} E={len(counts)} beta={beta} budget={budget} lam={lam}"
    np.testing.assert_array_equal(to_np(n), np.array(ref["n"]), err_msg=what)
    np.testing.assert_array_equal(to_np(rows), np.array(ref["rows"]), err_msg=what)
    np.testing.assert_array_equal(to_np(load), np.array(ref["load"]), err_msg=what)
    which = 4 if ref["search"] == "q0" else \
        [(d, f) for d in RP.DONOR_ORDERS for f in RP.FANOUTS].index(ref["search"])
    assert to_np(info).tolist() == [which, ref["tau"], len(ref["replicas"]),
                                    max(ref["load"])], what
    return ref


@pytest.mark.parametrize("seed", range(16))
def test_planner_matches_oracle_on_random_instances(seed):
    rng = np.random.default_rng(500 + seed)
    G = int(rng.choice([1, 2, 4, 8, 16]))
    E = G * int(rng.integers(1, 17))
    w = rng.zipf(1.4, E).astype(float)
    counts = np.minimum(w * int(rng.choice([8, 64, 512])), 40000).astype(int).tolist()
    budget = int(rng.integers(0, 5))
    beta = int(rng.choice([64, 128, 256]))
    compare(counts, G, beta, budget)
    compare(counts, G, beta, budget, lam=12)


def test_planner_edge_cases():
    compare([0] * 16, 4, 128, 2)                       # no routed rows
    compare([5], 1, 64, 0)                             # one GPU, one expert
    compare([64 * 40] + [64] * 15, 4, 64, 2)           # one hot expert
    compare([64 * 40] + [64] * 15, 4, 64, 2, lam=12)   # ... pruned back to q0
    compare([64 * 40] + [64] * 15, 4, 64, 2, lam=0)
    compare([1000, 3, 0, 7, 900, 2, 2, 2], 8, 16, 1, rounds=0)


@pytest.mark.parametrize("name", ["fine_grained", "skewed", "skewed_10x", "dbrx_prefill"])
def test_planner_on_workload_routings(name):
    """Counts from the workloads' routings, kept on the device from the
    permute to the planner; 8 GPUs with 25% spare expert slots."""
    wl = I.WORKLOADS[name]
    logits = I.make_logits(wl).cuda()
    idx, _ = moe.moe_route_topk(logits, wl.k)
    counts = moe.moe_permute(idx, wl.E)[0]
    G = 8
    budget = max(1, wl.E // G // 4)
    beta = 256 if wl.T * wl.k > 80 * wl.E else 128
    c = to_np(counts).tolist()
    ref = compare(c, G, beta, budget, counts_dev=counts)
    compare(c, G, beta, budget, lam=12, counts_dev=counts)
    if name == "skewed_10x":   # the hot experts get spread over several GPUs
        assert ref["replicas"]
