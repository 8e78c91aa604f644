"""Pins the replica planner's oracle (oracle/replica_planner.py) to facts that
do not come from it: brute force over every plan of tiny instances, closed
forms of special cases, and the invariants the planner states ("MegaFlux",
§3.1 and §A.1: routed work is preserved, replica budgets hold, refinement
neither opens replicas nor raises the maximum load; §A.2: reduction-aware
pruning keeps the no-replica plan unless it strictly lowers the penalised
load).  Mutation tests at the end plant plausible mistakes in it."""
import itertools
import math

import numpy as np
import pytest

from oracle import replica_planner as RP


# ------------------------------------------------------------ brute force
def compositions(total, parts):
    """Every way to write `total` as an ordered sum of `parts` non-negative ints."""
    if parts == 1:
        yield (total,)
        return
    for first in range(total + 1):
        for rest in compositions(total - first, parts - 1):
            yield (first,) + rest


def brute_force_best_max_load(b, G, budget):
    """The smallest maximum GPU load over every plan: each GPU holds its own
    experts plus at most `budget` others, and every expert's blocks are split
    over its holders in every possible way."""
    E = len(b)
    own = [RP.owner_of(e, E, G) for e in range(E)]
    best = math.inf
    choices = [[c for r in range(budget + 1)
                for c in itertools.combinations([e for e in range(E) if own[e] != g], r)]
               for g in range(G)]
    for reps in itertools.product(*choices):
        holders = [[own[e]] + [g for g in range(G) if e in reps[g]] for e in range(E)]
        splits = [list(compositions(b[e], len(holders[e]))) for e in range(E)]
        for pick in itertools.product(*splits):
            L = [0] * G
            for e in range(E):
                for g, v in zip(holders[e], pick[e]):
                    L[g] += v
            best = min(best, max(L))
    return best


def check_invariants(counts, G, beta, budget, plan):
    E = len(counts)
    b = [(c + beta - 1) // beta for c in counts]
    n = plan["n"]
    q0_max = max(sum(b[e] for e in range(E) if RP.owner_of(e, E, G) == g) for g in range(G))
    # routed work preserved, nothing negative
    for e in range(E):
        assert sum(n[e]) == b[e]
        assert min(n[e]) >= 0
    # budgets hold; a replica is a non-owner holder with work
    per_gpu = [0] * G
    for g, e in plan["replicas"]:
        assert g != RP.owner_of(e, E, G)
        assert n[e][g] > 0
        per_gpu[g] += 1
    assert max(per_gpu) <= budget
    # only holders get blocks
    reps = set(plan["replicas"])
    for e in range(E):
        for g in range(G):
            if n[e][g]:
                assert g == RP.owner_of(e, E, G) or (g, e) in reps
    # loads add up; the load-only plan is never worse than fixed placement
    assert plan["load"] == [sum(n[e][g] for e in range(E)) for g in range(G)]
    assert max(plan["load"]) <= q0_max
    # rows: each expert's rows cut at block boundaries, ascending GPU order
    for e in range(E):
        pos = 0
        for g in range(G):
            lo, hi = plan["rows"][e][g]
            assert lo == min(pos * beta, counts[e])
            pos += n[e][g]
            assert hi == min(pos * beta, counts[e])
        assert plan["rows"][e][G - 1][1] == counts[e]
    return q0_max


def random_counts(rng, E, scale):
    w = rng.zipf(1.5, E).astype(float)
    return [int(v) for v in np.minimum(w * scale, 50 * scale)]


# ----------------------------------------------------------------- pins
def test_budget_zero_is_fixed_placement():
    counts = [300, 10, 5, 700, 0, 40, 90, 1000]
    p = RP.plan_replicas(counts, 4, 64, budget=0)
    assert p["replicas"] == []
    for e in range(8):
        assert p["n"][e][RP.owner_of(e, 8, 4)] == (counts[e] + 63) // 64


def test_uniform_routing_needs_no_replicas():
    p = RP.plan_replicas([256] * 64, 8, 128, budget=2)
    assert p["replicas"] == [] and p["load"] == [16] * 8


def test_one_hot_expert_reaches_the_balanced_load():
    """One expert with most of the rows and a slot on every GPU: the plan
    reaches tau = ceil(total / G), which brute force confirms is optimal."""
    for G in (2, 3, 4):
        counts = [8 * 128 * G] + [128] * (2 * G - 1)
        p = RP.plan_replicas(counts, G, 128, budget=1)
        b = [(c + 127) // 128 for c in counts]
        tau = math.ceil(sum(b) / G)
        assert max(p["load"]) == tau
        if G <= 3:
            assert brute_force_best_max_load(b, G, 1) == tau


@pytest.mark.parametrize("seed", range(12))
def test_against_brute_force_on_tiny_instances(seed):
    rng = np.random.default_rng(seed)
    G = int(rng.integers(2, 4))
    E = int(rng.integers(G, 5))
    counts = [int(v) for v in rng.integers(0, 5 * 32, E)]
    budget = int(rng.integers(0, 2))
    p = RP.plan_replicas(counts, G, 32, budget)
    q0_max = check_invariants(counts, G, 32, budget, p)
    best = brute_force_best_max_load([(c + 31) // 32 for c in counts], G, budget)
    assert best <= max(p["load"]) <= q0_max
    # a greedy that stops short by more than one block of the optimum on these
    # sizes would be a defect of the search, not of the instance
    assert max(p["load"]) <= best + 1


@pytest.mark.parametrize("seed", range(20))
def test_invariants_on_skewed_instances(seed):
    rng = np.random.default_rng(100 + seed)
    G = int(rng.choice([2, 4, 8]))
    E = G * int(rng.integers(1, 9))
    counts = random_counts(rng, E, int(rng.choice([16, 128, 1024])))
    budget = int(rng.integers(0, 4))
    beta = int(rng.choice([64, 128, 256]))
    p = RP.plan_replicas(counts, G, beta, budget)
    check_invariants(counts, G, beta, budget, p)
    # refinement leaves no single-block move between two holders of an expert
    # that lowers the larger of their loads
    n, L = p["n"], p["load"]
    holders = [{g for g in range(G) if n[e][g] > 0} | {RP.owner_of(e, E, G)} for e in range(E)]
    for e in range(E):
        for g1 in holders[e]:
            for g2 in holders[e]:
                if g1 != g2 and n[e][g1] > 0:
                    assert L[g1] - L[g2] <= 1, (e, g1, g2, L)


def test_refinement_never_raises_the_maximum_load_or_opens_replicas():
    rng = np.random.default_rng(7)
    for _ in range(30):
        G, E = 4, 16
        counts = random_counts(rng, E, 64)
        b = RP.blocks_of(counts, 64)
        tau = math.ceil(sum(b) / G)
        q0 = RP.Plan(b, G)
        for donor in RP.DONOR_ORDERS:
            for fan in RP.FANOUTS:
                c = RP.greedy_search(q0, tau, 2, 4, donor, fan)
                RP.drop_empty_replicas(c)
                before, reps = max(c.load()), set(c.replicas())
                RP.prune_redundant(c)
                RP.single_block_moves(c)
                assert max(c.load()) <= before
                assert set(c.replicas()) <= reps


def test_reduction_aware_pruning():
    counts = [64 * 40] + [64] * 15           # one hot expert on GPU 0 of 4
    load_only = RP.plan_replicas(counts, 4, 64, budget=2)
    assert load_only["replicas"]
    # a huge penalty: no replica pays for itself, so the plan is q0
    p = RP.plan_replicas(counts, 4, 64, budget=2, lam=10 ** 6)
    assert p["replicas"] == [] and p["search"] == "q0"
    # penalty 0: nothing is pruned, and the plan is the load-only one
    p0 = RP.plan_replicas(counts, 4, 64, budget=2, lam=0)
    assert p0["n"] == load_only["n"]
    # the pages' penalty of 12 blocks: replicas with fewer than 12 blocks go,
    # and whatever is kept beats q0 on the penalised load
    p12 = RP.plan_replicas(counts, 4, 64, budget=2, lam=12)
    for g, e in p12["replicas"]:
        assert p12["n"][e][g] >= 12
    if p12["search"] != "q0":
        own = [0] * 4
        for g, e in p12["replicas"]:
            own[RP.owner_of(e, 16, 4)] += 1
        c12 = max(p12["load"][g] + 12 * own[g] for g in range(4))
        assert c12 < 40 + 3


def test_small_batches_keep_fixed_placement_under_the_reduction_penalty():
    """Few tokens per expert: every replica would carry fewer than lambda
    blocks, so the backward plan creates none ("MegaFlux" §4.5: at small
    token counts the reduction-aware planner makes no replicas)."""
    rng = np.random.default_rng(3)
    counts = random_counts(rng, 64, 8)
    p = RP.plan_replicas(counts, 8, 128, budget=2, lam=12)
    assert p["replicas"] == []


def test_plan_is_deterministic():
    rng = np.random.default_rng(11)
    counts = random_counts(rng, 32, 200)
    a = RP.plan_replicas(counts, 8, 128, 2)
    b = RP.plan_replicas(list(counts), 8, 128, 2)
    assert a == b


# --------------------------------------------------------- mutation tests
def test_pins_catch_planted_planner_mistakes(monkeypatch):
    # 1. replicas placed without looking at the budget
    real = RP.Plan.slots_used
    monkeypatch.setattr(RP.Plan, "slots_used", lambda self, g: 0)
    with pytest.raises(AssertionError):
        rng = np.random.default_rng(100)
        for seed in range(20):
            rng = np.random.default_rng(100 + seed)
            G = int(rng.choice([2, 4, 8]))
            E = G * int(rng.integers(1, 9))
            counts = random_counts(rng, E, int(rng.choice([16, 128, 1024])))
            budget = int(rng.integers(0, 4))
            beta = int(rng.choice([64, 128, 256]))
            check_invariants(counts, G, beta, budget, RP.plan_replicas(counts, G, beta, budget))
    monkeypatch.setattr(RP.Plan, "slots_used", real)

    # 2. blocks counted with floor instead of ceil (the partial block lost)
    real_blocks = RP.blocks_of
    monkeypatch.setattr(RP, "blocks_of", lambda counts, beta: [c // beta for c in counts])
    with pytest.raises(AssertionError):
        counts = [300, 10, 5, 700]
        check_invariants(counts, 2, 64, 1, RP.plan_replicas(counts, 2, 64, 1))
    monkeypatch.setattr(RP, "blocks_of", real_blocks)

    # 3. the single-block refinement skipped
    monkeypatch.setattr(RP, "single_block_moves", lambda p: None)
    with pytest.raises(AssertionError):
        for seed in range(20):
            test_invariants_on_skewed_instances(seed)
    monkeypatch.undo()

    # 4. rows handed out in descending GPU order
    real_rows = RP.assign_rows
    monkeypatch.setattr(RP, "assign_rows", lambda c, beta, n: [
        list(reversed(r)) for r in real_rows(c, beta, n)])
    with pytest.raises(AssertionError):
        counts = [300, 10, 5, 700]
        check_invariants(counts, 2, 64, 1, RP.plan_replicas(counts, 2, 64, 1))
