"""CPU oracle of the expert-replica planner -- TEST INFRASTRUCTURE.

Only the test suite may import this module; the library never does, and it
imports nothing from the library package.

What it computes: for expert-parallel execution on G GPUs, where each GPU
owns a contiguous range of experts, a plan that moves token blocks of
overloaded GPUs' experts to replicas of those experts on underloaded GPUs,
under a per-GPU budget of replica slots, without changing any routed
assignment ("MegaFlux: Skew-Resilient MoE Megakernels via Pipelined Expert
Replication", §3.1 Planner; §A.1 Greedy placement and refinement; §A.2
Reduction-aware planning).  The steps, in the pages' order:

  1. blocks: each expert's routed rows are cut into ceil(c_e / beta) blocks of
     beta rows, the last one partial (§3.1: at most one partial block per
     expert); the block count is the load proxy (§3.1);
  2. the no-replica assignment q0: every block on its expert's owner;
  3. four bounded greedy searches from q0, two donor priorities x two
     fan-out strategies (one new replica per expert per round, or several);
     a new replica goes to the least-loaded eligible GPU below the target
     load tau that has a free slot and does not hold the expert yet; a
     search stops after s + 2 rounds or after a round that moved nothing
     (§A.1);
  4. the candidate with the smallest maximum GPU load wins, ties going to the
     one with fewer replicas (§A.1);
  5. refinement: redundant replicas are pruned and single blocks move between
     GPUs that share an expert; neither opens a replica or raises the maximum
     load (§A.1);
  6. for backward plans, reduction-aware pruning with penalty lambda per
     remote replica charged to the expert's owner; the pruned plan is kept
     only if it strictly lowers the penalised maximum C_lambda below that of
     q0, else the plan is q0 (§A.2);
  7. the rows of each expert, in their routed order, are cut into its blocks
     and handed to the GPUs holding it in ascending GPU order, as many blocks
     each as the plan gives it (§A.2, routed-assignment ordering).

Readings where the pages leave a step open (each is listed in the design
notes):
  * owner(e) = floor(e * G / E): contiguous, equal ranges of experts;
  * tau = ceil(total blocks / G), the balanced load;
  * s, the length parameter of the searches, is the per-GPU replica budget;
  * donor priority "gpu": overloaded GPUs in descending load, each giving away
    its experts in descending block count; donor priority "expert": all
    (overloaded GPU, expert) pairs in descending block count;
  * a donor first moves blocks to GPUs that already hold the expert, then to
    new replicas; it moves min(its excess over tau, the receiver's room below
    tau, its blocks of the expert) at a time;
  * a redundant replica is one whose blocks the expert's other holders can
    take without any of them rising above the current maximum load;
  * single-block refinement moves one block from a holder to another holder
    of the same expert while their loads differ by two or more, heaviest
    donor first;
  * reduction-aware pruning repeatedly takes the GPU with the largest
    penalised load L + lambda * (remote replicas of experts it owns) and
    removes its remote replica with the smallest allocation below lambda
    (blocks back to the owner), while that GPU has such a replica.
Ties are always broken toward the lower GPU index, then the lower expert.
"""
from __future__ import annotations

DONOR_ORDERS = ("gpu", "expert")
FANOUTS = ("one", "multi")


def owner_of(e: int, E: int, G: int) -> int:
    return e * G // E


def blocks_of(counts, beta: int):
    """Step 1: blocks per expert, ceil(c_e / beta)."""
    return [(int(c) + beta - 1) // beta for c in counts]


def loads(n, G):
    L = [0] * G
    for row in n:
        for g in range(G):
            L[g] += row[g]
    return L


class Plan:
    """n[e][g] = blocks of expert e on GPU g; holders[e] = GPUs holding e."""

    def __init__(self, b, G):
        E = len(b)
        self.G = G
        self.n = [[0] * G for _ in range(E)]
        self.holders = [set() for _ in range(E)]
        for e in range(E):
            o = owner_of(e, E, G)
            self.n[e][o] = b[e]
            self.holders[e].add(o)

    def copy(self):
        p = Plan.__new__(Plan)
        p.G = self.G
        p.n = [row[:] for row in self.n]
        p.holders = [set(h) for h in self.holders]
        return p

    def owner(self, e):
        return owner_of(e, len(self.n), self.G)

    def load(self):
        return loads(self.n, self.G)

    def replicas(self):
        """(gpu, expert) of every replica (a holder that is not the owner)."""
        return sorted((g, e) for e in range(len(self.n)) for g in self.holders[e]
                      if g != self.owner(e))

    def slots_used(self, g):
        return sum(1 for e in range(len(self.n)) if g in self.holders[e] and g != self.owner(e))


def greedy_search(q0: Plan, tau: int, budget: int, rounds: int, donor: str, fanout: str) -> Plan:
    """Step 3: one bounded greedy search from q0."""
    p = q0.copy()
    G, E = p.G, len(p.n)
    L = p.load()
    for _ in range(rounds):
        moved = False
        new_this_round = [0] * E
        if donor == "gpu":
            over = sorted((g for g in range(G) if L[g] > tau), key=lambda g: (-L[g], g))
            pairs = [(d, e) for d in over
                     for e in sorted((e for e in range(E) if p.n[e][d] > 0),
                                     key=lambda e: (-p.n[e][d], e))]
        else:
            pairs = sorted(((d, e) for d in range(G) if L[d] > tau
                            for e in range(E) if p.n[e][d] > 0),
                           key=lambda de: (-p.n[de[1]][de[0]], -L[de[0]], de[0], de[1]))
        for d, e in pairs:
            while L[d] > tau and p.n[e][d] > 0:
                held = [g for g in sorted(p.holders[e]) if g != d and L[g] < tau]
                if held:
                    r = min(held, key=lambda g: (L[g], g))
                else:
                    if fanout == "one" and new_this_round[e] >= 1:
                        break
                    free = [g for g in range(G) if g not in p.holders[e] and L[g] < tau
                            and p.slots_used(g) < budget]
                    if not free:
                        break
                    r = min(free, key=lambda g: (L[g], g))
                    p.holders[e].add(r)
                    new_this_round[e] += 1
                m = min(L[d] - tau, tau - L[r], p.n[e][d])
                p.n[e][d] -= m
                p.n[e][r] += m
                L[d] -= m
                L[r] += m
                moved = True
        if not moved:
            break
    return p


def drop_empty_replicas(p: Plan):
    for g, e in p.replicas():
        if p.n[e][g] == 0:
            p.holders[e].discard(g)


def prune_redundant(p: Plan):
    """Step 5a: a replica whose blocks the other holders of the expert can
    take without rising above the current maximum load is removed."""
    drop_empty_replicas(p)
    changed = True
    while changed:
        changed = False
        L = p.load()
        M = max(L)
        for g, e in p.replicas():
            v = p.n[e][g]
            others = sorted((h for h in p.holders[e] if h != g), key=lambda h: (L[h], h))
            room = sum(M - L[h] for h in others)
            if v <= room:
                for h in others:
                    m = min(v, M - L[h])
                    p.n[e][h] += m
                    L[h] += m
                    v -= m
                p.n[e][g] = 0
                p.holders[e].discard(g)
                changed = True
                break


def single_block_moves(p: Plan):
    """Step 5b: move one block at a time from a holder of an expert to another
    holder of it whose load is at least two lower, heaviest donor first."""
    E = len(p.n)
    while True:
        L = p.load()
        best = None
        for g1 in sorted(range(p.G), key=lambda g: (-L[g], g)):
            for e in range(E):
                if p.n[e][g1] == 0:
                    continue
                rec = [g2 for g2 in p.holders[e] if g2 != g1 and L[g1] - L[g2] >= 2]
                if rec:
                    best = (g1, e, min(rec, key=lambda g: (L[g], g)))
                    break
            if best:
                break
        if best is None:
            return
        g1, e, g2 = best
        p.n[e][g1] -= 1
        p.n[e][g2] += 1


def penalised_max(p: Plan, lam: float) -> float:
    """C_lambda: max over GPUs of load + lambda * remote replicas of experts it owns."""
    L = p.load()
    own = [0] * p.G
    for g, e in p.replicas():
        own[p.owner(e)] += 1
    return max(L[g] + lam * own[g] for g in range(p.G))


def reduction_prune(p: Plan, lam: float) -> Plan:
    """Step 6a: remove remote replicas with allocation below lambda from the
    GPU with the largest penalised load, blocks back to the owner, while that
    GPU has such a replica."""
    p = p.copy()
    while True:
        L = p.load()
        own = [0] * p.G
        for g, e in p.replicas():
            own[p.owner(e)] += 1
        sel = min(range(p.G), key=lambda g: (-(L[g] + lam * own[g]), g))
        cands = [(p.n[e][g], e, g) for g, e in p.replicas()
                 if p.owner(e) == sel and p.n[e][g] < lam]
        if not cands:
            return p
        v, e, g = min(cands)
        p.n[e][sel] += v
        p.n[e][g] = 0
        p.holders[e].discard(g)


def plan_replicas(counts, G: int, beta: int, budget: int, lam=None, rounds=None):
    """The replica plan for expert row counts `counts` on G GPUs.

    Returns a dict: blocks [E]; n [E][G] blocks of each expert per GPU;
    replicas, the sorted (gpu, expert) pairs that are not owners; load [G];
    tau; the winning search (donor, fanout) or "q0"; row ranges
    rows[e][g] = (lo, hi) of expert e's rows (offsets inside its group) that
    GPU g computes."""
    E = len(counts)
    b = blocks_of(counts, beta)
    tau = (sum(b) + G - 1) // G
    s = budget if rounds is None else rounds
    q0 = Plan(b, G)
    cands = []
    for i, (dn, fo) in enumerate((d, f) for d in DONOR_ORDERS for f in FANOUTS):
        c = greedy_search(q0, tau, budget, s + 2, dn, fo)
        drop_empty_replicas(c)
        cands.append((max(c.load()), len(c.replicas()), i, c, (dn, fo)))
    _, _, _, best, which = min(cands, key=lambda t: (t[0], t[1], t[2]))
    best = best.copy()
    prune_redundant(best)
    single_block_moves(best)
    drop_empty_replicas(best)
    if lam is not None:
        pruned = reduction_prune(best, lam)
        if penalised_max(pruned, lam) < penalised_max(q0, lam):
            best = pruned
        else:
            best, which = q0.copy(), "q0"
    rows = assign_rows(counts, beta, best.n)
    return dict(blocks=b, n=best.n, replicas=best.replicas(), load=best.load(), tau=tau,
                search=which, rows=rows)


def assign_rows(counts, beta: int, n):
    """Step 7: expert e's rows, in routed order, cut into blocks of beta; GPUs
    holding e take their blocks in ascending GPU order."""
    rows = []
    for e, c in enumerate(counts):
        r, start = [], 0
        for g in range(len(n[e])):
            lo = min(start * beta, int(c))
            start += n[e][g]
            hi = min(start * beta, int(c))
            r.append((lo, hi))
        rows.append(r)
    return rows
