"""FC1 with 256-row token blocks on CTA pairs (F a multiple of 256, fewer
than two blocks per expert on average), against the oracle, with per-expert
row counts chosen at every boundary of the pair's layout: a block of r rows
is split between the two SMs as two halves of ceil(r / 32) * 16 rows (one
MMA over both, N = 2 of them), so the counts cover rows below, at and above
multiples of 16, 32 and 64, blocks of a single row, experts split into two
and three blocks, and an expert with no rows.  FC2 (one SM per tile) waits
for the pairs' FC1 block by block; the same experts with F = 384 (no pairs)
check the single-SM path on the same layout."""
import numpy as np
import pytest
import torch

import routing_grouped_expert_gb300 as moe
from oracle import moe_oracle as O
from routing_grouped_expert_gb300 import inputs as I
from tests.helpers import assert_moe_close

pytestmark = pytest.mark.gpu

# rows per expert: > 80 on average, so the layer takes 256-row blocks
COUNTS = [1, 16, 17, 31, 32, 33, 47, 100, 255, 256, 257, 300, 513, 0]

SHAPES = {  # name: (H, F)
    "pair_fc1": (1024, 512),
    "pair_fc1_unpaired_fc2_tiles": (640, 512),   # H / 128 odd: FC2 one W2 tile per CTA
    "no_pairs": (1024, 384),
}


def routed(counts, seed):
    """sorted_src / offsets of a one-choice routing with the given counts:
    each expert's rows are a random subset of the tokens."""
    rng = np.random.default_rng(seed)
    T = int(sum(counts))
    perm = rng.permutation(T).astype(np.int32)
    offsets = np.zeros(len(counts) + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    return T, perm, offsets


@pytest.mark.parametrize("shape", list(SHAPES))
def test_pair_block_layout_matches_oracle(shape):
    H, F = SHAPES[shape]
    E = len(COUNTS)
    T, src, offsets = routed(COUNTS, seed=11)
    wl = I.small(f"pair_{shape}", T=T, H=H, F=F, E=E, k=1)
    d = I.make_inputs(wl, "cpu")
    ref = O.grouped_ffn(d["x"], src, offsets, d["W1"], d["W3"], d["W2"], 1)
    dev = {n: d[n].cuda() for n in ("x", "W1", "W3", "W2")}
    y = moe.moe_grouped_ffn(dev["x"], torch.from_numpy(src).cuda(),
                            torch.from_numpy(offsets).cuda(), dev["W1"], dev["W3"], dev["W2"], 1)
    assert_moe_close(y, ref, f"{shape} y_sorted")
    # and again: the same bits (fixed tile order, fixed K order per element)
    y2 = moe.moe_grouped_ffn(dev["x"], torch.from_numpy(src).cuda(),
                             torch.from_numpy(offsets).cuda(), dev["W1"], dev["W3"], dev["W2"], 1)
    assert torch.equal(y, y2)


@pytest.mark.parametrize("shape", ["pair_fc1", "pair_fc1_unpaired_fc2_tiles"])
def test_pair_forward_matches_oracle(shape):
    """The fused forward (FC2 overlapping the pairs' FC1 per token block) with
    skewed routing: uneven blocks, some experts nearly empty."""
    H, F = SHAPES[shape]
    wl = I.small(f"pairfwd_{shape}", T=1500, H=H, F=F, E=8, k=2, skew_alpha=1.5)
    d = I.make_inputs(wl, "cpu")
    ref = O.forward_perm(d["x"], d["logits"].numpy(), d["W1"], d["W3"], d["W2"], wl.k)
    dev = {n: t.cuda() for n, t in d.items()}
    ws = moe.Workspace()
    out = moe.moe_forward(dev["x"], dev["logits"], dev["W1"], dev["W3"], dev["W2"], wl.k, ws=ws)
    assert moe.moe_get_device_status(ws) == 0
    assert_moe_close(out, ref["out"], f"{shape} out")
