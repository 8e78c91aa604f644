"""The multi-rank host logic on CPU ranks (gloo, world size 2): the slowest
rank's time sets the benchmark's whole-job throughput, the reference arm runs
on rank 0 only, and an expert-tensor-sharded layer (each rank holding a slice
of every expert's FFN features) is recovered by one all-reduce of the ranks'
partial outputs."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 100.0 + 50.0 * rank                    # rank 1 is the slow one
    slowest = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
    value = bench.throughput(world, 128, 10, slowest)
    ref = bench.bench_reference(None, rank, world, 0) if rank != 0 else "skipped"
    q.put((rank, slowest, value, ref))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, ref in got:
        assert slowest == 150.0
        assert value == pytest.approx(2 * 128 * 10 / 0.150)
    assert got[1][3] is None        # the reference arm does no work off rank 0


def test_single_rank_throughput():
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.throughput(1, 128, 500, 400.0) == pytest.approx(128 * 500 / 0.4)


def _shard_worker(rank, world, port, q):
    import numpy as np
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import moe_oracle as O
    g = torch.Generator().manual_seed(3)
    T, H, F, E, k = 24, 16, 32, 4, 2
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(E, H, F, generator=g) / 4).to(torch.bfloat16)
    W3 = (torch.randn(E, H, F, generator=g) / 4).to(torch.bfloat16)
    W2 = (torch.randn(E, F, H, generator=g) / 6).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g).numpy()
    s = np.array_split(np.arange(F), world)[rank]     # this rank's features
    part = O.forward_perm(x, logits, W1[:, :, s], W3[:, :, s], W2[:, s, :], k)["out"]
    t = torch.from_numpy(np.ascontiguousarray(part))
    dist.all_reduce(t)                                 # the one exchange step
    full = O.forward_perm(x, logits, W1, W3, W2, k)["out"]
    q.put((rank, float(np.abs(t.numpy() - full).max())))
    dist.barrier()
    dist.destroy_process_group()


def test_feature_sharded_layer_needs_one_all_reduce():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, err in got:
        assert err <= 1e-12


def _runner_worker(rank, world, port, q):
    """The package's feature-sharded runner on CPU ranks: each rank slices the
    weights with shard_weights, computes its partial (the oracle stands in for
    the GPU's moe_forward_f32), and sharded_forward all-reduces and rounds."""
    import numpy as np
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import moe_oracle as O
    from routing_grouped_expert_gb300 import sharded
    g = torch.Generator().manual_seed(4)
    T, H, F, E, k = 20, 16, 256 * world, 4, 2
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(E, H, F, generator=g) / 4).to(torch.bfloat16)
    W3 = (torch.randn(E, H, F, generator=g) / 4).to(torch.bfloat16)
    W2 = (torch.randn(E, F, H, generator=g) / 16).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g)
    W1s, W3s, W2s = sharded.shard_weights(W1, W3, W2, world, rank)
    assert W1s.shape[2] == F // world and W2s.shape[1] == F // world

    def partial(x_, l_, a, b, c, k_):
        return torch.from_numpy(O.forward_perm(x_, l_.numpy(), a, b, c, k_)["out"]).float()
    out = sharded.sharded_forward(x, logits, W1s, W3s, W2s, k, partial=partial,
                                  cast=lambda t: t.to(torch.bfloat16))
    full = O.forward_perm(x, logits.numpy(), W1, W3, W2, k)["out"]
    err = np.abs(out.double().numpy() - full)
    q.put((rank, float((err / (2.0 ** -8 * np.abs(full) + 1e-6)).max())))
    dist.barrier()
    dist.destroy_process_group()


def test_feature_sharded_runner_on_two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_runner_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, ratio in got:
        assert ratio <= 1.0      # fp32 partials summed, rounded to bf16 once


def test_feature_slices_are_aligned_and_cover_f():
    from routing_grouped_expert_gb300 import sharded
    for F, world in ((2048, 8), (16384, 4), (10752, 2), (256, 2)):
        cuts = [sharded.feature_slice(F, world, r) for r in range(world)]
        assert cuts[0][0] == 0 and cuts[-1][1] == F
        assert all(a[1] == b[0] for a, b in zip(cuts, cuts[1:]))
        assert all((hi - lo) % 128 == 0 for lo, hi in cuts)
    with pytest.raises(ValueError):
        sharded.feature_slice(384, 2, 0)

