"""Multi-rank host logic on CPU with gloo (world size 2): the bench's replica aggregation, and
expert-parallel shards of the oracle's layer summed across ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [12.5, 20.0][rank]
    mx = bench.reduce_max(ms, "cpu")
    q.put((rank, mx, bench.throughput(64 * 10, world, mx)))
    dist.destroy_process_group()


def test_reduce_max_and_throughput_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [20.0, 20.0]
    assert res[0][2] == pytest.approx(2 * 640 / 0.020)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.5, "cpu") == 3.5
    assert bench.throughput(64, 1, 2.0) == pytest.approx(32000.0)


def _shard_worker(rank, world, port, q):
    # each rank holds experts rank, rank + world, ... and computes its shard of the oracle's layer; the
    # shards' outputs summed across the ranks (the combine of an expert-parallel layer) give the layer
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    import test_oracle_ep as pep
    x, logits, w13, w2, s13, s2 = pep._tiny_layer(seed=21, T=8, E=6)
    part = pep._layer(x, logits, 2, w13, w2, s13, s2, list(range(rank, 6, world)))["out_f64"]
    t = torch.from_numpy(part.copy())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    if rank == 0:
        full = pep._layer(x, logits, 2, w13, w2, s13, s2)["out_f64"]
        q.put(float(abs(t.numpy() - full).max() / abs(full).max()))
    dist.destroy_process_group()


def test_expert_shards_all_reduce_to_the_layer():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    err = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert err <= 1e-12
