"""The bench's replica aggregation across ranks, on CPU with gloo (world size 2)."""
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
