"""bench.py's N > 1 aggregation on two gloo ranks (CPU): the job's time is
the slowest rank's, and throughput counts every rank's tokens."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [40.0, 55.0][rank]
    max_ms, value = bench.aggregate(ms, 8192 * 10, world)
    q.put((rank, max_ms, value))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, max_ms, value in out:
        assert max_ms == 55.0
        assert abs(value - 2 * 8192 * 10 / 0.055) < 1e-6 * value


def test_single_rank_aggregation():
    max_ms, value = __import__("bench").aggregate(20.0, 1000, 1)
    assert max_ms == 20.0 and abs(value - 50000.0) < 1e-9
