"""The N>1 host path of bench.py on CPU with the gloo backend: every rank runs
an independent replica, only the timing is reduced (max over ranks) and the
whole-job throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    value, ms = bench.aggregate(1000.0, times[rank], w)
    bench.barrier(w)
    q.put((rank, value, ms))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_weak_scaling_aggregate_over_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [10.0 + 5.0 * r for r in range(world)]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max(times)
    for _, value, ms in res:
        assert ms == pytest.approx(slowest)
        assert value == pytest.approx(world * 1000.0 / (slowest * 1e-3))
