"""The N > 1 host logic of bench.py on CPU ranks (gloo, world size 2): the
timed region's maximum over ranks and the weak-scaling job value."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r "took" 10 * (r + 1) ms; the job time is the slowest rank's
        t = bench.max_over_ranks(10.0 * (rank + 1))
        v = bench.job_value(units_per_rank=1000, steps=5, seconds=t / 1e3, world=world)
        q.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, t, v in res:
        assert t == 20.0                       # max over ranks, seen by every rank
        assert v == pytest.approx(2 * 1000 * 5 / 0.020)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value(10, 2, 0.5, 1) == 40.0
