"""The N > 1 host logic of the benchmark on CPU: two gloo ranks.  Each rank
runs an independent problem (no data-path collective); the only collectives
are the barrier and the max-over-ranks timing reduction, and the whole-job
value counts the units of every rank over the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    t = [0.25, 0.40][rank]
    bench.barrier(world)
    tmax = bench.max_over_ranks(t, world)
    v = bench.weak_scaling_value(1e12, world, tmax)
    # every rank's independent problem is computed without communication
    x = torch.full((4,), float(rank))
    local = (x * 2).sum().item()
    q.put((rank, tmax, v, local))
    dist.destroy_process_group()


def test_two_gloo_ranks_timing_reduction():
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
    assert [r[1] for r in res] == [0.40, 0.40]
    assert res[0][2] == pytest.approx(2 * 1e12 / 0.40 / 1e12)
    assert [r[3] for r in res] == [0.0, 8.0]


def test_single_rank_value():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.weak_scaling_value(2e12, 1, 0.5) == pytest.approx(4.0)
