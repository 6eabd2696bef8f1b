"""CPU test of the benchmark's multi-rank aggregation (replicas on N GPUs): two gloo ranks on the host.

Each rank reports its own time; the job's time is the slowest rank's, and the whole-job rate counts every
rank's bytes over it.  No GPU is involved (world size 2, backend gloo, 127.0.0.1 rendezvous).
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
    q.put((rank, t, bench.whole_job_gbs(1000, 10, world, t)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    world, port = 2, _free_port()
    times = [12.5, 20.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, gbs in got:
        assert t == 20.0                                     # every rank sees the slowest
        assert gbs == pytest.approx(2 * 1000 * 10 / 0.020 / 1e9)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1, None) == 3.0
    assert bench.whole_job_gbs(2_000_000, 5, 1, 1.0) == pytest.approx(10.0)
