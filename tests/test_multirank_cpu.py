"""The N > 1 path of bench.py on the CPU: two gloo ranks (no GPU).

The scan shards into independent (batch, head) problems, so N GPUs run N replicas with no
data-path collective; the only cross-rank steps are the barrier around the timed region and
the max over ranks of the elapsed time, which sets the whole-job rate.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    ws, r, local = bench.dist_setup()
    dist.init_process_group("gloo", rank=r, world_size=ws)
    dist.barrier()
    # each rank "measured" a different elapsed time; every rank must see the slowest
    elapsed = [0.5, 2.0, 1.25][r]
    slowest = bench.max_over_ranks(elapsed, "cpu", ws)
    rate = bench.whole_job_rate(1000.0, ws, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, ws, local, slowest, rate))


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_agree_on_the_slowest_time_and_the_job_rate(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(world))
    slowest = max([0.5, 2.0, 1.25][:world])
    for r, (rank, ws, local, s, rate) in enumerate(got):
        assert (rank, ws, local) == (r, world, r)
        assert s == slowest
        assert rate == pytest.approx(1000.0 * world / slowest)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, "cpu", 1) == 3.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
