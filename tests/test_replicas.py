"""Several GPUs run independent replicas of the decode pass (no data-path
collective); the job's step time is the slowest rank's and its throughput
counts every rank's bytes.  This host logic runs here as two gloo ranks on the
CPU; the GPU timing itself is covered by bench.py on a GB300."""
from __future__ import annotations

import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + 2.0 * rank, world)  # rank 1 is the slow one
        out.put((rank, ms, bench.replicas_gbs(6e9, ms, world)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_both():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = 29400 + os.getpid() % 500
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(2))
    for rank, ms, gbs in got:
        assert ms == pytest.approx(3.0)                 # both ranks see the max
        assert gbs == pytest.approx(2 * 6e9 / 3e-3 / 1e9)  # both ranks' bytes over the max time


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.replicas_gbs(6e9, 2.0, 1) == pytest.approx(3000.0)
