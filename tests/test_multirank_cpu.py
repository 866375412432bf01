"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Units (batch, head) are independent, so each rank runs its own batch with no
collective on the data path; ranks meet only for the barriers around the timed
region and for the maximum of their timings.  This checks that logic with two
gloo ranks on 127.0.0.1.
"""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        worst = bench.max_over_ranks(local_ms, world)
        tokens_per_rank = 1000
        value = bench.aggregate_throughput(tokens_per_rank, worst, world)
        results[rank] = (worst, value)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_max_timing_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(100)
            assert p.exitcode == 0
        res = dict(results)
    # Both ranks see the slowest rank's time; the whole-job value counts both ranks' tokens.
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == pytest.approx(2 * 1000 / 15e-3 / 1e6)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_throughput(2000, 2.0, 1) == pytest.approx(2000 / 2e-3 / 1e6)
