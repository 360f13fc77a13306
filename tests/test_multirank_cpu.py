"""The multi-replica host logic of bench.py on CPU: two gloo ranks.

Under torchrun every rank runs an independent replica (its own inputs, no
data-path collective); the job's rate divides the rounds of all ranks by the
slowest rank's time.  Here two processes with different elapsed times check
the max-over-ranks reduction, the whole-job rates and the per-rank seeds.
"""
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 1.0 + rank  # rank 1 is the slower one
        e2e = 2.0 + 0.5 * rank
        value, e2e_value, el, e2 = bench.job_throughput(dist, elapsed, e2e, steps=100, e2e_steps=10, world=world)
        out[rank] = (value, e2e_value, el, e2, bench.replica_seeds(rank, 3))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_whole_job_rate():
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        value, e2e_value, el, e2, seeds = res[rank]
        assert el == pytest.approx(2.0) and e2 == pytest.approx(2.5)   # slowest rank on every rank
        assert value == pytest.approx(100 * world / 2.0)
        assert e2e_value == pytest.approx(10 * world / 2.5)
    assert res[0][4] != res[1][4]                                      # replicas build different inputs
    assert res[1][4] == [100000, 100001, 100002]


def test_single_rank_needs_no_process_group():
    import bench
    value, e2e_value, el, e2 = bench.job_throughput(None, 0.5, 1.0, steps=10, e2e_steps=4, world=1)
    assert (value, e2e_value, el, e2) == (20.0, 4.0, 0.5, 1.0)
