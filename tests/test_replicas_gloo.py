"""The N > 1 bench path on CPU: two gloo ranks stand in for two GPUs.

The stage has no exchange step, so N GPUs run N independent replicas; the
only multi-rank logic is the timing aggregation: the maximum elapsed time
over ranks and the job's time per call derived from it.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    elapsed_ms = [120.0, 150.0][rank]  # rank 1 is the slowest replica
    slowest = bench.max_over_ranks(elapsed_ms)
    out[rank] = (slowest, bench.job_value_us(slowest, steps=30, world=world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for rank in (0, 1):
        slowest, value = res[rank]
        assert slowest == 150.0
        # 2 replicas x 30 steps = 60 calls in 150 ms -> 2500 us per call
        assert value == pytest.approx(2500.0)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value_us(4.5, steps=3, world=1) == pytest.approx(1500.0)
