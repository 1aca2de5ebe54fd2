"""The N > 1 path of the benchmark on CPU: replicas, two gloo ranks.

Every rank transcribes its own batch (no collective on the data path); the
only collective is the max-over-ranks of the step time, and the whole-job
rate counts the audio of all ranks over the slowest rank's time.  Here the
ranks are CPU processes with the gloo backend.
"""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 180.0][rank]                       # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms)
    rate = bench.whole_job_rate(960.0, world, m)
    q.put((rank, m, rate))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_reduce_to_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, rate in res:
        assert m == 180.0
        assert rate == pytest.approx(960.0 * 2 / 0.180)


def test_single_process_needs_no_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(42.0) == 42.0
    assert bench.whole_job_rate(30.0, 1, 1000.0) == 30.0
