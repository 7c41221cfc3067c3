"""The benchmark's multi-rank bookkeeping on CPU (gloo, world size 2): every
rank runs its own independent instance of the workload (weak scaling, no
data-path collective); the step time is the slowest rank's and the whole-job
throughput counts every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 135.5][rank]
    ms = bench.max_over_ranks(local_ms, dist, "cpu")
    value = bench.whole_job_tflops(world, 1.0e12, ms)
    results[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step_and_sum_the_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    for rank in range(world):
        ms, value = res[rank]
        assert ms == 135.5                        # max over ranks, seen by every rank
        assert value == pytest.approx(2 * 1.0e12 / 0.1355 / 1e12)


def test_single_rank_without_process_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(1, 2.0e12, 1000.0) == pytest.approx(2.0)
