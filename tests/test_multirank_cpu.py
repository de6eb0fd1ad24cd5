"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, slowest-rank timing and
whole-job throughput (each rank runs its own replica of the workload)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    slowest = bench.max_over_ranks(mine)
    value = bench.weak_scaling_value(100.0, world, slowest)
    q.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_slowest_time_and_total_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, value in got:
        assert slowest == 15.0
        assert value == pytest.approx(100.0 * 2 / 15.0)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.weak_scaling_value(10.0, 1, 2.0) == 5.0
