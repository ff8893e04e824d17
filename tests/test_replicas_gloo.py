"""The multi-GPU path of the benchmark is replicas only: every rank runs its
own copy of the workload and the job figure uses the slowest rank's time.
This checks that aggregation with two gloo ranks on the CPU."""

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
    per_rank = [2.0 + rank, 1.0 + 2 * rank]        # rank 1 is the slower replica
    ms, gbs = bench.aggregate_replicas(per_rank, 1e9, world, bench.torch_max_reducer("cpu"))
    dist.barrier()
    q.put((rank, ms, gbs))
    dist.destroy_process_group()


def test_two_replicas_report_slowest_rank_and_total_bytes():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, gbs in res:
        assert ms == [3.0, 3.0]                     # max over ranks, element-wise
        assert gbs == pytest.approx(2 * 1e9 / 3e-3 / 1e9)


def test_single_rank_needs_no_collective():
    import bench
    ms, gbs = bench.aggregate_replicas([4.0], 2e9, 1, None)
    assert ms == [4.0] and gbs == pytest.approx(500.0)
