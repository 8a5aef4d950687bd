"""The bench's multi-rank host logic on two CPU processes (gloo): every rank
runs its own replica, the ranks meet at barriers around the timed region, the
job's time is the slowest rank's and its throughput sums the replicas'.  No
GPU is involved; the GPU launch path is the same code with the nccl backend."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        my_ms = 2.0 + 3.0 * rank  # rank 1 is the slow replica
        slowest = bench.max_over_ranks(my_ms, world)
        value = bench.job_throughput(10.0, slowest, world)
        bench.barrier(world)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_slowest_time_and_summed_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for _, slowest, value in res:
        assert slowest == pytest.approx(5.0)
        # two replicas of 10 units each in the slowest rank's 5 ms
        assert value == pytest.approx(2 * 10.0 / 5e-3)


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(7.5, 1) == 7.5
    bench.barrier(1)
    assert bench.job_throughput(3.0, 1.5, 1) == pytest.approx(2000.0)
