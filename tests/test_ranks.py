"""The multi-process path of bench.py on CPU: two gloo ranks, each with its own
timed region; the job's time is the slowest rank's and the rate counts every
replica's tokens (replicas, weak scaling: no collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank            # rank 1 is the slower one
    total = bench.slowest_rank_ms(local_ms, "cpu")
    rate = bench.job_throughput(tokens_per_step=64, steps=4, world=world, total_ms=total)
    out[rank] = (total, rate)
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_slowest_rank_and_job_rate(world):
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    slow = 10.0 + 5.0 * (world - 1)
    for r in range(world):
        total, rate = out[r]
        assert total == slow
        assert rate == pytest.approx(world * 64 * 4 / (slow / 1e3))


def test_single_process_is_identity():
    import bench
    assert bench.slowest_rank_ms(12.5, "cpu") == 12.5
    assert bench.job_throughput(1, 10, 1, 1000.0) == pytest.approx(10.0)
