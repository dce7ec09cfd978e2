"""Multi-GPU host logic of bench.py on CPU: replicas share nothing but the
timing reduction, so a world-size-2 gloo group checks that every rank ends
with the slowest rank's time and that the whole-job rate counts every
replica's work over that time. The reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [1.0 + rank, 10.0 - 3 * rank]  # rank 0: [1, 10], rank 1: [2, 7]
    got = bench.max_over_ranks(mine, dist, "cpu")
    out[rank] = got + [bench.whole_job_rate(100.0, world, got[0])]
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_max_time_and_rate():
    world = 2
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        assert out[rank][:2] == [2.0, 10.0]
        assert out[rank][2] == pytest.approx(100.0 * 2 / 2.0)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0


def test_reference_arm_runs_on_rank_zero_only():
    import argparse

    import bench
    args = argparse.Namespace(steps=1, warmup=0)
    assert bench.run_reference(args, rank=1, world=2) is None  # no work, no output
