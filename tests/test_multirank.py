"""The N > 1 host path of bench.py with gloo on the CPU (world size 2): the
timed region ends when the slowest rank ends, and the reported value counts
the work of every rank; the CPU reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.5, 40.0][rank]
    ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
    val = bench.aggregate_gbs(world, 629248000, 100, ms)
    dist.barrier()
    out[rank] = (ms, val)
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 40.0
    expect = 2 * 629248000 * 100 / 0.040 / 1e9
    assert out[0][1] == pytest.approx(expect) and out[1][1] == pytest.approx(expect)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import argparse

    import bench
    args = argparse.Namespace(steps=3, warmup=3, reference_seconds=1.0)
    bench.run_reference(args, world=2, rank=1)
    assert capsys.readouterr().out == ""
