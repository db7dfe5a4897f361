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


def test_reference_arm_line_matches_the_gpu_config(capsys):
    """Rank 0 prints one reference line whose config carries the GPU line's
    workload keys with the same values (plus the sample size), so the two
    arms name the same workload."""
    import argparse
    import json

    import bench
    import oracle
    from optimizer_state_gb300 import inputs as I
    args = argparse.Namespace(steps=2, warmup=1, reference_seconds=0.6)
    bench.run_reference(args, world=1, rank=0)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    w = I.LAYER_D1024
    O = oracle.layout(w.numel, w.n_ranks)
    want = bench.layer_config("layer_d1024_nd8", w, O.psi, O.S)
    assert {k: line["config"][k] for k in want} == want
    assert 0 < line["config"]["sample_psi"] <= w.psi
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["cpu_baseline"]["cores"] >= 1 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
