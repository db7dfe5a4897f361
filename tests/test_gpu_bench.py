"""bench.py end to end on the GPU, short: one JSON line with the contract's
keys, the timed steps replayed as one CUDA graph of the library's launches,
the fused kernel's roofline, the e2e leg through the C ABI with its copies
declared, and clock samples."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is not available: the GPU tests need a GPU")
    r = subprocess.run([sys.executable, "bench.py", "--steps", "4", "--warmup", "3",
                        "--kernel-steps", "3", "--e2e-steps", "3", "--no-cpu-baseline",
                        "--cold-bytes", "1"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["steps"] == 4 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["gpu_launches"] == 3 * 4
    assert line["config"]["step_bytes"] == 50 * line["config"]["psi"]
    assert "CUDA graph" in line["config"]["launch"]
    roof = line["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-3)
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == 2 * 8 * line["config"]["psi"]
    assert e2e["d2h_bytes_per_step"] == 2 * 8 * line["config"]["S"]
    assert line["clocks"]["samples"] >= 1
