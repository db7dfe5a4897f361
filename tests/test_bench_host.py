"""Host-side logic of bench.py that needs no GPU: the committed DRAM-traffic
record is used only while its kernel-source digest matches, the digest
covers the kernel sources (and not the C-ABI validation layer), and the
reduce-kernel name follows the layout's phases."""
import json
import os

import bench
from optimizer_state_gb300 import z3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_record_is_current_for_every_entry():
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    digest = bench.kernel_source_digest()
    for kernel, per in rec.items():
        if kernel.startswith("_"):
            continue
        for workload, ent in per.items():
            assert ent["source_digest"] == digest, (kernel, workload)
            assert ent["dram_bytes_per_launch"] == ent["dram_bytes_read"] + ent["dram_bytes_write"]
            assert 0.5 < ent["dram_bytes_per_launch"] / ent["algorithmic_bytes_per_launch"] < 1.2
            assert bench.profiled_traffic(kernel, workload) == ent["dram_bytes_per_launch"]


def test_traffic_is_withheld_when_the_kernels_change(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "0" * 16)
    assert bench.profiled_traffic("k_reduce_rs_adam", "layer_d1024_nd8") is None
    monkeypatch.undo()
    assert bench.profiled_traffic("k_reduce_rs_adam", "no_such_workload") is None


def test_digest_covers_the_kernel_sources_only(tmp_path, monkeypatch):
    csrc = os.path.join(ROOT, "optimizer_state_gb300", "csrc")
    base = bench.kernel_source_digest()
    real_open = open

    def fake_open(path, *a, **k):
        f = real_open(path, *a, **k)
        if str(path).endswith(name) and "b" in (a[0] if a else k.get("mode", "r")):
            data = f.read() + b"\n// changed\n"
            f.close()
            import io
            return io.BytesIO(data)
        return f
    for name, counted in (("z3_kernels.cu", True), ("z3_launch.h", True),
                          ("z3_internal.h", True), ("z3_layout.cpp", True),
                          ("z3_api.cpp", False)):
        monkeypatch.setattr("builtins.open", fake_open)
        changed = bench.kernel_source_digest()
        monkeypatch.undo()
        assert (changed != base) == counted, name
    assert os.path.exists(os.path.join(csrc, "z3_api.cpp"))


def test_reduce_kernel_name_follows_the_phases():
    from optimizer_state_gb300 import build
    build.build()
    assert bench.reduce_kernel_name(z3.Layout([3072 * 1024, 1024], 8)) == "k_reduce_aligned"
    assert bench.reduce_kernel_name(z3.Layout([100003, 7, 4099], 3)) == "k_reduce_shifted"
    assert bench.reduce_kernel_name(z3.Layout([262147], 8)) == "k_reduce_aligned"


def test_full_step_workload_names():
    import pytest
    assert bench.parse_full_step("full_step_nd16") == (0, 1, 0)
    assert bench.parse_full_step("full_step_nd16_prefetch") == (1, 1, 0)
    assert bench.parse_full_step("full_step_nd16_prefetch2_bucket4") == (2, 4, 0)
    assert bench.parse_full_step("full_step_nd16_bucket6_persist100000") == (0, 6, 100000)
    assert bench.parse_full_step("full_step_nd16_prefetch3_bucket2_persist5") == (3, 2, 5)
    for bad in ("full_step_nd8", "full_step_nd16_bucket0", "full_step_nd16_prefetch9",
                "full_step_nd16_persist", "full_step_nd16_bucket4_prefetch2"):
        with pytest.raises(SystemExit):
            bench.parse_full_step(bad)
