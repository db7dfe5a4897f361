"""Host-side logic of bench.py that needs no GPU: the committed DRAM-traffic
record is used only while its kernel-source digest matches, the digest
covers the kernel sources and compiler flags (and not the C-ABI validation
layer), the reduce-kernel name follows the phases of each launch table, and
the all-core CPU baseline computes what the single-threaded oracle does."""
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
    assert bench.profiled_step_traffic("layer_d1024_nd8") is None
    monkeypatch.undo()
    assert bench.profiled_traffic("k_reduce_rs_adam", "no_such_workload") is None
    assert bench.profiled_step_traffic("no_such_workload") is None


def test_step_traffic_record_is_current_and_consistent():
    """The whole-step record: current digest, read + write = total, the
    three kernels add up to it, and no more DRAM bytes than algorithmic."""
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["_per_step"]
    for workload, ent in rec.items():
        assert ent["source_digest"] == bench.kernel_source_digest(), workload
        assert ent["dram_bytes_per_step"] == (ent["dram_bytes_read_per_step"] +
                                              ent["dram_bytes_write_per_step"])
        parts = ent["per_kernel"].values()
        assert abs(sum(p["read"] for p in parts) - ent["dram_bytes_read_per_step"]) <= 3
        assert abs(sum(p["write"] for p in parts) - ent["dram_bytes_write_per_step"]) <= 3
        assert 0.5 < ent["dram_bytes_per_step"] / ent["algorithmic_bytes_per_step"] <= 1.0
        got = bench.profiled_step_traffic(workload)
        assert got["dram_bytes"] == ent["dram_bytes_per_step"]


def test_digest_covers_the_kernel_sources_and_flags(tmp_path, monkeypatch):
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
    from optimizer_state_gb300 import build
    moved = [f if not f.startswith("-I") else "-I/elsewhere/include" for f in build.NVCC_FLAGS]
    monkeypatch.setattr(build, "NVCC_FLAGS", moved)
    assert bench.kernel_source_digest() == base       # where the repository sits does not count
    monkeypatch.setattr(build, "NVCC_FLAGS", build.NVCC_FLAGS + ["-DSOMETHING"])
    assert bench.kernel_source_digest() != base


def test_reduce_kernel_name_follows_the_phases():
    from optimizer_state_gb300 import build
    build.build()
    assert bench.reduce_kernel_name(z3.Layout([3072 * 1024, 1024], 8)) == "k_reduce_aligned"
    assert bench.reduce_kernel_name(z3.Layout([100003, 7, 4099], 3)) == "k_reduce_shifted"
    assert bench.reduce_kernel_name(z3.Layout([262147], 8)) == "k_reduce_aligned"
    # 40 aligned parameters fill the first launch table; in the second, the
    # 7-element parameter's chunks are misaligned (S = 328 keeps the first
    # table aligned), so that table's launch is the shifted kernel
    assert bench.reduce_kernel_name(z3.Layout([64] * 40 + [7, 56], 8)).startswith("mixed")
    assert bench.reduce_kernel_name(z3.Layout([64] * 41, 8)) == "k_reduce_aligned"


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


def test_all_core_oracle_split_is_bit_identical(orc):
    """The all-core CPU baseline runs the unchanged oracle on contiguous
    pieces of the layer, each its own one-parameter layer, one per thread.
    Re-laid into the layer's full index space, every piece's master, m, v
    and bf16 parameters after two layer steps (and after the single-kernel
    calls the baseline also times) equal the oracle's run on the whole
    layer, bit for bit."""
    import numpy as np
    from optimizer_state_gb300 import inputs as I
    w = I.Workload("split", ((1000,), (77,), (4099,), (5,), (0,), (13,)), n_ranks=4,
                   param_std=0.02, grad_std=1e-3)
    sample = bench.oracle_sample(w, w.psi, seed=3)
    sw, full, grads = sample
    O = orc.layout(sw.numel, sw.n_ranks)
    sh, ma, m, v = orc.partition(O, full)
    scale = 1.0 / sw.n_ranks
    for cores in (3, 7):
        pieces = bench.split_sample(orc, sample, cores)
        assert [p.a for p in pieces][0] == 0 and pieces[-1].b == sw.psi
        assert all(p.b == q.a for p, q in zip(pieces, pieces[1:]))
    pieces = bench.split_sample(orc, sample, 3)
    for t in (1, 2):
        orc.step_layer(O, sh, grads, sw.grad_stride, scale, ma, m, v, bench.HP, t)
        bench.run_pieces(orc, pieces, "step_layer", 1, t)
    gs = orc.reduce_scatter(O, grads, sw.grad_stride, scale)
    orc.reduce_scatter(O, grads, sw.grad_stride, scale, out=gs, accumulate=True)
    orc.adam(ma, m, v, gs, sh, bench.HP["lr"], bench.HP["beta1"], bench.HP["beta2"],
             bench.HP["eps"], bench.HP["weight_decay"], 3)
    for k in ("reduce_scatter", "reduce_scatter_accumulate", "adam"):
        bench.run_pieces(orc, pieces, k, 1, 3)
    for name, whole in (("master", ma), ("m", m), ("v", v)):
        got = np.concatenate([orc.allgather_f32(p.O, getattr(p, name)) for p in pieces])
        assert np.array_equal(got.view(np.uint32), orc.allgather_f32(O, whole).view(np.uint32)), \
            name
    got = np.concatenate([orc.allgather(p.O, p.shards) for p in pieces])
    assert np.array_equal(got, orc.allgather(O, sh))
    got = np.concatenate([orc.allgather_f32(p.O, p.gs) for p in pieces])
    assert np.array_equal(got.view(np.uint32), orc.allgather_f32(O, gs).view(np.uint32))


def test_cpu_kernel_bytes_match_the_library_accounting():
    from optimizer_state_gb300 import build
    build.build()
    st = z3.Layout([3072 * 1024, 1024, 1024], 8).stats()
    psi = st["psi"]
    assert bench.cpu_bytes_per_elem("allgather", 8) * psi == st["hbm_allgather"]
    assert bench.cpu_bytes_per_elem("reduce_scatter", 8) * psi == st["hbm_reduce_scatter"]
    assert bench.cpu_bytes_per_elem("reduce_scatter_accumulate", 8) * psi == \
        st["hbm_reduce_scatter_accumulate"]
    assert bench.cpu_bytes_per_elem("adam", 8) * psi == st["hbm_adam"]
    assert bench.cpu_bytes_per_elem("step_layer", 8) * psi == st["hbm_step_layer"]
