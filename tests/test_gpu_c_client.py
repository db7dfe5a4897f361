"""The C ABI from plain C: tests/c/abi_client.c allocates its own device
memory with cudaMalloc, drives z3_partition and three layer steps through
include/z3.h -- z3_step_layer from device gradients, the host-memory pipeline
z3_host_step_* from page-locked host gradients, or z3_model_step over one unit
per parameter with a resident unit and prefetch -- and its outputs must equal
the oracle's bit for bit.  No Python binding or torch tensor is involved on
that path."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.fail("CUDA is not available: the GPU tests need a GPU")
    from optimizer_state_gb300 import build
    lib = build.build()
    cuda = os.path.dirname(os.path.dirname(shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"))
    out = str(tmp_path_factory.mktemp("c") / "abi_client")
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", f"-I{ROOT}/include", f"-I{cuda}/include",
                    os.path.join(ROOT, "tests", "c", "abi_client.c"), "-o", out, f"-L{libdir}",
                    "-lz3", f"-L{cuda}/lib64", "-lcudart", f"-Wl,-rpath,{libdir}"], check=True)
    return out


def _inputs(orc, numel, n_ranks, steps, tmp_path):
    rng = np.random.default_rng(3)
    L = orc.layout(numel, n_ranks)
    stride = -(-L.psi // 8) * 8
    full = (rng.standard_normal(L.psi) * 0.02).astype(np.float32)
    grads = []
    for _ in range(steps):
        g = np.zeros((n_ranks, stride), np.uint16)
        g[:, :L.psi] = orc.bf16_from_f32(rng.standard_normal((n_ranks, L.psi)).astype(np.float32))
        grads.append(g)
    inp = tmp_path / "in.bin"
    with open(inp, "wb") as f:
        f.write(full.tobytes())
        for g in grads:
            f.write(g.tobytes())
    return L, stride, full, grads, inp


@pytest.mark.parametrize("mode", ["--layer", "--host"])
@pytest.mark.parametrize("numel,n_ranks", [([35, 13, 12], 4), ([100003, 7, 1, 0, 4099], 3),
                                           ([4096, 1024, 16], 8)])
def test_c_client_matches_oracle(client, orc, tmp_path, numel, n_ranks, mode):
    steps = 3
    L, stride, full, grads, inp = _inputs(orc, numel, n_ranks, steps, tmp_path)
    outp = tmp_path / "out.bin"
    r = subprocess.run([client, mode, str(inp), str(outp), str(n_ranks), str(steps),
                        str(len(numel)), *map(str, numel)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    raw = open(outp, "rb").read()
    T = L.psi_padded
    sh = np.frombuffer(raw, np.uint16, T, 0)
    ma, m, v = (np.frombuffer(raw, np.float32, T, 2 * T + 4 * T * i) for i in range(3))
    gathered = np.frombuffer(raw, np.uint16, L.psi, 2 * T + 12 * T)
    o_sh, o_ma, o_m, o_v = orc.partition(L, full)
    for t, g in enumerate(grads, start=1):
        _, fb, _ = orc.step_layer(L, o_sh, g.reshape(-1), stride, 1.0 / n_ranks, o_ma, o_m, o_v,
                                  HP, t)
    assert np.array_equal(sh, o_sh)
    for got, want in ((ma, o_ma), (m, o_m), (v, o_v)):
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.array_equal(gathered, fb)


@pytest.mark.parametrize("numel,n_ranks", [([1024, 100003, 7, 0, 4099], 3),
                                           ([77, 4096, 65536, 16], 8)])
def test_c_client_model_step_matches_oracle(client, orc, tmp_path, numel, n_ranks):
    """z3_model_step from C: one unit per parameter, unit 0 resident, prefetch
    depth 1; every unit's state equals the oracle's layer step on that
    parameter alone, and the resident copy equals the oracle's gather."""
    steps = 3
    L, stride, full, grads, inp = _inputs(orc, numel, n_ranks, steps, tmp_path)
    outp = tmp_path / "out.bin"
    r = subprocess.run([client, "--model", str(inp), str(outp), str(n_ranks), str(steps),
                        str(len(numel)), *map(str, numel)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    raw = open(outp, "rb").read()
    pos, F = 0, 0
    first_shards = None
    for p, n in enumerate(numel):
        O = orc.layout([n], n_ranks)
        T = O.psi_padded
        us = -(-n // 8) * 8
        o_sh, o_ma, o_m, o_v = orc.partition(O, full[F:F + n])
        for t, g in enumerate(grads, start=1):
            gu = np.zeros((n_ranks, us), np.uint16)
            gu[:, :n] = g[:, F:F + n]
            orc.step_layer(O, o_sh, gu.reshape(-1), us, 1.0 / n_ranks, o_ma, o_m, o_v, HP, t)
        sh = np.frombuffer(raw, np.uint16, T, pos)
        pos += 2 * T
        got = [np.frombuffer(raw, np.float32, T, pos + 4 * T * i) for i in range(3)]
        pos += 12 * T
        assert np.array_equal(sh, o_sh), p
        for a, b in zip(got, (o_ma, o_m, o_v)):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), p
        if p == 0:
            first_shards = (O, o_sh)
        F += n
    if numel[0] > 0:
        res = np.frombuffer(raw, np.uint16, numel[0], pos)
        assert np.array_equal(res, orc.allgather(*first_shards))
        pos += 2 * numel[0]
    assert pos == len(raw)
