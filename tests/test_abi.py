"""C-ABI library on the CPU: it builds for sm_103a, loads, exports every
symbol include/z3.h declares, and its host logic (layout, accounting,
argument validation) agrees with the oracle.  No kernel is launched here:
every device call below fails validation before reaching CUDA.  The tests
that pass made-up device addresses are marked no_device and run in a child
process that sees no CUDA device (tests/conftest.py), so a validation that
let a call through would end in a launch error, never in a memory access."""
import ctypes
import os
import re

import pytest

from optimizer_state_gb300 import build as z3build
from optimizer_state_gb300 import z3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    z3build.build()
    return z3.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "z3.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(z3_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 13
    assert sorted(z3.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert lib.z3_status_string(0) == b"Z3_OK"
    assert lib.z3_status_string(2) == b"Z3_ERR_ALIGNMENT"


CASES = [([35, 13, 12], 4), ([12584960 // 4] * 4, 8), ([0, 5, 0, 7], 3), ([1], 64),
         ([262147], 2), ([262147], 64), ([3, 0], 1), ([50257 * 1024], 16)]


@pytest.mark.parametrize("numel,n_ranks", CASES)
def test_layout_matches_oracle(lib, orc, numel, n_ranks):
    L = z3.Layout(numel, n_ranks)
    O = orc.layout(numel, n_ranks)
    assert (L.S, L.psi, L.psi_padded) == (O.S, O.psi, O.psi_padded)
    assert L.shard_numel == list(O.shard_numel)
    assert L.shard_off == list(O.shard_off)
    assert L.full_off == list(O.full_off)
    assert L.numel == list(O.numel)
    st = L.stats()
    acc = orc.accounting(O)
    assert st["state_bytes_per_rank"] == acc["state_bytes_per_rank"]
    assert st["state_bytes_per_rank_fp32_grad"] == acc["state_bytes_per_rank_fp32_grad"]
    assert st["step_volume_bytes"] == acc["step_volume_bytes"]
    assert st["dp_allreduce_bytes"] == acc["dp_volume_bytes"]
    N = n_ranks
    assert st["hbm_step_layer"] == (2 * N + 34) * L.psi
    assert st["hbm_reduce_scatter_adam"] == (2 * N + 26) * L.psi


def test_layout_errors(lib):
    with pytest.raises(z3.Z3Error) as e:
        z3.Layout([5], 0)
    assert e.value.status == z3.Z3_ERR_INVALID_ARG and "n_ranks" in str(e.value)
    with pytest.raises(z3.Z3Error) as e:
        z3.Layout([5, -1], 4)
    assert e.value.status == z3.Z3_ERR_INVALID_ARG
    with pytest.raises(z3.Z3Error) as e:
        z3.Layout([2 ** 62, 2 ** 62], 1)
    assert e.value.status == z3.Z3_ERR_OVERFLOW
    out = ctypes.c_void_p()
    assert lib.z3_layout_create(None, 1, 1, ctypes.byref(out)) == z3.Z3_ERR_INVALID_ARG
    arr = (ctypes.c_int64 * 1)(5)
    assert lib.z3_layout_create(ctypes.cast(arr, ctypes.c_void_p), 0, 1,
                                ctypes.byref(out)) == z3.Z3_ERR_INVALID_ARG
    assert lib.z3_layout_info(None, None, None, None, None, None) == z3.Z3_ERR_INVALID_ARG
    lib.z3_layout_destroy(None)  # no-op


@pytest.mark.no_device
def test_device_call_validation_without_gpu(lib):
    """Host-side checks return before any CUDA call (fake device addresses)."""
    L = z3.Layout([35, 13, 12], 4)
    A = 1 << 32                       # an aligned fake address
    far = A + (1 << 28)
    st = lambda s: (s, z3.last_error())  # noqa: E731
    # NULL / misaligned / overlapping buffers
    s, msg = st(lib.z3_allgather(L.handle, None, A, None))
    assert s == z3.Z3_ERR_INVALID_ARG and "shards" in msg
    s, msg = st(lib.z3_allgather(L.handle, A + 2, far, None))
    assert s == z3.Z3_ERR_ALIGNMENT
    s, msg = st(lib.z3_allgather(L.handle, A, A + 16, None))
    assert s == z3.Z3_ERR_INVALID_ARG and "overlaps" in msg
    # grad_stride rules
    s, msg = st(lib.z3_reduce_scatter(L.handle, A, 59, far, 0.25, 0, None))
    assert s == z3.Z3_ERR_INVALID_ARG and "grad_stride" in msg
    s, msg = st(lib.z3_reduce_scatter(L.handle, A, 61, far, 0.25, 0, None))
    assert s == z3.Z3_ERR_ALIGNMENT
    s, msg = st(lib.z3_reduce_scatter(L.handle, A, 64, far, float("nan"), 0, None))
    assert s == z3.Z3_ERR_INVALID_ARG
    # Adam: step and hyperparameters
    hp = z3.AdamHP(1e-3, 0.9, 0.999, 1e-8, 0.0)
    bufs = [A + i * (1 << 24) for i in range(5)]
    s, msg = st(lib.z3_adam_shard_step(L.handle, *bufs, ctypes.byref(hp), 0, None))
    assert s == z3.Z3_ERR_INVALID_ARG and "step" in msg
    bad = z3.AdamHP(float("inf"), 0.9, 0.999, 1e-8, 0.0)
    s, msg = st(lib.z3_adam_shard_step(L.handle, *bufs, ctypes.byref(bad), 1, None))
    assert s == z3.Z3_ERR_INVALID_ARG
    s, msg = st(lib.z3_adam_shard_step(L.handle, *bufs, None, 1, None))
    assert s == z3.Z3_ERR_INVALID_ARG
    s, msg = st(lib.z3_step_layer(None, *bufs[:2], A, 64, 0.25, *bufs[2:], None,
                                  ctypes.byref(hp), 1, None))
    assert s == z3.Z3_ERR_INVALID_ARG
    s, msg = st(lib.z3_step_layer(L.handle, bufs[0], bufs[1], A + (1 << 27), 64, 0.25,
                                  *bufs[2:], bufs[3] + 64, ctypes.byref(hp), 1, None))
    assert s == z3.Z3_ERR_INVALID_ARG and "grad_shards" in msg and "overlaps" in msg
    s, msg = st(lib.z3_step_layer(L.handle, bufs[0], bufs[1], A + (1 << 27), 64, 0.25,
                                  *bufs[2:], far + 8, ctypes.byref(hp), 1, None))
    assert s == z3.Z3_ERR_ALIGNMENT and "grad_shards" in msg
    s, msg = st(lib.z3_reduce_scatter_adam(L.handle, A, 64, 0.25, None, A, far, far + 4096,
                                           far + 8192, ctypes.byref(hp), 1, None))
    assert s == z3.Z3_ERR_INVALID_ARG and "overlaps" in msg


@pytest.mark.no_device
def test_zero_size_layer_is_a_noop(lib):
    L = z3.Layout([0, 0], 4)
    assert (L.S, L.psi, L.psi_padded) == (0, 0, 0)
    assert lib.z3_allgather(L.handle, None, None, None) == z3.Z3_OK
    assert lib.z3_partition(L.handle, None, None, None, None, None, None) == z3.Z3_OK


def test_product_never_reaches_the_oracle():
    """The package and its CUDA sources import, include or link nothing from
    oracle/; the oracle imports nothing from the package."""
    pkg = os.path.join(ROOT, "optimizer_state_gb300")
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"].*oracle)", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h")):
                assert not pat.search(open(os.path.join(dirpath, f)).read()), f
    back = re.compile(r"^\s*(import|from)\s+optimizer_state_gb300", re.M)
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            assert not back.search(open(os.path.join(ROOT, "oracle", f)).read()), f


@pytest.mark.no_device
def test_stage_and_reshard_entry_validation(lib):
    """z3_allreduce, z3_scatter and z3_reshard reject bad arguments on the
    host (fake device addresses; nothing reaches CUDA)."""
    L = z3.Layout([35, 13, 12], 4)
    A = 1 << 32
    far = A + (1 << 28)
    assert lib.z3_allreduce(L.handle, A, 59, far, 0.25, None) == z3.Z3_ERR_INVALID_ARG
    assert lib.z3_allreduce(L.handle, A, 61, far, 0.25, None) == z3.Z3_ERR_ALIGNMENT
    assert lib.z3_allreduce(L.handle, A, 64, A + 64, 0.25, None) == z3.Z3_ERR_INVALID_ARG
    assert lib.z3_allreduce(None, A, 64, far, 0.25, None) == z3.Z3_ERR_INVALID_ARG
    assert lib.z3_scatter(L.handle, A, A, None) == z3.Z3_ERR_INVALID_ARG
    assert lib.z3_scatter(L.handle, A + 4, far, None) == z3.Z3_ERR_ALIGNMENT
    L2 = z3.Layout([35, 13, 12], 8)
    L3 = z3.Layout([35, 13, 11], 8)
    assert lib.z3_reshard(L.handle, L2.handle, 3, A, far, None) == z3.Z3_ERR_INVALID_ARG
    assert lib.z3_reshard(L.handle, L3.handle, 4, A, far, None) == z3.Z3_ERR_INVALID_ARG
    assert "different parameters" in z3.last_error()
    assert lib.z3_reshard(L.handle, L2.handle, 4, A, A + 16, None) == z3.Z3_ERR_INVALID_ARG
    assert lib.z3_reshard(L.handle, None, 4, A, far, None) == z3.Z3_ERR_INVALID_ARG


@pytest.mark.no_device
def test_model_step_validation_without_gpu(lib):
    """z3_model_step rejects bad unit lists, buffer counts, streams and
    overlapping or misaligned buffers (resident copies included) before it
    creates an event or launches anything (fake device addresses)."""
    L = z3.Layout([35, 13, 12], 4)
    A = 1 << 32
    hp = z3.AdamHP(1e-3, 0.9, 0.999, 1e-8, 0.0)
    T = L.psi_padded

    def unit(base, resident=None, layout=L):
        # shards, master, m, v, grads laid out 1 MiB apart from base
        a = [base + i * (1 << 20) for i in range(5)]
        return z3.Unit(layout.handle.value if layout else None, a[0], a[1], a[2], a[3], a[4],
                       64, 0.25, resident)

    def call(units, fulls, n_full=None, gstream=None):
        arr = (z3.Unit * len(units))(*units) if units else None
        f = (ctypes.c_void_p * len(fulls))(*fulls)
        return lib.z3_model_step(arr, len(units), f, len(fulls) if n_full is None else n_full,
                                 ctypes.byref(hp), 1, None, gstream), z3.last_error()
    full = A + (64 << 20)
    s, msg = call([], [full])
    assert s == z3.Z3_ERR_INVALID_ARG and "no units" in msg
    s, msg = call([unit(A)], [full], n_full=0)
    assert s == z3.Z3_ERR_INVALID_ARG
    s, msg = call([unit(A)], [full] * 9)
    assert s == z3.Z3_ERR_INVALID_ARG
    s, msg = call([unit(A)], [full, full + (1 << 20)])           # prefetch without a stream
    assert s == z3.Z3_ERR_INVALID_ARG and "gather stream" in msg
    s, msg = call([unit(A, layout=None)], [full])
    assert s == z3.Z3_ERR_INVALID_ARG and "layout" in msg
    s, msg = call([unit(A)], [A + 16])                           # full overlaps shards
    assert s == z3.Z3_ERR_INVALID_ARG and "overlaps" in msg
    s, msg = call([unit(A, resident=A + (1 << 20))], [full])     # resident overlaps master
    assert s == z3.Z3_ERR_INVALID_ARG and "overlaps" in msg
    s, msg = call([unit(A, resident=A + (32 << 20) + 2)], [full])
    assert s == z3.Z3_ERR_ALIGNMENT and "resident" in msg
    s, msg = call([unit(A), unit(A + (8 << 20), resident=full + 16)], [full])
    assert s == z3.Z3_ERR_INVALID_ARG and "overlaps" in msg      # resident inside full
    s, msg = call([unit(A), unit(A + (2 << 20))], [full])        # two units share state
    assert s == z3.Z3_ERR_INVALID_ARG and "another unit" in msg
    s, msg = call([unit(A), unit(A + (8 << 20), resident=A + (4 << 20))], [full])
    assert s == z3.Z3_ERR_INVALID_ARG and "another unit" in msg  # resident over another's grads
    assert T == 64


@pytest.mark.no_device
def test_host_step_validation_without_gpu(lib):
    """z3_host_step_create rejects bad layouts, streams and staging buffers
    before it creates any CUDA object (fake addresses and stream handles)."""
    L = z3.Layout([35, 13, 12], 4)
    A = 1 << 32
    far = A + (1 << 28)
    up, down = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000)
    h = ctypes.c_void_p()

    def create(layout, s0, s1, stride, u, d, out=True):
        st = lib.z3_host_step_create(layout, s0, s1, stride, u, d,
                                     ctypes.byref(h) if out else None)
        return st, z3.last_error()
    s, msg = create(L.handle, A, far, 64, up, down, out=False)
    assert s == z3.Z3_ERR_INVALID_ARG and "out" in msg
    s, msg = create(None, A, far, 64, up, down)
    assert s == z3.Z3_ERR_INVALID_ARG and "layout" in msg
    s, msg = create(L.handle, A, far, 64, None, down)
    assert s == z3.Z3_ERR_INVALID_ARG and "stream" in msg
    s, msg = create(L.handle, A, far, 64, up, up)
    assert s == z3.Z3_ERR_INVALID_ARG and "stream" in msg
    s, msg = create(L.handle, A, far, 59, up, down)
    assert s == z3.Z3_ERR_INVALID_ARG and "grad_stride" in msg
    s, msg = create(L.handle, A, far, 68, up, down)
    assert s == z3.Z3_ERR_ALIGNMENT
    s, msg = create(L.handle, A, None, 64, up, down)
    assert s == z3.Z3_ERR_INVALID_ARG and "staging1" in msg
    s, msg = create(L.handle, A + 8, far, 64, up, down)
    assert s == z3.Z3_ERR_ALIGNMENT and "staging0" in msg
    s, msg = create(L.handle, A, A + 64, 64, up, down)       # 4 ranks x 64 x 2 B = 512 B
    assert s == z3.Z3_ERR_INVALID_ARG and "overlaps" in msg
    assert h.value is None
    assert lib.z3_host_step_run(None, A, A, A, 0.25, A, A, A, None, 1, None, None) == \
        z3.Z3_ERR_INVALID_ARG
    lib.z3_host_step_destroy(None)                           # a no-op


@pytest.mark.no_device
def test_model_step_checks_many_units_quickly(lib):
    """The cross-unit overlap check scales to thousands of units: 4000
    disjoint units plus one whose master overlaps the first unit's shards
    are rejected (naming both units) well within a second, before any CUDA
    call."""
    import time
    L = z3.Layout([35, 13, 12], 4)
    hp = z3.AdamHP(1e-3, 0.9, 0.999, 1e-8, 0.0)
    base = 1 << 36
    n = 4000

    def unit(a, master=None):
        return z3.Unit(L.handle.value, a, master if master is not None else a + 1024, a + 2048,
                       a + 3072, a + 4096, 64, 0.25, None)
    units = [unit(base + i * 8192) for i in range(n)] + [unit(base + n * 8192, master=base + 64)]
    arr = (z3.Unit * len(units))(*units)
    full = (ctypes.c_void_p * 1)(base - (1 << 20))
    t0 = time.perf_counter()
    s = lib.z3_model_step(arr, len(units), full, 1, ctypes.byref(hp), 1, None, None)
    dt = time.perf_counter() - t0
    msg = z3.last_error()
    assert s == z3.Z3_ERR_INVALID_ARG and "unit 0" in msg and f"({n})" in msg, msg
    assert dt < 1.0, dt


@pytest.mark.no_device
def test_adam_hyperparameter_rules(lib):
    """Hyperparameters that would turn the update into inf/NaN are rejected
    on the host: beta1 or beta2 outside [0, 1), eps <= 0 (a pad position
    would compute 0/0), negative lr or weight decay, and values whose binary32
    constants overflow or whose eps rounds to 0.  Accepted ones pass the
    checks and reach the launch, which fails here because the process sees
    no device."""
    L = z3.Layout([35, 13, 12], 4)
    A = 1 << 32
    bufs = [A + i * (1 << 24) for i in range(5)]
    good = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    bad = [dict(beta1=1.0), dict(beta2=1.0), dict(beta1=-0.1), dict(beta2=1.5), dict(eps=0.0),
           dict(eps=-1e-8), dict(lr=-1e-3), dict(weight_decay=-0.1), dict(eps=1e-50),
           dict(lr=1e300), dict(lr=1e200, weight_decay=1e200)]
    for change in bad:
        hp = z3.AdamHP(**{**good, **change})
        s = lib.z3_adam_shard_step(L.handle, *bufs, ctypes.byref(hp), 1, None)
        assert s == z3.Z3_ERR_INVALID_ARG, (change, z3.last_error())
        s = lib.z3_reduce_scatter_adam(L.handle, A, 64, 0.25, None, *bufs[1:4], bufs[4] + 4096,
                                       ctypes.byref(hp), 1, None)
        assert s == z3.Z3_ERR_INVALID_ARG, (change, z3.last_error())
    for change in ({}, dict(beta1=0.0, beta2=0.0), dict(weight_decay=0.1), dict(lr=0.0)):
        hp = z3.AdamHP(**{**good, **change})
        s = lib.z3_adam_shard_step(L.handle, *bufs, ctypes.byref(hp), 1, None)
        assert s == z3.Z3_ERR_CUDA, (change, z3.last_error())


_OOM_CHILD = r"""
import ctypes, resource, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
from optimizer_state_gb300 import z3
lib = z3.load()
n = 20_000_000                       # 160 MB of element counts; the layout needs 4x that
numel = np.ones(n, dtype=np.int64)
with open("/proc/self/statm") as f:
    vm = int(f.read().split()[0]) * resource.getpagesize()
resource.setrlimit(resource.RLIMIT_AS, (vm + (96 << 20), resource.RLIM_INFINITY))
out = ctypes.c_void_p()
st = lib.z3_layout_create(numel.ctypes.data_as(ctypes.c_void_p), n, 8, ctypes.byref(out))
msg = z3.last_error()
print(st, out.value, msg)
sys.exit(0 if st == z3.Z3_ERR_HOST_MEMORY and out.value is None and "host memory" in msg
         else 1)
"""


@pytest.mark.no_device
def test_host_out_of_memory_status(lib):
    """A host allocation that fails inside the library returns
    Z3_ERR_HOST_MEMORY (not Z3_ERR_INVALID_ARG) and leaves no layout: a
    child process caps its address space just above its current size and
    asks for a layout of 20 million parameters."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-c", _OOM_CHILD, ROOT], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert lib.z3_status_string(z3.Z3_ERR_HOST_MEMORY) == b"Z3_ERR_HOST_MEMORY"
