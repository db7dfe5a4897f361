"""Python face of the plain-C CPU oracle (``z3_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` are the only
callers.  The CUDA library never imports this module, and this module never
imports the CUDA library; the two meet only in the tests, on inputs drawn by
``optimizer_state_gb300.inputs``.

Arrays are numpy: bf16 values travel as ``uint16`` bit patterns, fp32 as
``float32``.  Each wrapper cites the passage its C function follows; the
citations are repeated in ``z3_oracle.c``.
"""
from __future__ import annotations

import ctypes
import fcntl
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "z3_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libz3oracle.so")
_lock = threading.Lock()
_lib = None

_I64P = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc: -O2, no FMA contraction, no fast-math
    (serialised across processes by a lock file)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    with open(os.path.join(_BUILD_DIR, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            return _build_locked(force)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(force: bool) -> str:
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c17", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    vp = ctypes.c_void_p
    i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    f64 = ctypes.c_double
    lib.or_layout.argtypes = [vp, i32, i32, vp, vp, vp, _I64P, _I64P, _I64P]
    lib.or_layout.restype = ctypes.c_int
    lib.or_bf16_from_f32.argtypes = [f32]
    lib.or_bf16_from_f32.restype = ctypes.c_uint16
    lib.or_f32_from_bf16.argtypes = [ctypes.c_uint16]
    lib.or_f32_from_bf16.restype = f32
    lib.or_bf16_from_f32_array.argtypes = [vp, vp, i64]
    lib.or_partition.argtypes = [vp, vp, vp, vp, i32, i32, i64, vp, vp, vp, vp, vp]
    lib.or_allgather.argtypes = [vp, vp, vp, vp, i32, i64, vp, vp]
    lib.or_allgather_f32.argtypes = [vp, vp, vp, vp, i32, i64, vp, vp]
    lib.or_reduce_scatter.argtypes = [vp, vp, vp, vp, i32, i32, i64, vp, i64, vp, f32, i32]
    lib.or_allreduce.argtypes = [i64, i32, vp, i64, vp, f32]
    lib.or_adam_constants.argtypes = [f64, f64, f64, f64, f64, i64, vp]
    lib.or_adam.argtypes = [i64, vp, vp, vp, vp, vp, f64, f64, f64, f64, f64, i64]
    lib.or_step_layer.argtypes = ([vp, vp, vp, vp, i32, i32, i64, vp, vp, vp, vp, i64, f32,
                                   vp, vp, vp, vp, vp, f64, f64, f64, f64, f64, i64])
    lib.or_accounting.argtypes = [i64, i64, i32, _I64P, _I64P, _I64P, _I64P,
                                  ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double)]
    return lib


def build_variant(source: str, out_dir: str) -> str:
    """Compile another copy of the oracle source (used by the mutation tests,
    which plant mistakes in a copy to show that the pins catch them)."""
    src = os.path.join(out_dir, "z3_oracle_variant.c")
    with open(src, "w") as f:
        f.write(source)
    lib = os.path.join(out_dir, "libz3oracle_variant.so")
    subprocess.run(["gcc", "-std=c17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", lib, src, "-lm"], check=True)
    return lib


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(a: np.ndarray, dtype, n: int, name: str):
    if a.dtype != dtype or a.size < n or not a.flags["C_CONTIGUOUS"]:
        raise ValueError(f"{name}: need C-contiguous {np.dtype(dtype)} with >= {n} elements, "
                         f"got {a.dtype} size {a.size}")


@dataclass(frozen=True)
class Layout:
    """Per-parameter flatten/pad/slice layout (page "The ZeRO-3 Diagram Most
    People Remember Is Wrong", s.2 "The Actual Parameter Partition")."""
    numel: np.ndarray        # n_p
    shard_numel: np.ndarray  # s_p = ceil(n_p / N)
    shard_off: np.ndarray    # o_p
    full_off: np.ndarray     # F_p
    n_ranks: int             # N
    S: int                   # rank stride
    psi: int                 # sum n_p
    psi_padded: int          # N * S

    @property
    def n_params(self) -> int:
        return int(self.numel.size)


def layout(numel, n_ranks: int) -> Layout:
    lib = _load()
    nm = np.ascontiguousarray(np.asarray(numel, dtype=np.int64))
    P = nm.size
    s = np.zeros(P, np.int64)
    o = np.zeros(P, np.int64)
    F = np.zeros(P, np.int64)
    S, psi, psip = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    rc = lib.or_layout(_ptr(nm), P, n_ranks, _ptr(s), _ptr(o), _ptr(F),
                       ctypes.byref(S), ctypes.byref(psi), ctypes.byref(psip))
    if rc != 0:
        raise ValueError("invalid layout arguments")
    return Layout(nm, s, o, F, int(n_ranks), S.value, psi.value, psip.value)


def _lay_args(L: Layout):
    return (_ptr(L.numel), _ptr(L.shard_numel), _ptr(L.shard_off), _ptr(L.full_off),
            L.n_params)


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even, from the IEEE-754 layout."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().or_bf16_from_f32_array(_ptr(x), _ptr(out), x.size)
    return out


def f32_from_bf16(h: np.ndarray) -> np.ndarray:
    """bf16 bits -> fp32 (exact): the 16 bits become the top half."""
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def partition(L: Layout, full: np.ndarray):
    """full fp32 [psi] -> (shards bf16, master, m, v), each [N*S]
    (page "The ZeRO-3 Diagram ...", s.2 steps 1-4)."""
    _check(full, np.float32, L.psi, "full")
    n = L.psi_padded
    sh = np.empty(n, np.uint16)
    ma = np.empty(n, np.float32)
    m = np.empty(n, np.float32)
    v = np.empty(n, np.float32)
    _load().or_partition(*_lay_args(L), L.n_ranks, L.S, _ptr(full), _ptr(sh), _ptr(ma),
                         _ptr(m), _ptr(v))
    return sh, ma, m, v


def allgather(L: Layout, shards: np.ndarray) -> np.ndarray:
    """bf16 [N*S] -> unpadded full bf16 [psi] (page "The ZeRO-3 Diagram ...",
    s.3 "The Collectives You Should Expect")."""
    _check(shards, np.uint16, L.psi_padded, "shards")
    out = np.empty(L.psi, np.uint16)
    _load().or_allgather(*_lay_args(L), L.S, _ptr(shards), _ptr(out))
    return out


def allgather_f32(L: Layout, shards: np.ndarray) -> np.ndarray:
    _check(shards, np.float32, L.psi_padded, "shards")
    out = np.empty(L.psi, np.float32)
    _load().or_allgather_f32(*_lay_args(L), L.S, _ptr(shards), _ptr(out))
    return out


def reduce_scatter(L: Layout, grads: np.ndarray, grad_stride: int, scale: float,
                   out: np.ndarray | None = None, accumulate: bool = False) -> np.ndarray:
    """bf16 grads [N][grad_stride] -> fp32 owned slices [N*S]
    (page "ZeRO Stages: ...", "Stage 2 also partitions gradients")."""
    _check(grads, np.uint16, (L.n_ranks - 1) * grad_stride + L.psi, "grads")
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs the running sums in `out`")
        out = np.empty(L.psi_padded, np.float32)
    _check(out, np.float32, L.psi_padded, "out")
    _load().or_reduce_scatter(*_lay_args(L), L.n_ranks, L.S, _ptr(grads), grad_stride,
                              _ptr(out), float(scale), 1 if accumulate else 0)
    return out


def allreduce(L: Layout, grads: np.ndarray, grad_stride: int, scale: float) -> np.ndarray:
    _check(grads, np.uint16, (L.n_ranks - 1) * grad_stride + L.psi, "grads")
    out = np.empty(L.psi, np.float32)
    _load().or_allreduce(L.psi, L.n_ranks, _ptr(grads), grad_stride, _ptr(out), float(scale))
    return out


ADAM_CONSTANT_NAMES = ("b1", "c1", "b2", "c2", "rb1", "rb2", "lr", "eps", "lwd")


def adam_constants(lr, beta1, beta2, eps, weight_decay, step) -> dict:
    """The binary32 constants of one Adam step (each rounded once from
    the real-valued hyperparameters)."""
    out = np.zeros(9, np.float32)
    _load().or_adam_constants(lr, beta1, beta2, eps, weight_decay, step, _ptr(out))
    return dict(zip(ADAM_CONSTANT_NAMES, out.tolist()))


def adam(master, m, v, grad, param_bf16, lr, beta1, beta2, eps, weight_decay, step):
    """In-place Adam over flat fp32 arrays (Kingma & Ba, Algorithm 1)."""
    n = master.size
    for a, nm in ((master, "master"), (m, "m"), (v, "v"), (grad, "grad")):
        _check(a, np.float32, n, nm)
    _check(param_bf16, np.uint16, n, "param_bf16")
    if step < 1:
        raise ValueError("step must be >= 1")
    _load().or_adam(n, _ptr(master), _ptr(m), _ptr(v), _ptr(grad), _ptr(param_bf16),
                    lr, beta1, beta2, eps, weight_decay, step)


def step_layer(L: Layout, shards, grads, grad_stride, scale, master, m, v, hp, step,
               grad_acc=None):
    """AG (forward), AG (backward), RS, Adam; updates shards/master/m/v in place.
    Returns (full_fwd, full_bwd, grad_shards)."""
    n = L.psi_padded
    _check(shards, np.uint16, n, "shards")
    for a, nm in ((master, "master"), (m, "m"), (v, "v")):
        _check(a, np.float32, n, nm)
    _check(grads, np.uint16, (L.n_ranks - 1) * grad_stride + L.psi, "grads")
    if grad_acc is not None:
        _check(grad_acc, np.float32, n, "grad_acc")
    ff = np.empty(L.psi, np.uint16)
    fb = np.empty(L.psi, np.uint16)
    gs = np.empty(n, np.float32)
    _load().or_step_layer(*_lay_args(L), L.n_ranks, L.S, _ptr(shards), _ptr(ff), _ptr(fb),
                          _ptr(grads), grad_stride, float(scale), _ptr(grad_acc), _ptr(gs),
                          _ptr(master), _ptr(m), _ptr(v), hp["lr"], hp["beta1"], hp["beta2"],
                          hp["eps"], hp["weight_decay"], step)
    return ff, fb, gs


def accounting(L: Layout) -> dict:
    """Byte accounting (page "ZeRO Stage 3: Parameter Partitioning", eq.
    M_Stage3 and the communication list; page "ZeRO Stages: ...", table)."""
    a, b, c, d = (ctypes.c_int64() for _ in range(4))
    e, f = ctypes.c_double(), ctypes.c_double()
    _load().or_accounting(L.S, L.psi, L.n_ranks, ctypes.byref(a), ctypes.byref(b),
                          ctypes.byref(c), ctypes.byref(d), ctypes.byref(e), ctypes.byref(f))
    return dict(state_bytes_per_rank=a.value, state_bytes_per_rank_fp32_grad=b.value,
                step_volume_bytes=c.value, dp_volume_bytes=d.value,
                per_rank_ring_elems_stage3=e.value, per_rank_ring_elems_dp=f.value)
