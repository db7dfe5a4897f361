"""Thin ctypes binding of the C ABI in ``include/z3.h``.

Argument marshalling only: every step of the path runs in the CUDA library
``_build/libz3.so``.  Functions keep the C names; device buffers may be
passed as CUDA tensors (their data pointer is used; dtype and size are
checked here, the library re-checks pointers, alignment and overlap) or as
raw integer device addresses.  ``stream`` defaults to torch's current CUDA
stream.  There is no CPU fallback: if the library is missing, loading fails
with an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

(Z3_OK, Z3_ERR_INVALID_ARG, Z3_ERR_ALIGNMENT, Z3_ERR_OVERFLOW, Z3_ERR_CUDA,
 Z3_ERR_HOST_MEMORY) = range(6)

# Every symbol include/z3.h declares.
EXPORTS = ("z3_layout_create", "z3_layout_destroy", "z3_layout_info", "z3_layout_params",
           "z3_stats", "z3_partition", "z3_allgather", "z3_reduce_scatter",
           "z3_adam_shard_step", "z3_reduce_scatter_adam", "z3_step_layer",
           "z3_allreduce", "z3_scatter", "z3_reshard", "z3_model_step",
           "z3_host_step_create", "z3_host_step_run", "z3_host_step_destroy",
           "z3_step_layer_noalloc", "z3_status_string", "z3_last_error")


class Z3Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


class AdamHP(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double)]


class Unit(ctypes.Structure):
    """struct z3_unit."""
    _fields_ = [("layout", ctypes.c_void_p), ("shards", ctypes.c_void_p),
                ("master", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("grads", ctypes.c_void_p), ("grad_stride", ctypes.c_int64),
                ("scale", ctypes.c_float), ("resident", ctypes.c_void_p),
                ("hp", ctypes.POINTER(AdamHP))]


class Traffic(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "psi", "ag_payload_bytes", "rs_payload_bytes", "step_volume_bytes",
        "dp_allreduce_bytes", "hbm_allgather", "hbm_reduce_scatter",
        "hbm_reduce_scatter_accumulate", "hbm_adam", "hbm_reduce_scatter_adam",
        "hbm_step_layer", "state_bytes_per_rank", "state_bytes_per_rank_fp32_grad")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load the CUDA library (built by ``optimizer_state_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is not built; run "
                               "`python -m optimizer_state_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(path)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        f32, st = ctypes.c_float, ctypes.c_int
        hp = ctypes.POINTER(AdamHP)
        sig = {
            "z3_layout_create": (st, [vp, i32, i32, ctypes.POINTER(vp)]),
            "z3_layout_destroy": (None, [vp]),
            "z3_layout_info": (st, [vp, vp, vp, vp, vp, vp]),
            "z3_layout_params": (st, [vp, vp, vp, vp, vp]),
            "z3_stats": (st, [vp, ctypes.POINTER(Traffic)]),
            "z3_partition": (st, [vp, vp, vp, vp, vp, vp, vp]),
            "z3_allgather": (st, [vp, vp, vp, vp]),
            "z3_reduce_scatter": (st, [vp, vp, i64, vp, f32, i32, vp]),
            "z3_adam_shard_step": (st, [vp, vp, vp, vp, vp, vp, hp, i64, vp]),
            "z3_reduce_scatter_adam": (st, [vp, vp, i64, f32, vp, vp, vp, vp, vp, hp, i64, vp]),
            "z3_step_layer": (st, [vp, vp, vp, vp, i64, f32, vp, vp, vp, vp, hp, i64, vp]),
            "z3_allreduce": (st, [vp, vp, i64, vp, f32, vp]),
            "z3_scatter": (st, [vp, vp, vp, vp]),
            "z3_reshard": (st, [vp, vp, i32, vp, vp, vp]),
            "z3_model_step": (st, [ctypes.POINTER(Unit), i32, ctypes.POINTER(vp), i32, hp, i64,
                                   vp, vp]),
            "z3_host_step_create": (st, [vp, vp, vp, i64, vp, vp, ctypes.POINTER(vp)]),
            "z3_host_step_run": (st, [vp, vp, vp, vp, f32, vp, vp, vp, hp, i64, vp, vp]),
            "z3_host_step_destroy": (None, [vp]),
            "z3_step_layer_noalloc": (st, [vp, vp, vp, i64, f32, vp, vp, vp, hp, i64, vp]),
            "z3_status_string": (ctypes.c_char_p, [st]),
            "z3_last_error": (ctypes.c_size_t, [ctypes.c_char_p, ctypes.c_size_t]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _status_name(status: int) -> str:
    try:
        return load().z3_status_string(status).decode()
    except Exception:  # noqa: BLE001 - only used while formatting an error
        return f"status {status}"


def last_error() -> str:
    lib = load()
    buf = ctypes.create_string_buffer(1024)
    lib.z3_last_error(buf, len(buf))
    return buf.value.decode(errors="replace")


def _check(status: int):
    if status != Z3_OK:
        raise Z3Error(status, last_error())


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t, dtypes, numel: int, name: str):
    """Device address of a tensor (or a raw int address).  A tensor must live
    on the current device: the library launches there, and every kernel
    treats its buffers as that device's own memory."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    import torch
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name}: on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name}: needs >= {numel} elements, has {t.numel()}")
    return t.data_ptr()


def _dtypes():
    import torch
    return (torch.bfloat16, torch.int16, torch.uint16), (torch.float32,)


class Layout:
    """Owns a ``z3_layout`` handle (z3_layout_create / z3_layout_destroy)."""

    def __init__(self, numel, n_ranks: int):
        lib = load()
        numel = [int(n) for n in numel]
        arr = (ctypes.c_int64 * len(numel))(*numel)
        h = ctypes.c_void_p()
        _check(lib.z3_layout_create(ctypes.cast(arr, ctypes.c_void_p), len(numel), n_ranks,
                                    ctypes.byref(h)))
        self._h = h
        self._lib = lib
        P, N = ctypes.c_int32(), ctypes.c_int32()
        S, psi, psip = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib.z3_layout_info(h, ctypes.byref(P), ctypes.byref(N), ctypes.byref(S),
                                  ctypes.byref(psi), ctypes.byref(psip)))
        self.n_params, self.n_ranks = P.value, N.value
        self.S, self.psi, self.psi_padded = S.value, psi.value, psip.value
        arrs = [(ctypes.c_int64 * self.n_params)() for _ in range(4)]
        _check(lib.z3_layout_params(h, *[ctypes.cast(a, ctypes.c_void_p) for a in arrs]))
        self.numel, self.shard_numel, self.shard_off, self.full_off = (list(a) for a in arrs)

    @property
    def handle(self):
        return self._h

    def stats(self) -> dict:
        t = Traffic()
        _check(self._lib.z3_stats(self._h, ctypes.byref(t)))
        return t.as_dict()

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.z3_layout_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass


def _hp(hp) -> AdamHP:
    if isinstance(hp, AdamHP):
        return hp
    return AdamHP(float(hp["lr"]), float(hp["beta1"]), float(hp["beta2"]), float(hp["eps"]),
                  float(hp.get("weight_decay", 0.0)))


def z3_partition(layout: Layout, full, shards, master, m, v, stream=None):
    b16, f32 = _dtypes()
    T = layout.psi_padded
    _check(load().z3_partition(layout.handle, _dev(full, f32, layout.psi, "full"),
                               _dev(shards, b16, T, "shards"), _dev(master, f32, T, "master"),
                               _dev(m, f32, T, "m"), _dev(v, f32, T, "v"), _stream(stream)))


def z3_allgather(layout: Layout, shards, full, stream=None):
    b16, _ = _dtypes()
    _check(load().z3_allgather(layout.handle, _dev(shards, b16, layout.psi_padded, "shards"),
                               _dev(full, b16, layout.psi, "full"), _stream(stream)))


def z3_reduce_scatter(layout: Layout, grads, grad_stride: int, grad_shards, scale: float,
                      accumulate: bool = False, stream=None):
    b16, f32 = _dtypes()
    _check(load().z3_reduce_scatter(
        layout.handle, _dev(grads, b16, layout.n_ranks * grad_stride, "grads"), grad_stride,
        _dev(grad_shards, f32, layout.psi_padded, "grad_shards"), scale, 1 if accumulate else 0,
        _stream(stream)))


def z3_adam_shard_step(layout: Layout, master, m, v, grad_shards, shards, hp, step: int,
                       stream=None):
    b16, f32 = _dtypes()
    T = layout.psi_padded
    h = _hp(hp)
    _check(load().z3_adam_shard_step(
        layout.handle, _dev(master, f32, T, "master"), _dev(m, f32, T, "m"),
        _dev(v, f32, T, "v"), _dev(grad_shards, f32, T, "grad_shards"),
        _dev(shards, b16, T, "shards"), ctypes.byref(h), step, _stream(stream)))


def z3_reduce_scatter_adam(layout: Layout, grads, grad_stride: int, scale: float, grad_acc,
                           master, m, v, shards, hp, step: int, stream=None):
    b16, f32 = _dtypes()
    T = layout.psi_padded
    h = _hp(hp)
    _check(load().z3_reduce_scatter_adam(
        layout.handle, _dev(grads, b16, layout.n_ranks * grad_stride, "grads"), grad_stride,
        scale, _dev(grad_acc, f32, T, "grad_acc"), _dev(master, f32, T, "master"),
        _dev(m, f32, T, "m"), _dev(v, f32, T, "v"), _dev(shards, b16, T, "shards"),
        ctypes.byref(h), step, _stream(stream)))


def z3_step_layer(layout: Layout, shards, full, grads, grad_stride: int, scale: float, master,
                  m, v, hp, step: int, stream=None, grad_shards=None):
    """grad_shards: None (the C call's grad_shards_or_NULL = NULL) or an fp32
    [N*S] tensor that receives the reduced gradient slices."""
    b16, f32 = _dtypes()
    T = layout.psi_padded
    h = _hp(hp)
    _check(load().z3_step_layer(
        layout.handle, _dev(shards, b16, T, "shards"), _dev(full, b16, layout.psi, "full"),
        _dev(grads, b16, layout.n_ranks * grad_stride, "grads"), grad_stride, scale,
        _dev(master, f32, T, "master"), _dev(m, f32, T, "m"), _dev(v, f32, T, "v"),
        _dev(grad_shards, f32, T, "grad_shards"), ctypes.byref(h), step, _stream(stream)))


def z3_step_layer_noalloc(layout: Layout, shards, grads, grad_stride: int, scale: float, master,
                          m, v, hp, step: int, stream=None):
    """z3_step_layer whose gathers write into the library's own static
    device array instead of a caller buffer: for callers that cannot
    allocate device memory (at most 16,777,216 elements per layer)."""
    b16, f32 = _dtypes()
    T = layout.psi_padded
    h = _hp(hp)
    _check(load().z3_step_layer_noalloc(
        layout.handle, _dev(shards, b16, T, "shards"),
        _dev(grads, b16, layout.n_ranks * grad_stride, "grads"), grad_stride, scale,
        _dev(master, f32, T, "master"), _dev(m, f32, T, "m"), _dev(v, f32, T, "v"),
        ctypes.byref(h), step, _stream(stream)))


def z3_allreduce(layout: Layout, grads, grad_stride: int, out, scale: float, stream=None):
    b16, f32 = _dtypes()
    _check(load().z3_allreduce(
        layout.handle, _dev(grads, b16, layout.n_ranks * grad_stride, "grads"), grad_stride,
        _dev(out, f32, layout.psi, "out"), scale, _stream(stream)))


def z3_scatter(layout: Layout, full, shards, stream=None):
    _, f32 = _dtypes()
    _check(load().z3_scatter(layout.handle, _dev(full, f32, layout.psi, "full"),
                             _dev(shards, f32, layout.psi_padded, "shards"), _stream(stream)))


def z3_reshard(src_layout: Layout, dst_layout: Layout, src, dst, stream=None):
    """Element size from the tensors' dtype (bf16: 2 bytes, fp32: 4 bytes)."""
    b16, f32 = _dtypes()
    dt = b16 + f32
    elem = 2 if src.dtype in b16 else 4
    if (dst.dtype in b16) != (elem == 2):
        raise ValueError("src and dst must have the same element size")
    _check(load().z3_reshard(src_layout.handle, dst_layout.handle, elem,
                             _dev(src, dt, src_layout.psi_padded, "src"),
                             _dev(dst, dt, dst_layout.psi_padded, "dst"), _stream(stream)))


def z3_model_step(units, full, hp, step: int, stream=None, gather_stream=None):
    """units: sequence of (layout, shards, master, m, v, grads, grad_stride,
    scale[, resident[, hp]]) -- resident is None for a unit gathered at each
    use, else that unit's persistent bf16 [Psi] copy; hp is None for the
    step's hyperparameters, else this unit's own; full: one transient buffer,
    or D + 1 of them for the prefetching schedule (then gather_stream is
    required)."""
    b16, f32 = _dtypes()
    arr = (Unit * len(units))()
    own_hp = []                     # kept alive until the call returns
    need = 0
    for i, u in enumerate(units):
        L, sh, ma, m, v, g, stride, scale = u[:8]
        res = u[8] if len(u) > 8 else None
        uhp = u[9] if len(u) > 9 else None
        T = L.psi_padded
        hp_ptr = None
        if uhp is not None:
            own_hp.append(_hp(uhp))
            hp_ptr = ctypes.pointer(own_hp[-1])
        arr[i] = Unit(L.handle.value, _dev(sh, b16, T, "shards"), _dev(ma, f32, T, "master"),
                      _dev(m, f32, T, "m"), _dev(v, f32, T, "v"),
                      _dev(g, b16, L.n_ranks * stride, "grads"), stride, scale,
                      None if res is None else _dev(res, b16, L.psi, "resident"), hp_ptr)
        if res is None:
            need = max(need, L.psi)
    fulls = (ctypes.c_void_p * len(full))(*[_dev(f, b16, need, "full") for f in full])
    h = _hp(hp)
    _check(load().z3_model_step(arr, len(units), fulls, len(full), ctypes.byref(h), step,
                                _stream(stream),
                                None if gather_stream is None else _stream(gather_stream)))


def _host(t, dtypes, numel: int, name: str):
    """Host address of a CPU tensor (or a raw int address)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if t.is_cuda:
        raise ValueError(f"{name}: must be a host (CPU) tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name}: needs >= {numel} elements, has {t.numel()}")
    return t.data_ptr()


class HostStep:
    """z3_host_step_create / _run / _destroy: the layer step fed from host
    memory through two device staging buffers (caller-owned tensors kept
    alive by this object)."""

    def __init__(self, layout: Layout, staging0, staging1, grad_stride: int, upload_stream,
                 download_stream):
        b16, _ = _dtypes()
        n = layout.n_ranks * grad_stride
        self._keep = (layout, staging0, staging1, upload_stream, download_stream)
        self.layout, self.grad_stride = layout, grad_stride
        h = ctypes.c_void_p()
        _check(load().z3_host_step_create(
            layout.handle, _dev(staging0, b16, n, "staging0"), _dev(staging1, b16, n, "staging1"),
            grad_stride, _stream(upload_stream), _stream(download_stream), ctypes.byref(h)))
        self._h = h

    def run(self, grads_host, shards, full, scale: float, master, m, v, hp, step: int,
            shards_host=None, stream=None):
        b16, f32 = _dtypes()
        L = self.layout
        T = L.psi_padded
        h = _hp(hp)
        _check(load().z3_host_step_run(
            self._h, _host(grads_host, b16, L.n_ranks * self.grad_stride, "grads_host"),
            _dev(shards, b16, T, "shards"), _dev(full, b16, L.psi, "full"), scale,
            _dev(master, f32, T, "master"), _dev(m, f32, T, "m"), _dev(v, f32, T, "v"),
            ctypes.byref(h), step, _host(shards_host, b16, T, "shards_host"), _stream(stream)))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load().z3_host_step_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass
