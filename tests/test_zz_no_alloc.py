"""z3_step_layer_noalloc against z3_step_layer, through the C ABI.

z3_step_layer_noalloc serves callers that cannot allocate device memory
(code inside an allocator callback, a plugin that only receives buffers from
its host framework, a process whose device memory is all reserved up front):
instead of a caller-supplied transient gather buffer it uses a 32 MiB static
array in the library's own device memory.  Its results must be those of the
ordinary layer step.  Two replicas of the same layer state take the same two
steps in a row, one through each entry point, and must agree after each
call within the tolerance of the other parity tests (fp32 state within
1e-6 relative or 1e-9 absolute, bf16 within 1 ulp); both run the same
kernels, so they are also checked bit for bit.  A layer above the array's
16,777,216 elements is refused with a clear error (a host-side check, run
in a child process that sees no device).

This file is collected last so that a run that stops at its first failure
has run every other test first; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import bf16_ulp_distance, bits32, f32, u16, within_adam_tolerance
from optimizer_state_gb300 import inputs as I

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)


@pytest.fixture(scope="module")
def z3mod():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is not available: the GPU tests need a GPU")
    from optimizer_state_gb300 import build, z3
    build.build()
    z3.load()
    return z3


class Replica:
    def __init__(self, z3, L, full):
        T = L.psi_padded
        self.shards = torch.empty(T, dtype=torch.bfloat16, device="cuda")
        self.master, self.m, self.v = (torch.empty(T, dtype=torch.float32, device="cuda")
                                       for _ in range(3))
        z3.z3_partition(L, full, self.shards, self.master, self.m, self.v)

    def state(self):
        torch.cuda.synchronize()
        return dict(shards=u16(self.shards), master=f32(self.master), m=f32(self.m),
                    v=f32(self.v))


def _agree(got, want):
    for k in ("master", "m", "v"):
        assert within_adam_tolerance(got[k], want[k]).all(), k
        assert np.array_equal(bits32(got[k]), bits32(want[k])), k
    assert bf16_ulp_distance(got["shards"], want["shards"]).max(initial=0) <= 1
    assert np.array_equal(got["shards"], want["shards"])


@pytest.mark.gpu
@pytest.mark.parametrize("workload", [
    I.LAYER_D1024,
    I.Workload("primes", ((100003,), (7,), (1,), (4099,)), n_ranks=3, param_std=0.02,
               grad_std=1e-3),
], ids=["d1024", "primes"])
def test_noalloc_step_matches_step_layer(z3mod, workload):
    z3 = z3mod
    lib = z3.load()
    w = workload
    L = z3.Layout(w.numel, w.n_ranks)
    gen = I.make_generator(21, "cuda")
    full = I.draw_master(w, gen, "cuda")
    ref, noalloc = Replica(z3, L, full), Replica(z3, L, full)
    gathered = torch.empty(L.psi, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    hp = z3.AdamHP(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"])
    scale = 1.0 / w.n_ranks
    for step in (1, 2):
        grads = I.draw_grads(w, gen, "cuda")
        z3.z3_step_layer(L, ref.shards, gathered, grads, w.grad_stride, scale, ref.master,
                         ref.m, ref.v, HP, step)
        st = lib.z3_step_layer_noalloc(L.handle, noalloc.shards.data_ptr(), grads.data_ptr(),
                                       w.grad_stride, scale, noalloc.master.data_ptr(),
                                       noalloc.m.data_ptr(), noalloc.v.data_ptr(),
                                       ctypes.byref(hp), step, stream)
        assert st == z3.Z3_OK, z3.last_error()
        _agree(noalloc.state(), ref.state())


@pytest.mark.no_device
def test_noalloc_refuses_a_layer_beyond_its_scratch():
    """Host-side checks of the entry point: the size limit, and the empty
    layer."""
    from optimizer_state_gb300 import build, z3
    build.build()
    lib = z3.load()
    L = z3.Layout([(1 << 24) + 1], 8)
    hp = z3.AdamHP(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"])
    a = 1 << 32                  # a made-up address: the size check comes first
    st = lib.z3_step_layer_noalloc(L.handle, a, a, L.psi + 7, 0.125, a, a, a, ctypes.byref(hp),
                                   1, None)
    msg = z3.last_error()
    assert st == z3.Z3_ERR_INVALID_ARG
    assert "16777217" in msg and "16777216" in msg, msg
    # an empty layer is a no-op that needs neither the array nor a device
    L0 = z3.Layout([0, 0], 4)
    assert lib.z3_step_layer_noalloc(L0.handle, None, None, 8, 0.25, None, None, None,
                                     ctypes.byref(hp), 1, None) == z3.Z3_OK
