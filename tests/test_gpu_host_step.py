"""The layer step fed from host memory (z3_host_step_*): gradients uploaded
from page-locked host buffers through two alternating device staging
buffers, the layer step, and the updated bf16 shards downloaded to host
buffers, with the uploads of later steps overlapping earlier steps.  Every
downloaded shard set and the final device state equal the oracle's layer
steps bit for bit."""
import numpy as np
import pytest
import torch

from gpu_helpers import bits32, f32, u16
from optimizer_state_gb300 import inputs as I

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)


@pytest.fixture(scope="module")
def z3mod():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is not available: the GPU tests need a GPU")
    from optimizer_state_gb300 import build, z3
    build.build()
    z3.load()
    return z3


@pytest.mark.parametrize("numel,n_ranks,steps", [([100003, 7, 4099], 3, 5),
                                                 (I.LAYER_D1024.numel, 8, 3)])
def test_host_step_matches_oracle(z3mod, orc, numel, n_ranks, steps):
    dev = torch.device("cuda")
    w = I.Workload("h", tuple((n,) for n in numel), n_ranks, 0.02, 1e-3)
    L, O = z3mod.Layout(numel, n_ranks), orc.layout(numel, n_ranks)
    T, stride = L.psi_padded, w.grad_stride
    gen = I.make_generator(17, dev)
    full0 = I.draw_master(w, gen, dev).to(dev)
    shards = torch.empty(T, dtype=torch.bfloat16, device=dev)
    master, m, v = (torch.empty(T, dtype=torch.float32, device=dev) for _ in range(3))
    z3mod.z3_partition(L, full0, shards, master, m, v)
    o_sh, o_ma, o_m, o_v = orc.partition(O, f32(full0))
    grads_host = []
    for _ in range(steps):
        g = I.draw_grads(w, gen, dev)
        h = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
        h.copy_(g)
        grads_host.append(h)
    shards_host = [torch.empty(T, dtype=torch.bfloat16, pin_memory=True) for _ in range(steps)]
    staging = [torch.empty(n_ranks * stride, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    full = torch.empty(L.psi, dtype=torch.bfloat16, device=dev)
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    pipe = z3mod.HostStep(L, staging[0], staging[1], stride, up, down)
    for t in range(1, steps + 1):
        pipe.run(grads_host[t - 1], shards, full, 1.0 / n_ranks, master, m, v, HP, t,
                 shards_host=shards_host[t - 1])
    torch.cuda.synchronize()
    for t in range(1, steps + 1):
        gh = u16(grads_host[t - 1]).reshape(-1)
        _, fb, _ = orc.step_layer(O, o_sh, gh, stride, 1.0 / n_ranks, o_ma, o_m, o_v, HP, t)
        assert np.array_equal(u16(shards_host[t - 1]), o_sh), f"downloaded shards, step {t}"
    for got, want in ((master, o_ma), (m, o_m), (v, o_v)):
        assert np.array_equal(bits32(f32(got)), bits32(want))
    assert np.array_equal(u16(shards), o_sh)
    assert np.array_equal(u16(full), fb)
    pipe.close()


def test_host_step_rejects_its_own_streams(z3mod):
    dev = torch.device("cuda")
    L = z3mod.Layout([4099, 77], 4)
    stride = -(-L.psi // 8) * 8
    staging = [torch.empty(4 * stride, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    pipe = z3mod.HostStep(L, staging[0], staging[1], stride, up, down)
    T = L.psi_padded
    shards = torch.zeros(T, dtype=torch.bfloat16, device=dev)
    master, m, v = (torch.zeros(T, dtype=torch.float32, device=dev) for _ in range(3))
    full = torch.empty(L.psi, dtype=torch.bfloat16, device=dev)
    grads = torch.zeros(4 * stride, dtype=torch.bfloat16, pin_memory=True)
    with pytest.raises(z3mod.Z3Error):
        pipe.run(grads, shards, full, 0.25, master, m, v, HP, 1, stream=up)
    with pytest.raises(z3mod.Z3Error):                     # staging buffer as the shards
        pipe.run(grads, staging[1][:T], full, 0.25, master, m, v, HP, 1)
    with pytest.raises(ValueError):                        # device tensor as the host buffer
        pipe.run(staging[0], shards, full, 0.25, master, m, v, HP, 1)
    pipe.close()
