"""The ABI calls inside a captured CUDA graph: a layer step captured once
(fixed step t) and replayed equals the same step run eagerly, bit for bit.
The calls allocate nothing and make no synchronous CUDA call, and their
programmatic-dependent-launch attribute becomes a graph edge."""
import numpy as np
import pytest
import torch

from gpu_helpers import bits32, f32, u16
from optimizer_state_gb300 import inputs as I

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is not available: the GPU tests need a GPU")
    from optimizer_state_gb300 import build, schedule, z3
    build.build()
    z3.load()
    return z3, schedule


@pytest.mark.parametrize("numel,n_ranks", [(I.LAYER_D1024.numel, 8), ([100003, 7, 4099], 3)])
def test_captured_step_equals_eager(mods, numel, n_ranks):
    z3, sch = mods
    dev = torch.device("cuda")
    w = I.Workload("g", tuple((n,) for n in numel), n_ranks, 0.02, 1e-3)
    a = sch.Unit(w, dev, I.make_generator(6, dev))
    b = sch.Unit(w, dev, I.make_generator(6, dev))
    fa = torch.empty(a.L.psi, dtype=torch.bfloat16, device=dev)
    fb = torch.empty(a.L.psi, dtype=torch.bfloat16, device=dev)
    z3.z3_step_layer(a.L, a.shards, fa, a.grads, w.grad_stride, 1.0 / n_ranks, a.master, a.m,
                     a.v, HP, 1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        z3.z3_step_layer(b.L, b.shards, fb, b.grads, w.grad_stride, 1.0 / n_ranks, b.master,
                         b.m, b.v, HP, 1, stream=s.cuda_stream)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    # capture only recorded the work: b is still the initial state
    assert not torch.equal(a.master, b.master)
    g.replay()
    torch.cuda.synchronize()
    for k in ("master", "m", "v"):
        assert np.array_equal(bits32(f32(getattr(a, k))), bits32(f32(getattr(b, k)))), k
    assert np.array_equal(u16(a.shards), u16(b.shards))
    assert np.array_equal(u16(fa), u16(fb))


def test_side_stream(mods):
    """Calls enqueue on the stream they are given."""
    z3, sch = mods
    dev = torch.device("cuda")
    w = I.Workload("s", ((4099,), (77,)), 8, 0.02, 1e-3)
    a = sch.Unit(w, dev, I.make_generator(2, dev))
    b = sch.Unit(w, dev, I.make_generator(2, dev))
    fa = torch.empty(a.L.psi, dtype=torch.bfloat16, device=dev)
    fb = torch.empty(a.L.psi, dtype=torch.bfloat16, device=dev)
    z3.z3_step_layer(a.L, a.shards, fa, a.grads, w.grad_stride, 0.125, a.master, a.m, a.v, HP, 1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    z3.z3_step_layer(b.L, b.shards, fb, b.grads, w.grad_stride, 0.125, b.master, b.m, b.v, HP, 1,
                     stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert np.array_equal(bits32(f32(a.master)), bits32(f32(b.master)))


@pytest.mark.parametrize("depth", [0, 2])
def test_captured_model_step_equals_eager(mods, depth):
    """A whole model step (z3_model_step: the units' gathers, updates and,
    with prefetch, the fork onto the gather stream and the join back) with
    a resident unit, captured once and replayed twice, equals two eager
    steps at the same t, bit for bit."""
    z3, sch = mods
    dev = torch.device("cuda")
    ws = [I.Workload("res", ((77,), (1024,)), 8, 0.02, 1e-3, resident=True),
          I.Workload("u1", ((100003,), (4099,)), 8, 0.02, 1e-3),
          I.Workload("u2", ((65536,), (3, 1001)), 8, 0.02, 1e-3),
          I.Workload("u3", ((262147,),), 8, 0.02, 1e-3)]

    def model(seed):
        gen = I.make_generator(seed, dev)
        units = [sch.Unit(w, dev, gen) for w in ws]
        return sch.PrefetchModel(units, dev, depth) if depth else sch.Model(units, dev)
    a, b = model(9), model(9)
    for _ in range(2):
        a.step(HP, t=1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        b.step(HP, stream=s.cuda_stream, t=1)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for ua, ub in zip(a.units, b.units):
        for k in ("master", "m", "v"):
            assert np.array_equal(bits32(f32(getattr(ua, k))), bits32(f32(getattr(ub, k)))), k
        assert np.array_equal(u16(ua.shards), u16(ub.shards))
    assert np.array_equal(u16(a.units[0].resident), u16(b.units[0].resident))
