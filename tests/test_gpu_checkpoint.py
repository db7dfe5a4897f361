"""Checkpoint and reshard on the GPU.

z3_reshard against the oracle's definition (gather the old shards, partition
for the new rank count), for bf16 and fp32 buffers; save/load at the same
rank count resumes bit for bit; load at another rank count gives exactly the
state a fresh partition at that count would hold, and training continues
from it ('ZeRO Stages: ...', 'Where the shards live and what happens on
failure').
"""
import numpy as np
import pytest
import torch

from gpu_helpers import bits32, f32, u16
from optimizer_state_gb300 import inputs as I

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
PAIRS = [([35, 13, 12], 4, 3), ([100003, 7, 1, 0, 4099], 3, 8), ([262147], 64, 2),
         ([262147], 2, 64), (I.LAYER_D1024.numel, 8, 16), (I.LAYER_D1024.numel, 8, 1)]


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is not available: the GPU tests need a GPU")
    from optimizer_state_gb300 import build, checkpoint, schedule, z3
    build.build()
    z3.load()
    return z3, schedule, checkpoint


@pytest.mark.parametrize("numel,n_src,n_dst", PAIRS)
def test_reshard_matches_oracle(mods, orc, numel, n_src, n_dst):
    z3, sch, _ = mods
    dev = torch.device("cuda")
    w = I.Workload("r", tuple((n,) for n in numel), n_src, 0.02, 1e-3)
    u = sch.Unit(w, dev, I.make_generator(4, dev), grads=False)
    Os, Od = orc.layout(numel, n_src), orc.layout(numel, n_dst)
    Ld = z3.Layout(numel, n_dst)
    full = orc.allgather_f32(Os, f32(u.master))
    _, want_ma, _, _ = orc.partition(Od, full)
    want_sh = orc.partition(Od, orc.f32_from_bf16(orc.allgather(Os, u16(u.shards))))[0]
    got_ma = torch.full((Ld.psi_padded,), 7.0, dtype=torch.float32, device=dev)
    got_sh = torch.full((Ld.psi_padded,), 7.0, dtype=torch.bfloat16, device=dev)
    z3.z3_reshard(u.L, Ld, u.master, got_ma)
    z3.z3_reshard(u.L, Ld, u.shards, got_sh)
    torch.cuda.synchronize()
    assert np.array_equal(bits32(f32(got_ma)), bits32(want_ma))
    assert np.array_equal(u16(got_sh), want_sh)


def test_reshard_rejects_other_parameters(mods):
    z3, _, _ = mods
    a, b = z3.Layout([100, 28], 4), z3.Layout([100, 29], 4)
    x = torch.zeros(a.psi_padded, dtype=torch.float32, device="cuda")
    y = torch.zeros(b.psi_padded, dtype=torch.float32, device="cuda")
    with pytest.raises(z3.Z3Error):
        z3.z3_reshard(a, b, x, y)


def _steps(z3, u, full, t0, n, gen, dev):
    for t in range(t0, t0 + n):
        g = I.draw_grads(u.w, gen, dev)
        z3.z3_step_layer(u.L, u.shards, full, g, u.w.grad_stride, 1.0 / u.w.n_ranks, u.master,
                         u.m, u.v, HP, t)


def test_save_load_resume(mods, orc, tmp_path):
    z3, sch, ck = mods
    dev = torch.device("cuda")
    w = I.Workload("ck", tuple((n,) for n in (4099, 77, 1024, 131)), 8, 0.02, 1e-3)
    a = sch.Unit(w, dev, I.make_generator(1, dev), grads=False)
    full = torch.empty(a.L.psi, dtype=torch.bfloat16, device=dev)
    gen_a = I.make_generator(2, dev)
    _steps(z3, a, full, 1, 2, gen_a, dev)
    ck.save(str(tmp_path / "c"), a.L, a.shards, a.master, a.m, a.v, step=2)
    # reference: continue without the checkpoint
    state_gen = gen_a.get_state()
    _steps(z3, a, full, 3, 1, gen_a, dev)
    # resume at the same rank count
    L, s, t = ck.load(str(tmp_path / "c"))
    assert t == 2 and L.n_ranks == 8
    b = sch.Unit(w, dev, None, grads=False)
    for k in ("shards", "master", "m", "v"):
        getattr(b, k).copy_(s[k])
    gen_b = I.make_generator(0, dev)
    gen_b.set_state(state_gen)
    _steps(z3, b, full, 3, 1, gen_b, dev)
    torch.cuda.synchronize()
    for k in ("master", "m", "v"):
        assert np.array_equal(bits32(f32(getattr(a, k))), bits32(f32(getattr(b, k)))), k
    assert np.array_equal(u16(a.shards), u16(b.shards))
    # resume at another rank count: the state a fresh partition would hold
    O8 = orc.layout(w.numel, 8)
    for n_new in (4, 16):
        L2, s2, _ = ck.load(str(tmp_path / "c"), n_ranks=n_new)
        O2 = orc.layout(w.numel, n_new)
        for k in ("master", "m", "v"):
            saved = ck.read_host(str(tmp_path / "c"))[1][k]
            want = orc.partition(O2, orc.allgather_f32(O8, saved))[1]
            assert np.array_equal(bits32(f32(s2[k])), bits32(want)), (n_new, k)
        # and a step runs from it (checked against the oracle at the new N)
        w2 = I.Workload("ck2", w.shapes, n_new, 0.02, 1e-3)
        g = I.draw_grads(w2, I.make_generator(5, dev), dev)
        sh, ma, m, v = (u16(s2["shards"]), f32(s2["master"]).copy(), f32(s2["m"]).copy(),
                        f32(s2["v"]).copy())
        full2 = torch.empty(L2.psi, dtype=torch.bfloat16, device=dev)
        z3.z3_step_layer(L2, s2["shards"], full2, g, w2.grad_stride, 1.0 / n_new, s2["master"],
                         s2["m"], s2["v"], HP, 3)
        orc.step_layer(O2, sh, u16(g).reshape(-1), w2.grad_stride, 1.0 / n_new, ma, m, v, HP, 3)
        torch.cuda.synchronize()
        assert np.array_equal(bits32(f32(s2["master"])), bits32(ma))
        assert np.array_equal(u16(s2["shards"]), sh)


def _model(sch, dev, seed, n_ranks, depth):
    """A small three-unit model: a resident unit of small parameters and two
    layers of odd lengths, every unit at n_ranks."""
    ws = [I.Workload("res", ((77,), (1024,)), n_ranks, 0.02, 1e-3, resident=True),
          I.Workload("l0", ((100003,), (4099,), (3, 7)), n_ranks, 0.02, 1e-3),
          I.Workload("l1", ((65536,), (262147,)), n_ranks, 0.02, 1e-3)]
    gen = I.make_generator(seed, dev)
    units = [sch.Unit(w, dev, gen) for w in ws]
    return sch.PrefetchModel(units, dev, depth) if depth else sch.Model(units, dev)


@pytest.mark.parametrize("n_src,n_dst,depth", [(4, 4, 0), (4, 4, 2), (6, 3, 1)])
def test_model_save_load_resume(mods, tmp_path, n_src, n_dst, depth):
    """A whole model (resident unit included) saved between steps and loaded
    into another model: every unit's gathered parameters and fp32 state equal
    the saved model's (resharded on the device when the rank count differs),
    the resident copy is rebuilt from the loaded shards and the step counter
    is restored.  At the same rank count, two more steps on both models agree
    bit for bit."""
    z3, sch, ckpt = mods
    dev = torch.device("cuda")
    a = _model(sch, dev, 11, n_src, depth)
    for _ in range(2):
        a.step(HP)
    ckpt.save_model(str(tmp_path / "m"), a)
    b = _model(sch, dev, 99, n_dst, depth)          # another initial state, then loaded
    if n_src == n_dst:
        for ub, ua in zip(b.units, a.units):        # the same gradients from here on
            ub.grads.copy_(ua.grads)
    ckpt.load_model(str(tmp_path / "m"), b)
    assert b.t == a.t == 2

    def per_unit(model, name):
        out = []
        for u in model.units:
            L1 = z3.Layout(u.w.numel, 1)
            dt = torch.bfloat16 if name == "shards" else torch.float32
            t = torch.empty(u.L.psi, dtype=dt, device=dev)
            z3.z3_reshard(u.L, L1, getattr(u, name), t)
            out.append(t)
        return out
    for name in ("shards", "master", "m", "v"):
        for x, y in zip(per_unit(a, name), per_unit(b, name)):
            vt = torch.int16 if name == "shards" else torch.int32
            assert torch.equal(x.view(vt), y.view(vt)), name
    assert torch.equal(a.units[0].resident.view(torch.int16), b.units[0].resident.view(torch.int16))
    if n_src == n_dst:
        for _ in range(2):
            a.step(HP)
            b.step(HP)
        torch.cuda.synchronize()
        for ua, ub in zip(a.units, b.units):
            for name in ("master", "m", "v"):
                assert torch.equal(getattr(ua, name).view(torch.int32),
                                   getattr(ub, name).view(torch.int32)), name
            assert torch.equal(ua.shards.view(torch.int16), ub.shards.view(torch.int16))
        assert torch.equal(a.units[0].resident.view(torch.int16),
                           b.units[0].resident.view(torch.int16))
