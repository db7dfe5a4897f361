"""Parity at the full sizes of the larger workloads, in the launch
configuration bench.py uses: the 7B-style layer at N_d = 8 and 64, the
24-layer full step at N_d = 16, and the prime-length sweep with four
micro-batches (including the largest points).  The oracle computes a sample
of outputs one by one from the input bytes read back at those positions:
every rank's first and last owned element of every parameter, both sides of
every pad boundary, and random positions.
"""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import (bits32, f32, gather_rows, pick, sampled_shard_positions,
                         shard_to_full, u16)
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


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


class Probe:
    """State of one layer at sampled shard positions, before a step."""

    def __init__(self, orc, O, shards, master, m, v, n_random=1 << 20, seed=0):
        self.O = O
        self.xs = sampled_shard_positions(O, n_random, seed)
        self.e, self.valid = shard_to_full(O, self.xs)
        self.shards = u16(pick(shards, self.xs))
        self.master = f32(pick(master, self.xs))
        self.m = f32(pick(m, self.xs))
        self.v = f32(pick(v, self.xs))

    def expected(self, orc, grads, stride, scale, hp, t, acc=None):
        """Oracle outputs at the sampled positions after one fused
        reduce-scatter + Adam (acc: running sums at the positions, or None)."""
        O, ev = self.O, self.e[self.valid]
        nv = int(ev.size)
        G = np.ascontiguousarray(gather_rows(grads, O.n_ranks, stride, ev))
        fold = orc.allreduce(orc.layout([nv], O.n_ranks), G.reshape(-1), nv, scale)
        g = np.zeros(self.xs.size, np.float32)
        g[self.valid] = fold
        if acc is not None:
            g[self.valid] = (acc[self.valid] + g[self.valid]).astype(np.float32)
        p, m, v = self.master.copy(), self.m.copy(), self.v.copy()
        bf = np.zeros(self.xs.size, np.uint16)
        grad = g.copy()
        orc.adam(p, m, v, g, bf, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"],
                 hp["weight_decay"], t)
        return dict(master=p, m=m, v=v, shards=bf, grad=grad)

    def check_after(self, want, shards, master, m, v):
        got = dict(shards=u16(pick(shards, self.xs)), master=f32(pick(master, self.xs)),
                   m=f32(pick(m, self.xs)), v=f32(pick(v, self.xs)))
        for k in ("master", "m", "v"):
            assert np.array_equal(bits32(got[k]), bits32(want[k])), k
        assert np.array_equal(got["shards"], want["shards"])

    def check_gather(self, full):
        """The gathered buffer holds the pre-step bf16 shard values."""
        got = u16(pick(full, self.e[self.valid]))
        assert np.array_equal(got, self.shards[self.valid])


def _layer_step(z3mod, orc, w, seed):
    dev = torch.device("cuda")
    L = z3mod.Layout(w.numel, w.n_ranks)
    O = orc.layout(w.numel, w.n_ranks)
    gen = I.make_generator(seed, dev)
    full32 = I.draw_master(w, gen, dev)
    T = L.psi_padded
    shards = torch.empty(T, dtype=torch.bfloat16, device=dev)
    master, m, v = (torch.empty(T, dtype=torch.float32, device=dev) for _ in range(3))
    z3mod.z3_partition(L, full32, shards, master, m, v)
    # partition at the sampled positions
    pr = Probe(orc, O, shards, master, m, v)
    ev = pr.e[pr.valid]
    assert np.array_equal(bits32(pr.master[pr.valid]), bits32(f32(pick(full32, ev))))
    assert not pr.master[~pr.valid].any() and not pr.shards[~pr.valid].any()
    del full32
    full = torch.empty(L.psi, dtype=torch.bfloat16, device=dev)
    for t in (1, 2):
        grads = I.draw_grads(w, gen, dev)
        pr = Probe(orc, O, shards, master, m, v, seed=t)
        want = pr.expected(orc, grads, w.grad_stride, 1.0 / w.n_ranks, w.hp, t)
        # the second step also stores the reduced gradient (grad_shards_or_NULL)
        gsh = torch.full((T,), float("nan"), dtype=torch.float32, device=dev) if t == 2 else None
        z3mod.z3_step_layer(L, shards, full, grads, w.grad_stride, 1.0 / w.n_ranks, master, m,
                            v, w.hp, t, grad_shards=gsh)
        torch.cuda.synchronize()
        pr.check_gather(full)
        pr.check_after(want, shards, master, m, v)
        if gsh is not None:
            assert np.array_equal(bits32(f32(pick(gsh, pr.xs))), bits32(want["grad"]))
        del grads, gsh


@pytest.mark.parametrize("n_ranks", [8, 64])
def test_layer_7b(z3mod, orc, n_ranks):
    _layer_step(z3mod, orc, I.layer_7b(n_ranks), seed=7)


@pytest.mark.parametrize("n_ranks", [8, 3])
def test_layer_primes_mixed_phases(z3mod, orc, n_ranks):
    """Three prime-length parameters: the generic, window-shifting kernels."""
    from optimizer_state_gb300 import z3
    w = I.layer_primes(n_ranks)
    L = z3.Layout(w.numel, n_ranks)
    assert L.psi == 101711929
    _layer_step(z3mod, orc, w, seed=8)


def test_full_step_24_layers(z3mod, orc):
    """24 d=1024 layers + embedding, N_d = 16: forward gathers of every unit,
    then backward gather + fused reduce-scatter/Adam in reverse unit order,
    all through one transient buffer."""
    from optimizer_state_gb300 import schedule
    dev = torch.device("cuda")
    model = schedule.full_step_model(dev, seed=3)
    assert model.psi == 353502208
    assert model.full.numel() == 50257 * 1024          # the largest unit
    probes = []
    for u in model.units:
        O = orc.layout(u.w.numel, u.w.n_ranks)
        probes.append(Probe(orc, O, u.shards, u.master, u.m, u.v, n_random=1 << 15))
    wants = [pr.expected(orc, u.grads, u.w.grad_stride, 1.0 / u.w.n_ranks, HP, 1)
             for pr, u in zip(probes, model.units)]
    watch = {("forward", 0), ("forward", 1), ("forward", 24), ("backward", 24),
             ("backward", 1), ("backward", 0)}
    snaps = {}

    def on_gather(phase, i):
        if (phase, i) in watch:
            snaps[(phase, i)] = model.full[:model.units[i].L.psi].clone()
    model.step(HP, on_gather=on_gather)
    torch.cuda.synchronize()
    for (phase, i), buf in snaps.items():
        probes[i].check_gather(buf)          # every gather saw pre-step shards
    for pr, want, u in zip(probes, wants, model.units):
        pr.check_after(want, u.shards, u.master, u.m, u.v)


def _sweep_point(z3mod, orc, n, n_ranks, full_check: bool, seed=5):
    """One step of the sweep workload: forward and backward gathers, then 4
    micro-batches reduce-scattered and accumulated into fp32 slices, the last
    one fused with Adam ('ZeRO Stages: ...', stage-2 accumulation)."""
    w = I.sweep(n, n_ranks)
    dev = torch.device("cuda")
    L = z3mod.Layout(w.numel, n_ranks)
    O = orc.layout(w.numel, n_ranks)
    gen = I.make_generator(seed, dev)
    full32 = I.draw_master(w, gen, dev)
    T, stride, scale = L.psi_padded, w.grad_stride, 1.0 / n_ranks
    shards = torch.empty(T, dtype=torch.bfloat16, device=dev)
    master, m, v, acc = (torch.empty(T, dtype=torch.float32, device=dev) for _ in range(4))
    full = torch.empty(L.psi, dtype=torch.bfloat16, device=dev)
    z3mod.z3_partition(L, full32, shards, master, m, v)
    if full_check:
        o_sh, o_ma, o_m, o_v = orc.partition(O, f32(full32))
        assert np.array_equal(u16(shards), o_sh) and np.array_equal(bits32(f32(master)),
                                                                    bits32(o_ma))
    del full32
    pr = None if full_check else Probe(orc, O, shards, master, m, v, n_random=1 << 20)
    z3mod.z3_allgather(L, shards, full)
    z3mod.z3_allgather(L, shards, full)
    grads = torch.zeros((n_ranks, stride), dtype=torch.bfloat16, device=dev)
    o_acc = None
    p_acc = None
    for mb in range(w.micro_batches):
        I.draw_grads(w, gen, dev, out=grads)
        last = mb == w.micro_batches - 1
        if full_check:
            gh = u16(grads).reshape(-1)
            if mb == 0:
                o_acc = orc.reduce_scatter(O, gh, stride, scale)
            elif not last:
                orc.reduce_scatter(O, gh, stride, scale, out=o_acc, accumulate=True)
            else:
                want_full = orc.allgather(O, o_sh)
                orc.step_layer(O, o_sh, gh, stride, scale, o_ma, o_m, o_v, w.hp, 1,
                               grad_acc=o_acc.copy())
        else:
            ev = pr.e[pr.valid]
            G = np.ascontiguousarray(gather_rows(grads, n_ranks, stride, ev))
            fold = orc.allreduce(orc.layout([int(ev.size)], n_ranks), G.reshape(-1),
                                 int(ev.size), scale)
            if mb == 0:
                p_acc = np.zeros(pr.xs.size, np.float32)
                p_acc[pr.valid] = fold
            elif not last:
                p_acc[pr.valid] = (p_acc[pr.valid] + fold).astype(np.float32)
            else:
                want = pr.expected(orc, grads, stride, scale, w.hp, 1, acc=p_acc)
        if mb == 0:
            z3mod.z3_reduce_scatter(L, grads, stride, acc, scale)
        elif not last:
            z3mod.z3_reduce_scatter(L, grads, stride, acc, scale, accumulate=True)
        else:
            z3mod.z3_reduce_scatter_adam(L, grads, stride, scale, acc, master, m, v, shards,
                                         w.hp, 1)
    torch.cuda.synchronize()
    if full_check:
        assert np.array_equal(u16(full), want_full)
        assert np.array_equal(bits32(f32(acc)), bits32(o_acc))
        assert np.array_equal(bits32(f32(master)), bits32(o_ma))
        assert np.array_equal(bits32(f32(m)), bits32(o_m))
        assert np.array_equal(bits32(f32(v)), bits32(o_v))
        assert np.array_equal(u16(shards), o_sh)
    else:
        pr.check_gather(full)
        assert np.array_equal(bits32(f32(pick(acc, pr.xs))), bits32(p_acc))
        pr.check_after(want, shards, master, m, v)


@pytest.mark.parametrize("n_ranks", [2, 8, 64])
@pytest.mark.parametrize("n", [262147, 4194319])
def test_sweep_full_check(z3mod, orc, n, n_ranks):
    _sweep_point(z3mod, orc, n, n_ranks, full_check=True)


@pytest.mark.parametrize("n,n_ranks", [(67108879, 8), (2 ** 31 - 1, 2), (2 ** 31 - 1, 8),
                                       (1073741827, 64)])
def test_sweep_largest_points_sampled(z3mod, orc, n, n_ranks):
    """The largest sweep points that fit HBM (2^30+3 at N_d = 64 reads a
    137 GB gradient buffer; 2^31-1 at N_d = 64 would need 275 GB and is the
    capacity cap)."""
    _sweep_point(z3mod, orc, n, n_ranks, full_check=False)


def test_full_step_with_prefetch_matches(z3mod, orc):
    """The backward gathers prefetched one unit ahead on a second stream into
    two transient buffers: identical results, and each backward gather still
    sees the pre-step shards."""
    from optimizer_state_gb300 import schedule
    dev = torch.device("cuda")
    plain = schedule.full_step_model(dev, seed=11)
    pre = schedule.full_step_model(dev, seed=11, prefetch=True)
    snaps = {}

    def on_gather(phase, i):
        if phase == "backward" and i in (0, 1, 23, 24):
            snaps[i] = pre.bufs[i % 2][:pre.units[i].L.psi].clone()
    before = {i: u16(pre.units[i].shards) for i in snaps or (0, 1, 23, 24)}
    for t in (1, 2):
        plain.step(HP)
        pre.step(HP, on_gather=on_gather if t == 1 else None)
        torch.cuda.synchronize()
        if t == 1:
            for i, buf in snaps.items():
                O = orc.layout(pre.units[i].w.numel, 16)
                assert np.array_equal(u16(buf), orc.allgather(O, before[i]))
    for a, b in zip(plain.units, pre.units):
        for k in ("master", "m", "v"):
            assert np.array_equal(bits32(f32(getattr(a, k))), bits32(f32(getattr(b, k)))), k
        assert np.array_equal(u16(a.shards), u16(b.shards))


@pytest.mark.parametrize("bucket", [2, 6, 24])
def test_bucketed_full_step_matches_per_layer(z3mod, bucket):
    """Buckets of consecutive layers (one gather and one fused update launch
    per bucket): the parameters and fp32 state after two steps equal those of
    the per-layer schedule, bit for bit."""
    from optimizer_state_gb300 import schedule
    dev = torch.device("cuda")
    gen = I.make_generator(21, dev)
    per = I.full_step_units(1)
    psi = sum(w.psi for w in per)
    master = torch.empty(psi, dtype=torch.float32, device=dev).normal_(0, 0.02, generator=gen)
    grads = torch.empty((16, psi), dtype=torch.float32, device=dev).normal_(0, 1e-3,
                                                                          generator=gen)
    grads = grads.to(torch.bfloat16)

    def build(units_w):
        units, a = [], 0
        for w in units_w:
            units.append(schedule.Unit.from_full(w, dev, master[a:a + w.psi],
                                                 grads[:, a:a + w.psi]))
            a += w.psi
        return schedule.Model(units, dev)
    m1, mb = build(per), build(I.full_step_units(bucket))
    assert len(mb.units) == 1 + -(-24 // bucket)
    for _ in range(2):
        m1.step(HP)
        mb.step(HP)
    torch.cuda.synchronize()

    def gathered(model, name):
        out = []
        for u in model.units:
            full = torch.empty(u.L.psi, dtype=torch.float32, device=dev)
            # an fp32 gather: reshard the [N][S] buffer to one rank (S = Psi)
            L1 = z3mod.Layout(u.w.numel, 1)
            z3mod.z3_reshard(u.L, L1, getattr(u, name), full)
            out.append(full)
        return torch.cat(out)
    for name in ("master", "m", "v"):
        assert torch.equal(gathered(m1, name).view(torch.int32),
                           gathered(mb, name).view(torch.int32)), name


@pytest.mark.parametrize("stream", [None, 0])
@pytest.mark.parametrize("prefetch", [False, True])
def test_native_model_step_matches_issued_schedule(z3mod, prefetch, stream):
    """z3_model_step (the schedule inside the library) against the same
    schedule issued call by call: identical state after three steps, with
    the stream given as torch's current stream or as the raw handle 0 (the
    legacy default stream, which must not turn into a stream of its own)."""
    from optimizer_state_gb300 import schedule
    dev = torch.device("cuda")
    a = schedule.full_step_model(dev, seed=31, prefetch=prefetch, bucket_layers=3)
    b = schedule.full_step_model(dev, seed=31, prefetch=prefetch, bucket_layers=3)
    for _ in range(3):
        a.step(HP, stream=stream)                                   # native
        b.step(HP, stream=stream, on_gather=lambda phase, i: None)  # issued from Python
    torch.cuda.synchronize()
    for ua, ub in zip(a.units, b.units):
        for k in ("master", "m", "v"):
            assert torch.equal(getattr(ua, k).view(torch.int32), getattr(ub, k).view(torch.int32))
        assert torch.equal(ua.shards.view(torch.int16), ub.shards.view(torch.int16))


def test_model_step_argument_checks(z3mod):
    from optimizer_state_gb300 import schedule
    dev = torch.device("cuda")
    m = schedule.full_step_model(dev, seed=1, bucket_layers=24)
    with pytest.raises(z3mod.Z3Error):
        z3mod.z3_model_step(m.unit_args(), [m.full, m.full], HP, 1)        # no gather stream
    other = torch.empty_like(m.full)
    with pytest.raises(z3mod.Z3Error):                                      # overlapping buffers
        z3mod.z3_model_step(m.unit_args(), [m.full, other, other], HP, 1,
                            gather_stream=torch.cuda.Stream())
    with pytest.raises(z3mod.Z3Error):
        z3mod.z3_model_step(m.unit_args(), [m.full], HP, 0)                # step < 1
    small = torch.empty(16, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        z3mod.z3_model_step(m.unit_args(), [small], HP, 1)                 # too small


@pytest.mark.parametrize("depth", [2, 3])
def test_deeper_prefetch_matches(z3mod, depth):
    """Gathers up to `depth` units ahead (depth + 1 transient buffers): the
    same state as the unprefetched step."""
    from optimizer_state_gb300 import schedule
    dev = torch.device("cuda")
    a = schedule.full_step_model(dev, seed=41, bucket_layers=2)
    b = schedule.full_step_model(dev, seed=41, prefetch=depth, bucket_layers=2)
    assert len(b.bufs) == depth + 1
    for _ in range(2):
        a.step(HP)
        b.step(HP)
    torch.cuda.synchronize()
    for ua, ub in zip(a.units, b.units):
        for k in ("master", "m", "v"):
            assert torch.equal(getattr(ua, k).view(torch.int32), getattr(ub, k).view(torch.int32))
        assert torch.equal(ua.shards.view(torch.int16), ub.shards.view(torch.int16))


def _per_param(z3mod, model, ids, name):
    """Every parameter's fp32 state (or, for name == "shards", its bf16
    parameters) gathered to one rank, keyed by its model-order index."""
    dev = torch.device("cuda")
    out = {}
    for u, pid in zip(model.units, ids):
        buf = getattr(u, name)
        dt = torch.float32 if buf.dtype == torch.float32 else torch.bfloat16
        full = torch.empty(u.L.psi, dtype=dt, device=dev)
        z3mod.z3_reshard(u.L, z3mod.Layout(u.w.numel, 1), buf, full)
        a = 0
        for i, n in zip(pid, u.w.numel):
            out[i] = full[a:a + n]
            a += n
    return out


@pytest.mark.parametrize("bucket,prefetch,threshold,issued", [
    (1, 0, 100000, False), (4, 2, 100000, False), (2, 1, 100000, True), (1, 0, 100000, True),
    (6, 1, 4194305, False), (1, 0, 10 ** 9, False)])
def test_persistent_units_match_per_layer(z3mod, bucket, prefetch, threshold, issued):
    """Persistence threshold: parameters below it form one resident unit that
    is gathered once per step, after its update, and never released.  The
    state after three steps equals the per-layer schedule's bit for bit, and
    every resident copy holds exactly the current bf16 parameters."""
    from optimizer_state_gb300 import schedule
    dev = torch.device("cuda")
    gen = I.make_generator(23, dev)
    shapes = I._full_step_shapes()
    numel = [math.prod(s) for s in shapes]
    off = [0]
    for n in numel:
        off.append(off[-1] + n)
    psi = off[-1]
    master = torch.empty(psi, dtype=torch.float32, device=dev).normal_(0, 0.02, generator=gen)
    grads = torch.empty((16, psi), dtype=torch.float32, device=dev).normal_(0, 1e-3,
                                                                          generator=gen)
    grads = grads.to(torch.bfloat16)

    def build(b, T, depth):
        ws, ids = I.full_step_units(b, T), I.full_step_param_ids(b, T)
        units = []
        for w, pid in zip(ws, ids):
            mf = torch.cat([master[off[i]:off[i + 1]] for i in pid])
            gf = torch.cat([grads[:, off[i]:off[i + 1]] for i in pid], dim=1)
            units.append(schedule.Unit.from_full(w, dev, mf, gf))
        model = schedule.PrefetchModel(units, dev, depth) if depth else schedule.Model(units, dev)
        return model, ids
    ref, ref_ids = build(1, 0, 0)
    mp, ids = build(bucket, threshold, prefetch)
    assert mp.units[0].resident is not None
    for _ in range(3):
        ref.step(HP)
        if issued:
            mp.step(HP, on_gather=lambda phase, i: None)
        else:
            mp.step(HP)
    torch.cuda.synchronize()
    for name in ("master", "m", "v", "shards"):
        a, b = _per_param(z3mod, ref, ref_ids, name), _per_param(z3mod, mp, ids, name)
        vt = torch.int16 if name == "shards" else torch.int32
        for i in range(len(shapes)):
            assert torch.equal(a[i].view(vt), b[i].view(vt)), (name, i)
    bf = _per_param(z3mod, mp, ids, "shards")
    u0 = mp.units[0]
    want = torch.cat([bf[i] for i in ids[0]])
    assert torch.equal(u0.resident.view(torch.int16), want.view(torch.int16))
    assert torch.equal(want.view(torch.int16),
                       torch.cat([_per_param(z3mod, mp, ids, "master")[i] for i in ids[0]])
                       .to(torch.bfloat16).view(torch.int16))


def test_long_run_schedules_agree(z3mod):
    """Fifty steps of the 24-layer model under three schedules -- one layer
    per unit with stream launches; resident norm gains, gathers two units
    ahead; 5-layer buckets, gathers three units ahead, the steps replayed
    from a CUDA graph -- end in the same parameters and fp32 state, bit for
    bit.  The schedules order their dependent launches differently, so a
    missing dependency would show up as a difference here."""
    from optimizer_state_gb300 import schedule
    dev = torch.device("cuda")
    gen = I.make_generator(77, dev)
    shapes = I._full_step_shapes()
    numel = [math.prod(s) for s in shapes]
    off = [0]
    for n in numel:
        off.append(off[-1] + n)
    master = torch.empty(off[-1], dtype=torch.float32, device=dev).normal_(0, 0.02, generator=gen)
    grads = torch.empty((16, off[-1]), dtype=torch.float32, device=dev).normal_(
        0, 1e-3, generator=gen).to(torch.bfloat16)

    def build(b, T, depth):
        ws, ids = I.full_step_units(b, T), I.full_step_param_ids(b, T)
        units = [schedule.Unit.from_full(
            w, dev, torch.cat([master[off[i]:off[i + 1]] for i in pid]),
            torch.cat([grads[:, off[i]:off[i + 1]] for i in pid], dim=1))
            for w, pid in zip(ws, ids)]
        m = schedule.PrefetchModel(units, dev, depth) if depth else schedule.Model(units, dev)
        return m, ids
    a, ids_a = build(1, 0, 0)
    b, ids_b = build(1, 100000, 2)
    c, ids_c = build(5, 0, 3)
    steps = 50
    for _ in range(steps):
        a.step(HP)
        b.step(HP)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s), torch.cuda.graph(g, stream=s):
        for _ in range(steps):
            c.step(HP, stream=s.cuda_stream)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    for name in ("master", "m", "v", "shards"):
        pa = _per_param(z3mod, a, ids_a, name)
        pb = _per_param(z3mod, b, ids_b, name)
        pc = _per_param(z3mod, c, ids_c, name)
        vt = torch.int16 if name == "shards" else torch.int32
        for i in range(len(shapes)):
            assert torch.equal(pa[i].view(vt), pb[i].view(vt)), (name, i, "resident/prefetch")
            assert torch.equal(pa[i].view(vt), pc[i].view(vt)), (name, i, "bucket/graph")
