"""CUDA path vs oracle, element by element, through the C-ABI.

Every ABI device call (partition, all-gather, reduce-scatter with and
without accumulation, shard Adam, fused reduce-scatter + Adam with and
without running sums, the layer step) runs on seeded inputs on the GPU; the
oracle runs on the same input bytes read back to the host.  Layout,
partition, gathers and the fixed-order fp32 reduction must be bit-exact; the
Adam outputs must meet the contract tolerance (fp32 within 1e-6 relative or
1e-9 absolute, bf16 within 1 ulp) and, by construction of both sides
(IEEE-rounded binary32 operations in one order), are checked bit-exact too.
Every output buffer carries guard words that must survive each call.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import Guarded, bf16_ulp_distance, bits32, f32, u16, within_adam_tolerance
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


def assert_adam_equal(got: dict, want: dict, exact: bool = True):
    for name in ("master", "m", "v"):
        g, w = got[name], want[name]
        ok = within_adam_tolerance(g, w)
        assert ok.all(), f"{name}: {np.count_nonzero(~ok)} elements outside tolerance"
        if exact:
            assert np.array_equal(bits32(g), bits32(w)), f"{name}: not bit-exact"
    d = bf16_ulp_distance(got["shards"], want["shards"])
    assert d.max(initial=0) <= 1, "bf16 shard beyond 1 ulp"
    if exact:
        assert np.array_equal(got["shards"], want["shards"])


class Case:
    """Device and oracle state of one layer."""

    def __init__(self, z3, orc, numel, n_ranks, seed, param_std=0.02, grad_std=1e-3,
                 gen_device="cuda"):
        self.z3, self.orc = z3, orc
        self.w = I.Workload("case", tuple((n,) for n in numel), n_ranks, param_std, grad_std)
        self.L = z3.Layout(numel, n_ranks)
        self.O = orc.layout(numel, n_ranks)
        self.N = n_ranks
        self.stride = self.w.grad_stride
        self.gen = I.make_generator(seed, gen_device)
        self.gen_device = gen_device
        T, psi = self.L.psi_padded, self.L.psi
        full = I.draw_master(self.w, self.gen, gen_device).to("cuda")
        self.full_host = f32(full)
        self.shards = Guarded(T, torch.bfloat16)
        self.master = Guarded(T, torch.float32)
        self.m = Guarded(T, torch.float32)
        self.v = Guarded(T, torch.float32)
        self.gathered = Guarded(psi, torch.bfloat16)
        self.bufs = [self.shards, self.master, self.m, self.v, self.gathered]
        z3.z3_partition(self.L, full, self.shards.t, self.master.t, self.m.t, self.v.t)
        sh, ma, m, v = orc.partition(self.O, self.full_host)
        self.o = dict(shards=sh, master=ma, m=m, v=v)

    def grads(self):
        g = I.draw_grads(self.w, self.gen, self.gen_device).to("cuda")
        return g, u16(g).reshape(-1)

    def device_state(self):
        torch.cuda.synchronize()
        return dict(shards=u16(self.shards.t), master=f32(self.master.t), m=f32(self.m.t),
                    v=f32(self.v.t))

    def guards_ok(self):
        torch.cuda.synchronize()
        return all(b.guards_intact() for b in self.bufs)


def _check_partition(c: Case):
    got = c.device_state()
    for k in ("master", "m", "v"):
        assert np.array_equal(bits32(got[k]), bits32(c.o[k])), k
    assert np.array_equal(got["shards"], c.o["shards"])
    assert c.guards_ok()


def run_all_calls(z3, orc, numel, n_ranks, seed, steps=2):
    c = Case(z3, orc, numel, n_ranks, seed)
    _check_partition(c)
    scale = 1.0 / n_ranks
    T = c.L.psi_padded
    gs = Guarded(T, torch.float32)
    c.bufs.append(gs)
    for step in range(1, steps + 1):
        # all-gather
        z3.z3_allgather(c.L, c.shards.t, c.gathered.t)
        want_full = orc.allgather(c.O, c.o["shards"])
        torch.cuda.synchronize()
        assert np.array_equal(u16(c.gathered.t), want_full)
        # reduce-scatter, then accumulate a second micro-batch
        g1, g1h = c.grads()
        g2, g2h = c.grads()
        z3.z3_reduce_scatter(c.L, g1, c.stride, gs.t, scale)
        want = orc.reduce_scatter(c.O, g1h, c.stride, scale)
        torch.cuda.synchronize()
        assert np.array_equal(bits32(f32(gs.t)), bits32(want))
        z3.z3_reduce_scatter(c.L, g2, c.stride, gs.t, scale, accumulate=True)
        orc.reduce_scatter(c.O, g2h, c.stride, scale, out=want, accumulate=True)
        torch.cuda.synchronize()
        assert np.array_equal(bits32(f32(gs.t)), bits32(want))
        # shard Adam on the accumulated gradient
        z3.z3_adam_shard_step(c.L, c.master.t, c.m.t, c.v.t, gs.t, c.shards.t, HP, 2 * step - 1)
        orc.adam(c.o["master"], c.o["m"], c.o["v"], want, c.o["shards"], HP["lr"], HP["beta1"],
                 HP["beta2"], HP["eps"], HP["weight_decay"], 2 * step - 1)
        assert_adam_equal(c.device_state(), c.o)
        # fused reduce-scatter + Adam with running sums (micro-batch tail)
        g3, g3h = c.grads()
        acc = want.copy()
        z3.z3_reduce_scatter_adam(c.L, g3, c.stride, scale, gs.t, c.master.t, c.m.t, c.v.t,
                                  c.shards.t, HP, 2 * step)
        orc.step_layer(c.O, c.o["shards"], g3h, c.stride, scale, c.o["master"], c.o["m"],
                       c.o["v"], HP, 2 * step, grad_acc=acc)
        assert_adam_equal(c.device_state(), c.o)
        assert np.array_equal(bits32(f32(gs.t)), bits32(want)), "grad_acc must be read only"
    # the layer step: AG fwd, AG bwd, fused RS + Adam; the second one also
    # stores the reduced gradient (grad_shards_or_NULL)
    for step in range(2 * steps + 1, 2 * steps + 3):
        g, gh = c.grads()
        out = gs.t if step % 2 == 0 else None
        if out is not None:
            out.fill_(float("nan"))
        z3.z3_step_layer(c.L, c.shards.t, c.gathered.t, g, c.stride, scale, c.master.t, c.m.t,
                         c.v.t, HP, step, grad_shards=out)
        ff, fb, want_gs = orc.step_layer(c.O, c.o["shards"], gh, c.stride, scale, c.o["master"],
                                         c.o["m"], c.o["v"], HP, step)
        got = c.device_state()
        assert np.array_equal(u16(c.gathered.t), fb)
        assert_adam_equal(got, c.o)
        if out is not None:
            assert np.array_equal(bits32(f32(out)), bits32(want_gs))
    assert c.guards_ok()
    return c


# Layouts that span several tiles per chunk, ragged tails, every phase of
# the two index spaces, pad-only ranks, empty parameters, N = 1, and more
# parameters than one launch table holds.
ODD = [
    ([35, 13, 12], 4),                      # the Tiny layer
    ([100003, 7, 1, 0, 4099], 3),
    ([262147], 2),
    ([262147], 8),
    ([65537, 33, 8191], 64),
    ([5, 3, 2], 8),                         # n < N: pad-only ranks
    ([123457, 31], 1),
    ([int(x) for x in np.random.default_rng(7).integers(0, 3000, size=97)], 5),
    ([8192, 4096, 16], 8),                  # fully aligned
    ([5000, 123], 1000),                    # 1000 ranks: most own one element or only pad
]


@pytest.mark.parametrize("numel,n_ranks", ODD, ids=[f"{len(a)}p-N{b}" for a, b in ODD])
def test_all_calls_odd_layouts(z3mod, orc, numel, n_ranks):
    run_all_calls(z3mod, orc, numel, n_ranks, seed=11)


def test_tiny_workload_three_steps(z3mod, orc):
    """The Tiny workload as defined: 3 parameters, N = 4, params N(0, 0.02),
    grads N(0, 1), 3 layer steps, everything bit-exact."""
    w = I.TINY
    c = Case(z3mod, orc, w.numel, w.n_ranks, seed=0, param_std=w.param_std,
             grad_std=w.grad_std, gen_device="cpu")
    _check_partition(c)
    assert (c.L.S, c.L.psi_padded) == (16, 64)
    for step in range(1, w.steps + 1):
        g, gh = c.grads()
        z3mod.z3_step_layer(c.L, c.shards.t, c.gathered.t, g, c.stride, 1.0 / w.n_ranks,
                            c.master.t, c.m.t, c.v.t, w.hp, step)
        _, fb, _ = orc.step_layer(c.O, c.o["shards"], gh, c.stride, 1.0 / w.n_ranks,
                                  c.o["master"], c.o["m"], c.o["v"], w.hp, step)
        assert np.array_equal(u16(c.gathered.t), fb)
        assert_adam_equal(c.device_state(), c.o)
    assert c.guards_ok()


def test_layer_d1024_full_check(z3mod, orc):
    """One d=1024 transformer layer, N = 8, two layer steps, every element."""
    w = I.LAYER_D1024
    c = Case(z3mod, orc, w.numel, w.n_ranks, seed=0)
    _check_partition(c)
    for step in (1, 2):
        g, gh = c.grads()
        z3mod.z3_step_layer(c.L, c.shards.t, c.gathered.t, g, c.stride, 1.0 / w.n_ranks,
                            c.master.t, c.m.t, c.v.t, w.hp, step)
        _, fb, _ = orc.step_layer(c.O, c.o["shards"], gh, c.stride, 1.0 / w.n_ranks,
                                  c.o["master"], c.o["m"], c.o["v"], w.hp, step)
        assert np.array_equal(u16(c.gathered.t), fb)
        assert_adam_equal(c.device_state(), c.o)
    assert c.guards_ok()


@pytest.mark.parametrize("numel,n_ranks", [([35, 13, 12], 4), ([100003, 7, 1, 0, 4099], 3),
                                            ([65537, 33, 8191], 64), ([5, 3, 2], 8),
                                            (list(I.LAYER_D1024.numel), 8)],
                         ids=["tiny", "5p-N3", "3p-N64", "pad-only", "d1024"])
def test_step_layer_writes_grad_shards(z3mod, orc, numel, n_ranks):
    """z3_step_layer with grad_shards_or_NULL set: the reduced fp32 gradient
    slices it stores equal the oracle's reduce-scatter output bit for bit
    (pad 0), and the updated state equals the oracle's step as with NULL."""
    c = Case(z3mod, orc, numel, n_ranks, seed=5)
    gs = Guarded(c.L.psi_padded, torch.float32, fill=float("nan"))
    c.bufs.append(gs)
    for step in (1, 2, 3):
        g, gh = c.grads()
        z3mod.z3_step_layer(c.L, c.shards.t, c.gathered.t, g, c.stride, 1.0 / n_ranks,
                            c.master.t, c.m.t, c.v.t, HP, step, grad_shards=gs.t)
        _, fb, want_gs = orc.step_layer(c.O, c.o["shards"], gh, c.stride, 1.0 / n_ranks,
                                        c.o["master"], c.o["m"], c.o["v"], HP, step)
        got = c.device_state()
        assert np.array_equal(bits32(f32(gs.t)), bits32(want_gs))
        assert np.array_equal(u16(c.gathered.t), fb)
        assert_adam_equal(got, c.o)
    assert c.guards_ok()


def test_weight_decay_and_other_hparams(z3mod, orc):
    hp = dict(lr=3e-4, beta1=0.8, beta2=0.95, eps=1e-6, weight_decay=0.1)
    c = Case(z3mod, orc, [4099, 77, 1024], 8, seed=3, grad_std=1.0)
    for step in (1, 2, 7):
        g, gh = c.grads()
        z3mod.z3_step_layer(c.L, c.shards.t, c.gathered.t, g, c.stride, 0.5, c.master.t,
                            c.m.t, c.v.t, hp, step)
        orc.step_layer(c.O, c.o["shards"], gh, c.stride, 0.5, c.o["master"], c.o["m"],
                       c.o["v"], hp, step)
        assert_adam_equal(c.device_state(), c.o)
    assert c.guards_ok()


def test_rejects_bad_arguments_on_device(z3mod):
    """Overlap is rejected with real buffers too (had the check slipped, the
    gather would have stayed inside its own buffer).  Misaligned pointers are
    checked in tests/test_abi.py, in a process that sees no device, since a
    16-byte access at a misaligned address would fault."""
    L = z3mod.Layout([100, 28], 4)
    sh = torch.zeros(L.psi_padded, dtype=torch.bfloat16, device="cuda")
    full = torch.zeros(L.psi, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(z3mod.Z3Error) as e:
        z3mod.z3_allgather(L, sh, sh)          # in place: overlapping buffers
    assert e.value.status == z3mod.Z3_ERR_INVALID_ARG
    z3mod.z3_allgather(L, sh, full)
    torch.cuda.synchronize()


def _fuzz_layouts(n=24, seed=123):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        P = int(rng.integers(1, 61))
        kind = rng.integers(0, 3, size=P)
        sizes = np.where(kind == 0, rng.integers(0, 40, size=P),
                         np.where(kind == 1, rng.integers(0, 5000, size=P),
                                  rng.integers(0, 60000, size=P)))
        N = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 64, 100]))
        out.append(([int(x) for x in sizes], N))
    return out


FUZZ = _fuzz_layouts()


@pytest.mark.parametrize("numel,n_ranks", FUZZ, ids=[f"fuzz{i}" for i in range(len(FUZZ))])
def test_all_calls_fuzzed_layouts(z3mod, orc, numel, n_ranks):
    """Seeded random layouts (empty, tiny and large parameters, up to 60 of
    them, rank counts up to 100): every call bit-exact against the oracle."""
    if sum(numel) == 0:
        numel = numel + [1]
    run_all_calls(z3mod, orc, numel, n_ranks, seed=5, steps=1)


def test_wide_gradient_pitch_and_late_steps(z3mod, orc):
    """Rank rows further apart than required (pitch 96 elements beyond Psi,
    a multiple of 8) and step counts where the bias corrections round to 1."""
    numel, N = [4099, 77, 1024, 13], 8
    c = Case(z3mod, orc, numel, N, seed=17)
    stride = c.w.grad_stride + 96
    for step in (1, 1000, 10 ** 6):
        g = I.draw_grads(c.w, c.gen, "cuda")
        wide = torch.zeros((N, stride), dtype=torch.bfloat16, device="cuda")
        wide[:, :c.L.psi].copy_(g[:, :c.L.psi])
        wide[:, c.L.psi:].fill_(float("nan"))        # never read
        z3mod.z3_step_layer(c.L, c.shards.t, c.gathered.t, wide, stride, 1.0 / N, c.master.t,
                            c.m.t, c.v.t, HP, step)
        orc.step_layer(c.O, c.o["shards"], u16(wide).reshape(-1), stride, 1.0 / N,
                       c.o["master"], c.o["m"], c.o["v"], HP, step)
        assert_adam_equal(c.device_state(), c.o)
    k = orc.adam_constants(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], 0.0, 10 ** 6)
    assert k["rb1"] == 1.0 and k["rb2"] == 1.0
    assert c.guards_ok()


@pytest.mark.parametrize("depth", [0, 1, 2])
def test_model_step_matches_oracle(z3mod, orc, depth):
    """z3_model_step over four units (one resident, odd lengths, N_d = 5),
    three steps, with 0, 1 and 2 units of gather prefetch: every unit's
    state equals the oracle's layer step bit for bit, the resident copy
    equals the oracle's gather of the updated shards, each transient buffer
    holds the backward gather of the last unit that used it, and no call
    writes outside its buffers."""
    N = 5
    specs = [([77, 1024, 5], True), ([100003, 7], False), ([4099, 65536, 1], False),
             ([262147], False)]
    cases = [Case(z3mod, orc, numel, N, seed=40 + i) for i, (numel, _) in enumerate(specs)]
    resident = [Guarded(c.L.psi, torch.bfloat16) if res else None
                for c, (_, res) in zip(cases, specs)]
    for c, r in zip(cases, resident):
        if r is not None:
            z3mod.z3_allgather(c.L, c.shards.t, r.t)
    nb = depth + 1
    big = max(c.L.psi for c, (_, res) in zip(cases, specs) if not res)
    fulls = [Guarded(big, torch.bfloat16) for _ in range(nb)]
    gstream = torch.cuda.Stream() if depth else None
    scale = 1.0 / N
    for t in (1, 2, 3):
        drawn = [c.grads() for c in cases]
        units = [(c.L, c.shards.t, c.master.t, c.m.t, c.v.t, g, c.stride, scale,
                  None if r is None else r.t) for c, (g, _), r in zip(cases, drawn, resident)]
        z3mod.z3_model_step(units, [f.t for f in fulls], HP, t, gather_stream=gstream)
        last_bwd = {}
        for i in range(len(cases) - 1, -1, -1):      # backward order
            c, (_, gh) = cases[i], drawn[i]
            _, fb, _ = orc.step_layer(c.O, c.o["shards"], gh, c.stride, scale, c.o["master"],
                                      c.o["m"], c.o["v"], HP, t)
            if resident[i] is None:
                last_bwd[i % nb] = fb
        torch.cuda.synchronize()
        for c in cases:
            assert_adam_equal(c.device_state(), c.o)
            assert c.guards_ok()
        for c, r in zip(cases, resident):
            if r is not None:
                assert np.array_equal(u16(r.t), orc.allgather(c.O, c.o["shards"]))
                assert r.guards_intact()
        for b, fb in last_bwd.items():
            assert np.array_equal(u16(fulls[b].t)[:fb.size], fb), f"buffer {b}"
        assert all(f.guards_intact() for f in fulls)


def _fuzz_model_configs(n=12, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        N = int(rng.choice([1, 2, 3, 5, 8, 16]))
        units = []
        for _ in range(int(rng.integers(1, 7))):
            numel = [int(x) for x in rng.integers(0, 20000, size=int(rng.integers(1, 9)))]
            if rng.random() < 0.2:
                numel[0] = 0
            units.append((numel, bool(rng.random() < 0.25)))
        out.append((N, units, int(rng.integers(0, 4))))
    return out


@pytest.mark.parametrize("N,specs,depth", _fuzz_model_configs())
def test_model_step_fuzzed(z3mod, orc, N, specs, depth):
    """Seeded random models through z3_model_step: 1-6 units of 1-8
    parameters (empty ones included), some resident, N_d from 1 to 16,
    prefetch depth 0-3; two steps against the oracle's layer step, bit for
    bit, with guard words around every buffer."""
    if all(res for _, res in specs):
        specs = [(specs[0][0], False)] + list(specs[1:])
    cases = [Case(z3mod, orc, numel, N, seed=300 + i) for i, (numel, _) in enumerate(specs)]
    resident = [Guarded(max(c.L.psi, 1), torch.bfloat16) if res else None
                for c, (_, res) in zip(cases, specs)]
    for c, r in zip(cases, resident):
        if r is not None:
            z3mod.z3_allgather(c.L, c.shards.t, r.t)
    big = max([c.L.psi for c, (_, res) in zip(cases, specs) if not res] + [1])
    fulls = [Guarded(big, torch.bfloat16) for _ in range(depth + 1)]
    gstream = torch.cuda.Stream() if depth else None
    for t in (1, 2):
        drawn = [c.grads() for c in cases]
        units = [(c.L, c.shards.t, c.master.t, c.m.t, c.v.t, g, c.stride, 1.0 / N,
                  None if r is None else r.t) for c, (g, _), r in zip(cases, drawn, resident)]
        z3mod.z3_model_step(units, [f.t for f in fulls], HP, t, gather_stream=gstream)
        for c, (_, gh) in zip(cases, drawn):
            orc.step_layer(c.O, c.o["shards"], gh, c.stride, 1.0 / N, c.o["master"], c.o["m"],
                           c.o["v"], HP, t)
        torch.cuda.synchronize()
        for c, r in zip(cases, resident):
            assert_adam_equal(c.device_state(), c.o)
            assert c.guards_ok()
            if r is not None:
                assert np.array_equal(u16(r.t)[:c.L.psi], orc.allgather(c.O, c.o["shards"]))
                assert r.guards_intact()
        assert all(f.guards_intact() for f in fulls)


@pytest.mark.parametrize("depth", [0, 1])
def test_model_step_per_unit_hyperparameters(z3mod, orc, depth):
    """Units with their own hyperparameters (a parameter group without weight
    decay, one with another learning rate) next to units that use the
    step's: every unit equals the oracle's layer step with its own
    hyperparameters, bit for bit."""
    N = 4
    step_hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    own = [dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0), None,
           dict(lr=3e-3, beta1=0.8, beta2=0.99, eps=1e-6, weight_decay=0.05), None]
    specs = [[77, 1024], [100003, 7], [4099, 65536], [262147]]
    cases = [Case(z3mod, orc, numel, N, seed=500 + i) for i, numel in enumerate(specs)]
    big = max(c.L.psi for c in cases)
    fulls = [Guarded(big, torch.bfloat16) for _ in range(depth + 1)]
    gstream = torch.cuda.Stream() if depth else None
    for t in (1, 2, 3):
        drawn = [c.grads() for c in cases]
        units = [(c.L, c.shards.t, c.master.t, c.m.t, c.v.t, g, c.stride, 1.0 / N, None, h)
                 for c, (g, _), h in zip(cases, drawn, own)]
        z3mod.z3_model_step(units, [f.t for f in fulls], step_hp, t, gather_stream=gstream)
        for c, (_, gh), h in zip(cases, drawn, own):
            orc.step_layer(c.O, c.o["shards"], gh, c.stride, 1.0 / N, c.o["master"], c.o["m"],
                           c.o["v"], h or step_hp, t)
        torch.cuda.synchronize()
        for c in cases:
            assert_adam_equal(c.device_state(), c.o)
            assert c.guards_ok()
