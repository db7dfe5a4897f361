"""Oracle pins: the sharded Adam update and the layer step.

Pins: torch.optim.Adam / AdamW on the CPU (an independent implementation of
Kingma & Ba, Algorithm 1, with different rounding order) within 1e-6
relative; the t = 1 closed form in fp64; the data-parallel-semantics claim
of 'The ZeRO-3 Diagram Most People Remember Is Wrong', s.4 (one sharded step
equals one unsharded data-parallel step, bit-exact); pad positions stay 0.
"""
import numpy as np
import pytest
import torch

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)


def _close(a, b, rtol, atol):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.all(np.abs(a - b) <= np.maximum(rtol * np.abs(b), atol))


@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_against_torch_adam(orc, wd):
    rng = np.random.default_rng(60)
    n = 4099
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    master, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    bf = np.zeros(n, np.uint16)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    cls = torch.optim.AdamW if wd else torch.optim.Adam
    opt = cls([tp], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
              weight_decay=wd, foreach=False, fused=False)
    u = 2.0 ** -24
    m_tol = np.zeros(n)
    v_tol = np.zeros(n)
    for step in range(1, 6):
        g = rng.standard_normal(n).astype(np.float32) * (1.0 if step % 2 else 1e-3)
        g64 = np.abs(g.astype(np.float64))
        # each two-term moment update rounds to within a few u of its terms'
        # magnitudes, and earlier differences decay by beta (torch forms m
        # with lerp, so its rounding differs from ours)
        m_tol = 0.9 * m_tol + 8 * u * (np.abs(m.astype(np.float64)) + g64)
        v_tol = 0.999 * v_tol + 8 * u * (np.abs(v.astype(np.float64)) + g64 * g64)
        orc.adam(master, m, v, g, bf, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], wd, step)
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
        st = opt.state[tp]
        assert _close(master, tp.detach().numpy(), 1e-6, 1e-9)
        assert _close(m, st["exp_avg"].numpy(), 1e-6, m_tol)
        assert _close(v, st["exp_avg_sq"].numpy(), 1e-6, v_tol)
    # the bf16 copy is the RNE cast of the master
    want = torch.from_numpy(master).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf, want)


def test_first_step_closed_form(orc):
    """t = 1: m_hat = g and v_hat = g^2 up to rounding, so
    p1 = p0 - lr * g / (|g| + eps)."""
    rng = np.random.default_rng(61)
    n = 10000
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * np.exp(rng.uniform(-12, 3, n))).astype(np.float32)
    master, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    bf = np.zeros(n, np.uint16)
    orc.adam(master, m, v, g, bf, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], 0.0, 1)
    g64 = g.astype(np.float64)
    p1 = p0.astype(np.float64) - HP["lr"] * g64 / (np.abs(g64) + HP["eps"])
    assert _close(master, p1, 1e-6, 1e-9)
    assert _close(m, (1 - 0.9) * g64, 1e-6, 0)
    assert _close(v, (1 - 0.999) * g64 * g64, 1e-6, 0)


def test_zero_gradient_keeps_zero_state(orc):
    n = 64
    z = np.zeros(n, np.float32)
    master, m, v, bf = z.copy(), z.copy(), z.copy(), np.ones(n, np.uint16)
    for step in (1, 2, 3):
        orc.adam(master, m, v, z, bf, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], 0.01, step)
    assert not master.view(np.uint32).any() and not m.any() and not v.any() and not bf.any()


def test_constants_are_rounded_once(orc):
    """Each binary32 constant is the real-valued quantity rounded once; in
    particular 1 - beta2 is not formed from an already-rounded beta2."""
    for step in (1, 2, 10, 1000):
        k = orc.adam_constants(1e-3, 0.9, 0.999, 1e-8, 0.1, step)
        assert k["rb1"] == np.float32(1 / (1 - 0.9 ** step))
        assert k["rb2"] == np.float32(1 / (1 - 0.999 ** step))
        assert k["c2"] == np.float32(0.001) and k["c2"] != np.float32(1) - np.float32(0.999)
        assert k["lwd"] == np.float32(1e-4)
    with pytest.raises(ValueError):
        orc.adam(*(np.zeros(1, np.float32) for _ in range(4)), np.zeros(1, np.uint16),
                 1e-3, 0.9, 0.999, 1e-8, 0.0, 0)


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("n_ranks,numel", [(4, [35, 13, 12]), (3, [101, 7, 1, 64]),
                                           (8, [257, 33]), (64, [1000, 3])])
def test_sharded_step_equals_unsharded_dp_step(orc, n_ranks, numel):
    """Three sharded layer steps (AG, AG, RS, shard Adam) against three
    unsharded data-parallel steps (all-reduce mean, Adam on the whole tensor):
    masters, moments and bf16 params identical bit for bit."""
    rng = np.random.default_rng(70 + n_ranks)
    L = orc.layout(numel, n_ranks)
    stride = L.psi + (-L.psi) % 8
    full = (rng.standard_normal(L.psi) * 0.02).astype(np.float32)
    sh, ma, m, v = orc.partition(L, full)
    dp_p, dp_m, dp_v = full.copy(), np.zeros(L.psi, np.float32), np.zeros(L.psi, np.float32)
    dp_bf = _bf16_bits(full)
    for step in (1, 2, 3):
        g = np.zeros((n_ranks, stride), np.uint16)
        g[:, :L.psi] = _bf16_bits(rng.standard_normal((n_ranks, L.psi)).astype(np.float32))
        g = g.reshape(-1)
        before = orc.allgather(L, sh)
        ff, fb, gs = orc.step_layer(L, sh, g, stride, 1.0 / n_ranks, ma, m, v, HP, step)
        # both gathers see the parameters of the previous step
        assert np.array_equal(ff, before) and np.array_equal(fb, before)
        assert np.array_equal(ff, dp_bf)
        dg = orc.allreduce(L, g, stride, 1.0 / n_ranks)
        orc.adam(dp_p, dp_m, dp_v, dg, dp_bf, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"],
                 HP["weight_decay"], step)
        assert np.array_equal(orc.allgather_f32(L, ma).view(np.uint32), dp_p.view(np.uint32))
        assert np.array_equal(orc.allgather_f32(L, m).view(np.uint32), dp_m.view(np.uint32))
        assert np.array_equal(orc.allgather_f32(L, v).view(np.uint32), dp_v.view(np.uint32))
        assert np.array_equal(orc.allgather(L, sh), dp_bf)
        # pad positions stay zero in every buffer
        pad = np.ones(L.psi_padded, bool)
        pad[np.flatnonzero(orc.partition(L, np.ones(L.psi, np.float32))[1])] = False
        for buf in (ma, m, v, gs):
            assert not buf[pad].any()
        assert not sh[pad].any()


def test_step_with_accumulated_micro_batches(orc):
    """The reduced gradient of the last micro-batch is added to the running
    fp32 sums before Adam; equals reduce (accumulate) then Adam."""
    rng = np.random.default_rng(80)
    n_ranks, numel = 8, [131, 7]
    L = orc.layout(numel, n_ranks)
    stride = L.psi + (-L.psi) % 8
    full = (rng.standard_normal(L.psi) * 0.02).astype(np.float32)
    sh, ma, m, v = orc.partition(L, full)
    sh2, ma2, m2, v2 = (a.copy() for a in (sh, ma, m, v))
    gs = [np.zeros((n_ranks, stride), np.uint16) for _ in range(4)]
    for g in gs:
        g[:, :L.psi] = _bf16_bits(rng.standard_normal((n_ranks, L.psi)).astype(np.float32))
    gs = [g.reshape(-1) for g in gs]
    acc = orc.reduce_scatter(L, gs[0], stride, 0.125)
    for g in gs[1:3]:
        orc.reduce_scatter(L, g, stride, 0.125, out=acc, accumulate=True)
    _, _, red = orc.step_layer(L, sh, gs[3], stride, 0.125, ma, m, v, HP, 1, grad_acc=acc)
    acc2 = acc.copy()
    orc.reduce_scatter(L, gs[3], stride, 0.125, out=acc2, accumulate=True)
    assert np.array_equal(red.view(np.uint32), acc2.view(np.uint32))
    orc.adam(ma2, m2, v2, acc2, sh2, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], 0.0, 1)
    assert np.array_equal(ma.view(np.uint32), ma2.view(np.uint32))
    assert np.array_equal(sh, sh2)
