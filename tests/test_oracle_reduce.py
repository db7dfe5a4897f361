"""Oracle pins: reduce-scatter, all-reduce identity, micro-batch accumulation.

Pins: hand-derived fold cases (tests/golden/rs_fold_cases.json), exact
integer-valued sums against torch.sum, the recursive-summation error bound
against an fp64 sum, and the reduce-scatter + all-gather = all-reduce
identity ('ZeRO Stages: ...', 'Stage 2 also partitions gradients').
"""
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _grads(rank_rows: list, stride: int) -> np.ndarray:
    g = np.zeros((len(rank_rows), stride), np.uint16)
    for k, row in enumerate(rank_rows):
        g[k, :len(row)] = _bf16_bits(np.asarray(row, np.float32))
    return g.reshape(-1)


def test_golden_fold_cases(orc):
    cases = json.load(open(os.path.join(GOLDEN, "rs_fold_cases.json")))["cases"]
    for c in cases:
        n_ranks = len(c["ranks"])
        L = orc.layout([1], n_ranks)          # one element, owned by rank 0
        g = _grads([[x] for x in c["ranks"]], 8)
        assert np.array_equal(orc.f32_from_bf16(g.reshape(n_ranks, 8)[:, 0]),
                              np.asarray(c["ranks"], np.float32)), "inputs must be bf16-exact"
        out = orc.reduce_scatter(L, g, 8, c["scale"])
        if "expected_bits" in c:
            assert int(out[:1].view(np.uint32)[0]) == c["expected_bits"], c["name"]
        else:
            assert out[0] == np.float32(c["expected"]), (c["name"], out[0])
        assert not out[1:].any()               # the pad of ranks 1.. is zero
        # the all-reduce uses the same fold
        ar = orc.allreduce(L, g, 8, c["scale"])
        assert ar.view(np.uint32)[0] == out.view(np.uint32)[0]


def _layout_reference(L, full_vals: np.ndarray) -> np.ndarray:
    """Shard-space image [N*S] of a full-space vector, built with numpy
    reshapes (pad zero)."""
    out = np.zeros(L.psi_padded, full_vals.dtype)
    mat = out.reshape(L.n_ranks, L.S)
    for p in range(L.n_params):
        o, s, n, F = (int(L.shard_off[p]), int(L.shard_numel[p]), int(L.numel[p]),
                      int(L.full_off[p]))
        padded = np.zeros(s * L.n_ranks, full_vals.dtype)
        padded[:n] = full_vals[F:F + n]
        mat[:, o:o + s] = padded.reshape(L.n_ranks, s)
    return out


@pytest.mark.parametrize("n_ranks", [1, 2, 3, 5, 8, 16, 64])
def test_integer_grads_equal_torch_sum(orc, n_ranks):
    """Integer-valued grads in [-8, 8]: every partial sum is exact, so the
    result is order-free and equals torch.sum; a power-of-two 1/N scale is
    exact too."""
    rng = np.random.default_rng(10 + n_ranks)
    numel = [37, 11, 1, 0, 97, 13]
    L = orc.layout(numel, n_ranks)
    stride = L.psi + 5
    vals = rng.integers(-8, 9, size=(n_ranks, L.psi)).astype(np.float32)
    g = _grads(list(vals), stride)
    scale = 1.0 / n_ranks if (n_ranks & (n_ranks - 1)) == 0 else 1.0
    out = orc.reduce_scatter(L, g, stride, scale)
    want_full = (torch.from_numpy(vals).sum(dim=0) * scale).numpy()
    assert np.array_equal(out, _layout_reference(L, want_full))


@pytest.mark.parametrize("n_ranks", [2, 3, 8, 64])
def test_float_grads_within_summation_bound(orc, n_ranks):
    """Random bf16 grads: |fold - exact| <= (N-1) u sum|g| plus the final
    rounding of the scaled value (u = 2^-24); a dropped term, a wrong sign or
    a wrong index fails by far more."""
    rng = np.random.default_rng(20 + n_ranks)
    numel = [101, 7, 64, 3]
    L = orc.layout(numel, n_ranks)
    stride = L.psi + (-L.psi) % 8
    raw = rng.standard_normal((n_ranks, L.psi)).astype(np.float32)
    g = _grads(list(raw), stride)
    vals = orc.f32_from_bf16(g.reshape(n_ranks, stride)[:, :L.psi]).astype(np.float64)
    scale = np.float32(1.0 / n_ranks)
    out = orc.reduce_scatter(L, g, stride, float(scale))
    exact = vals.sum(axis=0) * np.float64(scale)
    bound = ((n_ranks - 1) * 2.0 ** -24 * np.abs(vals).sum(axis=0) * float(scale)
             + 2.0 ** -24 * np.abs(exact) + 1e-45)
    got = orc.allgather_f32(L, out).astype(np.float64)
    assert np.all(np.abs(got - exact) <= bound * 1.0001)
    # pad positions are zero
    ref_mask = _layout_reference(L, np.ones(L.psi, np.float32))
    assert not out[ref_mask == 0].any()


@pytest.mark.parametrize("n_ranks", [1, 2, 4, 7, 8, 64])
def test_reduce_scatter_then_allgather_is_allreduce(orc, n_ranks):
    rng = np.random.default_rng(30 + n_ranks)
    numel = [int(x) for x in rng.integers(1, 300, size=4)]
    L = orc.layout(numel, n_ranks)
    stride = L.psi + (-L.psi) % 8
    g = _grads(list(rng.standard_normal((n_ranks, L.psi)).astype(np.float32)), stride)
    scale = 1.0 / n_ranks
    rs = orc.reduce_scatter(L, g, stride, scale)
    ar = orc.allreduce(L, g, stride, scale)
    assert np.array_equal(orc.allgather_f32(L, rs).view(np.uint32), ar.view(np.uint32))


def test_brute_force_tiny_primes(orc):
    """Prime lengths, every owned element checked against an fp64 sum of
    integer-valued grads (exact), mapped with numpy's split of the padded
    buffer."""
    rng = np.random.default_rng(40)
    for n in (2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37, 41, 43, 47):
        for n_ranks in (2, 3, 5, 8):
            L = orc.layout([n], n_ranks)
            vals = rng.integers(-4, 5, size=(n_ranks, n)).astype(np.float32)
            g = _grads(list(vals), n + 8)
            out = orc.reduce_scatter(L, g, n + 8, 1.0)
            pad = (-n) % n_ranks
            ref = np.split(np.concatenate([vals.astype(np.float64).sum(0), np.zeros(pad)]),
                           n_ranks)
            assert np.array_equal(out.astype(np.float64), np.concatenate(ref))


def test_micro_batch_accumulation(orc):
    """'ZeRO Stages: ...', second subtlety of stage 2: reduce each
    micro-batch, accumulate the reduced slices in fp32."""
    rng = np.random.default_rng(50)
    numel = [131, 7, 1]
    n_ranks = 8
    L = orc.layout(numel, n_ranks)
    stride = L.psi + (-L.psi) % 8
    mbs = [_grads(list(rng.standard_normal((n_ranks, L.psi)).astype(np.float32)), stride)
           for _ in range(4)]
    acc = orc.reduce_scatter(L, mbs[0], stride, 1.0 / n_ranks)
    singles = [acc.copy()]
    for g in mbs[1:]:
        singles.append(orc.reduce_scatter(L, g, stride, 1.0 / n_ranks))
        orc.reduce_scatter(L, g, stride, 1.0 / n_ranks, out=acc, accumulate=True)
    want = singles[0]
    for s in singles[1:]:
        want = (want + s).astype(np.float32)     # fp32 add, in micro-batch order
    assert np.array_equal(acc.view(np.uint32), want.view(np.uint32))
    ref_mask = _layout_reference(L, np.ones(L.psi, np.float32))
    assert not acc[ref_mask == 0].any()
