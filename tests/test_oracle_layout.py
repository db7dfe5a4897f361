"""Oracle pins: layout, partition and all-gather (CPU only).

The layout is checked against numpy's own contiguous equal split of the
padded flat buffer (``np.split``), not against a retyped formula; the gather
against a reshape of the [N][s_p] block; the Tiny layout against a golden file
derived by hand from the partition steps.
"""
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RANKS = list(range(1, 10)) + [16, 64]


def _split_reference(values: np.ndarray, n_ranks: int):
    """Flatten -> pad with zeros to the next multiple of N -> N equal
    contiguous pieces, using numpy's split (independent of the oracle)."""
    pad = (-values.size) % n_ranks
    padded = np.concatenate([values, np.zeros(pad, values.dtype)])
    return np.split(padded, n_ranks), pad


@pytest.mark.parametrize("n_ranks", RANKS)
def test_single_param_bruteforce(orc, n_ranks):
    for n in range(0, 301):
        L = orc.layout([n], n_ranks)
        pieces, pad = _split_reference(np.arange(1, n + 1, dtype=np.float32), n_ranks)
        # minimal pad: fewer than N pad elements, and s * N covers n
        assert L.psi_padded - n == pad and pad < n_ranks
        assert L.S == (pieces[0].size if n_ranks else 0)
        full = np.arange(1, n + 1, dtype=np.float32)
        sh, ma, m, v = orc.partition(L, full)
        for r in range(n_ranks):
            got = ma[r * L.S:(r + 1) * L.S]
            assert np.array_equal(got, pieces[r]), (n, n_ranks, r)
        # each original element appears exactly once among the shards
        nz = ma[ma != 0]
        assert np.array_equal(np.sort(nz), full)
        assert not m.any() and not v.any()


def test_multi_param_concatenation(orc):
    rng = np.random.default_rng(1)
    for trial in range(60):
        n_ranks = int(rng.choice(RANKS))
        numel = [int(x) for x in rng.integers(0, 200, size=int(rng.integers(1, 7)))]
        L = orc.layout(numel, n_ranks)
        full = rng.standard_normal(sum(numel)).astype(np.float32)
        sh, ma, m, v = orc.partition(L, full)
        # reference: per parameter split, then rank r's shard is the
        # concatenation of its pieces in parameter order
        splits = []
        off = 0
        for n in numel:
            splits.append(_split_reference(full[off:off + n], n_ranks)[0])
            off += n
        for r in range(n_ranks):
            ref = np.concatenate([s[r] for s in splits])
            assert np.array_equal(ma[r * L.S:(r + 1) * L.S], ref)
        assert L.psi_padded == sum(s[0].size for s in splits) * n_ranks


def test_tiny_golden(orc):
    g = json.load(open(os.path.join(GOLDEN, "tiny_layout.json")))
    L = orc.layout(g["numel"], g["n_ranks"])
    assert list(L.shard_numel) == g["shard_numel"]
    assert list(L.shard_off) == g["shard_off"]
    assert list(L.full_off) == g["full_off"]
    assert (L.S, L.psi, L.psi_padded) == (g["S"], g["psi"], g["psi_padded"])
    assert [int(s) * g["n_ranks"] - int(n) for s, n in zip(L.shard_numel, L.numel)] == g["pad"]
    # owning rank of selected elements: place a marker and find it
    for p, table in enumerate([g["rank_of_element"][k] for k in ("p0", "p1", "p2")]):
        for idx, rank in table.items():
            full = np.zeros(L.psi, np.float32)
            full[L.full_off[p] + int(idx)] = 1.0
            _, ma, _, _ = orc.partition(L, full)
            hit = int(np.flatnonzero(ma)[0])
            assert hit // L.S == rank


def test_layout_rejects_bad_arguments(orc):
    with pytest.raises(ValueError):
        orc.layout([5], 0)
    with pytest.raises(ValueError):
        orc.layout([-1], 4)


def test_partition_pad_is_zero_and_bf16_is_torch_rne(orc):
    rng = np.random.default_rng(2)
    numel = [7, 1, 0, 13, 64, 3]
    for n_ranks in (3, 4, 8, 64):
        L = orc.layout(numel, n_ranks)
        full = (rng.standard_normal(L.psi) * 0.02).astype(np.float32)
        sh, ma, m, v = orc.partition(L, full)
        # every pad position is zero in all four buffers
        pad_mask = np.ones(L.psi_padded, bool)
        for p in range(L.n_params):
            s, o, n = int(L.shard_numel[p]), int(L.shard_off[p]), int(L.numel[p])
            for r in range(n_ranks):
                valid = max(0, min(s, n - r * s))
                pad_mask[r * L.S + o: r * L.S + o + valid] = False
        assert not ma[pad_mask].any() and not sh[pad_mask].any()
        # the bf16 shard equals torch's round-to-nearest-even cast of the master
        ref = torch.from_numpy(ma).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(sh, ref)


@pytest.mark.parametrize("n_ranks", [1, 2, 3, 4, 7, 8, 16, 64])
def test_allgather_round_trip_and_reshape(orc, n_ranks):
    rng = np.random.default_rng(3)
    numel = [int(x) for x in rng.integers(0, 500, size=5)] + [1, 2, 129]
    L = orc.layout(numel, n_ranks)
    full = rng.standard_normal(L.psi).astype(np.float32)
    sh, ma, _, _ = orc.partition(L, full)
    got = orc.allgather(L, sh)
    # round trip: AG(partition(x)) == bf16(x) bit-exact, torch's cast as reference
    want = torch.from_numpy(full).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    # independent formulation: parameter p is the row-major flatten of the
    # [N, s_p] block of the shard matrix, truncated to n_p
    mat = sh.reshape(n_ranks, L.S)
    for p in range(L.n_params):
        o, s, n, F = (int(L.shard_off[p]), int(L.shard_numel[p]), int(L.numel[p]),
                      int(L.full_off[p]))
        assert np.array_equal(got[F:F + n], mat[:, o:o + s].reshape(-1)[:n])
    # fp32 gather of the master gives the exact input back
    assert np.array_equal(orc.allgather_f32(L, ma), full)


def test_single_rank_is_identity(orc):
    rng = np.random.default_rng(4)
    numel = [5, 17, 3]
    L = orc.layout(numel, 1)
    assert L.S == L.psi == L.psi_padded == 25
    full = rng.standard_normal(L.psi).astype(np.float32)
    sh, ma, _, _ = orc.partition(L, full)
    assert np.array_equal(ma, full)
    assert np.array_equal(orc.allgather(L, sh), sh)
