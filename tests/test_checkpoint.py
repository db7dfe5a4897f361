"""Per-rank shard-set checkpoints on the CPU: the file format round-trips,
a missing rank file is reported as that rank's lost slice, corruption and
truncation are detected ('ZeRO Stages: ...', 'Where the shards live and what
happens on failure')."""
import os

import numpy as np
import pytest

from optimizer_state_gb300 import checkpoint as ck


def _state(orc, numel, n_ranks, seed=0):
    rng = np.random.default_rng(seed)
    L = orc.layout(numel, n_ranks)
    full = rng.standard_normal(L.psi).astype(np.float32)
    sh, ma, m, v = orc.partition(L, full)
    m[:] = rng.standard_normal(m.size).astype(np.float32) * (ma != 0)
    return L, dict(shards=sh, master=ma, m=m, v=v)


def test_round_trip(orc, tmp_path):
    L, arrays = _state(orc, [35, 13, 12], 4)
    ck.write_host(str(tmp_path), L.numel, 4, L.S, 7, arrays)
    assert sorted(os.listdir(tmp_path)) == ["meta.json"] + [ck.rank_file(r) for r in range(4)]
    meta, back = ck.read_host(str(tmp_path))
    assert meta["step"] == 7 and meta["n_ranks"] == 4 and meta["S"] == 16
    for k in arrays:
        assert np.array_equal(back[k].view(np.uint8), arrays[k].view(np.uint8))
    # each rank file holds exactly that rank's slices: 14 bytes per element
    assert os.path.getsize(tmp_path / ck.rank_file(0)) == 14 * L.S


def test_lost_rank_is_reported(orc, tmp_path):
    L, arrays = _state(orc, [101, 7], 8)
    ck.write_host(str(tmp_path), L.numel, 8, L.S, 1, arrays)
    os.remove(tmp_path / ck.rank_file(5))
    with pytest.raises(ck.CheckpointError, match=r"rank\(s\) \[5\]"):
        ck.read_host(str(tmp_path))


def test_corruption_and_truncation_detected(orc, tmp_path):
    L, arrays = _state(orc, [101, 7], 3)
    ck.write_host(str(tmp_path), L.numel, 3, L.S, 1, arrays)
    p = tmp_path / ck.rank_file(1)
    raw = bytearray(p.read_bytes())
    raw[10] ^= 0xFF
    p.write_bytes(bytes(raw))
    with pytest.raises(ck.CheckpointError, match="checksum"):
        ck.read_host(str(tmp_path))
    with pytest.raises(ck.CheckpointError, match="metadata"):
        ck.read_host(str(tmp_path / "nowhere"))


def test_model_metadata_checks(tmp_path):
    """load_model refuses a missing or foreign model file, another unit count
    and other parameters before it touches any device buffer."""
    import json
    from types import SimpleNamespace as NS

    def fake_model(numels):
        return NS(units=[NS(L=NS(numel=n, n_ranks=4)) for n in numels], t=0)
    d = tmp_path / "m"
    with pytest.raises(ck.CheckpointError, match="no model metadata"):
        ck.load_model(str(d), fake_model([[5, 3]]))
    d.mkdir()
    (d / "model.json").write_text(json.dumps({"format": "other", "units": []}))
    with pytest.raises(ck.CheckpointError, match="unknown model checkpoint format"):
        ck.load_model(str(d), fake_model([[5, 3]]))
    units = [{"dir": "unit000", "name": "a", "numel": [5, 3], "resident": False}]
    (d / "model.json").write_text(json.dumps({"format": ck.MODEL_FORMAT, "step": 3,
                                              "units": units}))
    with pytest.raises(ck.CheckpointError, match="units"):
        ck.load_model(str(d), fake_model([[5, 3], [7]]))
    with pytest.raises(ck.CheckpointError, match="parameters differ"):
        ck.load_model(str(d), fake_model([[5, 4]]))
