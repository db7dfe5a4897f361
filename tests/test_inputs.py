"""The full-step unit plans (host logic only): buckets of consecutive layers
and the persistence threshold regroup parameters, never drop or repeat one,
and keep every parameter's shape."""
import math

import pytest

from optimizer_state_gb300 import inputs as I

N_PARAMS = 1 + 24 * 6          # the embedding, then 6 parameters per layer


@pytest.mark.parametrize("bucket", [1, 2, 4, 5, 6, 24])
@pytest.mark.parametrize("threshold", [0, 1024, 1025, 100000, 4194305, 10 ** 9])
def test_every_parameter_in_exactly_one_unit(bucket, threshold):
    ids = I.full_step_param_ids(bucket, threshold)
    flat = [i for u in ids for i in u]
    assert sorted(flat) == list(range(N_PARAMS))
    units = I.full_step_units(bucket, threshold)
    assert len(units) == len(ids)
    shapes = I._full_step_shapes()
    for w, u in zip(units, ids):
        assert w.shapes == tuple(shapes[i] for i in u)
        assert list(u) == sorted(u)                      # model order inside a unit
        assert w.n_ranks == 16
    assert sum(w.psi for w in units) == 353502208
    small = [i for i in range(N_PARAMS) if math.prod(shapes[i]) < threshold]
    if small:
        assert units[0].resident and list(ids[0]) == small
        assert not any(w.resident for w in units[1:])
        assert all(math.prod(shapes[i]) >= threshold for u in ids[1:] for i in u)
    else:
        assert not any(w.resident for w in units)


def test_plain_buckets():
    units = I.full_step_units(1)
    assert [w.name for w in units[:3]] == ["embed", "layers0-0", "layers1-1"]
    assert len(units) == 25
    units = I.full_step_units(5)
    assert [w.name for w in units] == ["embed", "layers0-4", "layers5-9", "layers10-14",
                                       "layers15-19", "layers20-23"]


def test_norm_gains_become_resident():
    """A threshold between the norm gains (1024 elements) and the smallest
    matrix (1024 x 1024) moves exactly the 48 gain vectors."""
    units = I.full_step_units(4, 100000)
    res = units[0]
    assert res.resident and res.name == "persistent"
    assert res.shapes == ((1024,),) * 48 and res.psi == 48 * 1024
    assert units[1].name == "embed" and len(units) == 1 + 1 + 6
    assert all(len(w.shapes) == 4 * 4 for w in units[2:])  # 4 matrices per layer remain
