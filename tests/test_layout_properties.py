"""Property tests of the library's host layout logic against the oracle
(random parameter lists with empty and very large parameters, rank counts up
to 1024), and of the overflow guards."""
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")

from optimizer_state_gb300 import build as z3build  # noqa: E402
from optimizer_state_gb300 import z3  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    z3build.build()
    z3.load()


@hyp.settings(max_examples=300, deadline=None)
@hyp.given(numel=st.lists(st.one_of(st.integers(0, 64), st.integers(0, 10 ** 6),
                                    st.integers(0, 2 ** 40)), min_size=1, max_size=90),
           n_ranks=st.one_of(st.integers(1, 9), st.sampled_from([16, 64, 128, 1024])))
def test_layout_and_stats_match_oracle(orc, numel, n_ranks):
    try:
        L = z3.Layout(numel, n_ranks)
    except z3.Z3Error as e:
        # only the tile count of an enormous parameter may overflow a launch grid
        assert e.status == z3.Z3_ERR_OVERFLOW
        return
    O = orc.layout(numel, n_ranks)
    assert (L.S, L.psi, L.psi_padded) == (O.S, O.psi, O.psi_padded)
    assert L.shard_numel == list(O.shard_numel) and L.shard_off == list(O.shard_off)
    assert L.full_off == list(O.full_off)
    st_ = L.stats()
    acc = orc.accounting(O)
    assert st_["state_bytes_per_rank"] == acc["state_bytes_per_rank"]
    assert st_["step_volume_bytes"] == acc["step_volume_bytes"] == 3 * acc["dp_volume_bytes"]
    # minimal padding: fewer than N pad elements per parameter
    for n, s in zip(L.numel, L.shard_numel):
        assert s * n_ranks >= n and (s - 1) * n_ranks < n or n == 0


def test_overflow_guards():
    with pytest.raises(z3.Z3Error) as e:
        z3.Layout([2 ** 62, 2 ** 62], 1)
    assert e.value.status == z3.Z3_ERR_OVERFLOW
    with pytest.raises(z3.Z3Error) as e:
        z3.Layout([2 ** 61], 4)           # [N][S] fp32 bytes overflow int64
    assert e.value.status == z3.Z3_ERR_OVERFLOW
