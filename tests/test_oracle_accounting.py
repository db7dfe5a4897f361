"""Oracle pins: model-state bytes and step traffic against the figures the
pages print (tests/golden/page_figures.json)."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FIG = json.load(open(os.path.join(GOLDEN, "page_figures.json")))


def test_worked_7b_example(orc):
    f = FIG["worked_7b_64"]
    # 7e9 parameters as seven 1e9-element tensors; 64 divides each
    L = orc.layout([f["params"] // 7] * 7, f["n_ranks"])
    a = orc.accounting(L)
    assert a["state_bytes_per_rank"] == f["bytes_per_gpu"]
    assert a["state_bytes_per_rank"] * f["n_ranks"] == f["total_state_bytes"]
    assert FIG["stage3_state_bytes_per_param"]["value"] * L.psi == f["total_state_bytes"]


def test_sixteen_psi_over_n_when_divisible(orc):
    # one d=1024 transformer layer, N = 8: every n_p divides by 8
    numel = [3072 * 1024, 1024 * 1024, 4096 * 1024, 1024 * 4096, 1024, 1024]
    L = orc.layout(numel, 8)
    a = orc.accounting(L)
    assert a["state_bytes_per_rank"] * 8 == 16 * L.psi
    # when N does not divide, the pad is what is stored beyond 16*Psi/N
    L2 = orc.layout([35, 13, 12], 4)
    a2 = orc.accounting(L2)
    assert a2["state_bytes_per_rank"] * 4 - 16 * L2.psi == 16 * (L2.psi_padded - L2.psi)


def test_largest_layer_d4096(orc):
    f = FIG["largest_layer_d4096"]
    n = 4 * f["d_model"] ** 2
    assert abs(n - f["params_approx"]) / f["params_approx"] < 0.01
    L = orc.layout([n], 8)
    gathered_bytes = 2 * L.psi          # one fp16/bf16 full copy
    assert abs(gathered_bytes / 1e9 - f["gb_fp16_approx"]) < 0.005


def test_step_volume_six_vs_two(orc):
    f = FIG["step_volume"]
    for numel, n_ranks in (([35, 13, 12], 4), ([12584960], 8), ([10 ** 6] * 3, 64)):
        L = orc.layout(numel, n_ranks)
        a = orc.accounting(L)
        assert a["step_volume_bytes"] == f["stage3_bytes_per_psi"] * L.psi
        assert a["dp_volume_bytes"] == f["dp_bytes_per_psi"] * L.psi
        assert a["step_volume_bytes"] == 3 * a["dp_volume_bytes"]
        assert sum(f["stage3_breakdown"].values()) == f["stage3_bytes_per_psi"]


def test_per_rank_table_column(orc):
    f = FIG["per_rank_volume_table"]
    for n_ranks in (2, 8, 64):
        L = orc.layout([1 << 20], n_ranks)
        a = orc.accounting(L)
        frac = (n_ranks - 1) / n_ranks
        assert np.isclose(a["per_rank_ring_elems_dp"], f["baseline_allreduce_factor"] * L.psi * frac)
        assert np.isclose(a["per_rank_ring_elems_stage3"], f["stage3_factor_approx"] * L.psi * frac)


def test_eighteen_byte_variant(orc):
    f = FIG["mixed_precision_bytes"]
    L = orc.layout([4096], 8)
    a = orc.accounting(L)
    assert a["state_bytes_per_rank_fp32_grad"] == f["per_param_total"] * L.S
    assert a["state_bytes_per_rank_fp32_grad"] - a["state_bytes_per_rank"] == \
        (f["gradient"] - 2) * L.S
    assert f["optimizer_state"] == 4 + 4 + 4
