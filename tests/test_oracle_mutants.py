"""The pins catch plausible mistakes: each case plants one mistake in a copy
of the oracle source (on the CPU), builds it, binds it in place of the
oracle, and requires at least one pin test to fail.  A mutant that every pin
accepts would mean the pins do not constrain that part of the oracle."""
import ctypes

import pytest

import oracle as orc_pkg
from oracle import oracle as orc_mod
import test_oracle_accounting as T_acc
import test_oracle_adam as T_adam
import test_oracle_bf16 as T_bf16
import test_oracle_layout as T_lay
import test_oracle_reduce as T_red

FOLD = """    float acc = or_f32_from_bf16(grads[e]);
    for (int32_t k = 1; k < n_ranks; ++k)
        acc = acc + or_f32_from_bf16(grads[(int64_t)k * grad_stride + e]);"""

MUTANTS = {
    "fold starts from +0": (FOLD, """    float acc = 0.0f;
    for (int32_t k = 0; k < n_ranks; ++k)
        acc = acc + or_f32_from_bf16(grads[(int64_t)k * grad_stride + e]);"""),
    "fold in descending rank order": (FOLD, """    float acc = or_f32_from_bf16(grads[(int64_t)(n_ranks - 1) * grad_stride + e]);
    for (int32_t k = n_ranks - 2; k >= 0; --k)
        acc = acc + or_f32_from_bf16(grads[(int64_t)k * grad_stride + e]);"""),
    "pad at the front of the parameter": (
        """                float x = 0.0f;
                if (i < numel[p])
                    x = full[full_off[p] + i];""",
        """                float x = 0.0f;
                int64_t pad = shard_numel[p] * n_ranks - numel[p];
                if (i >= pad)
                    x = full[full_off[p] + i - pad];"""),
    "gathered slice reversed": (
        "src + (size_t)(r * S + shard_off[p] + j) * elem, elem);",
        "src + (size_t)(r * S + shard_off[p] + (shard_numel[p] - 1 - j)) * elem, elem);"),
    "scale applied to each rank before the sum": (
        FOLD + "\n    return acc * scale;",
        """    float acc = or_f32_from_bf16(grads[e]) * scale;
    for (int32_t k = 1; k < n_ranks; ++k)
        acc = acc + or_f32_from_bf16(grads[(int64_t)k * grad_stride + e]) * scale;
    return acc;"""),
    "weight decay dropped": ("float pd = p - k.lwd * p;", "float pd = p;"),
    "weight decay also added to the gradient": (
        "float g = grad[i];", "float g = grad[i] + (k.lwd / k.lr) * master[i];"),
    "bias corrections one step late": (
        "k.rb1 = (float)(1.0 / (1.0 - pow(beta1, (double)step)));",
        "k.rb1 = (float)(1.0 / (1.0 - pow(beta1, (double)(step + 1))));"),
    "second-moment correction uses beta1": (
        "k.rb2 = (float)(1.0 / (1.0 - pow(beta2, (double)step)));",
        "k.rb2 = (float)(1.0 / (1.0 - pow(beta1, (double)step)));"),
    "reduce-scatter leaves the pad untouched": (
        """                if (i >= numel[p]) {
                    out[at] = 0.0f;
                    continue;
                }""",
        """                if (i >= numel[p]) {
                    continue;
                }"""),
    "reduce-scatter reads the next rank's slice": (
        "full_off[p] + i, scale);", "full_off[p] + (i + shard_numel[p] < numel[p] ? i + shard_numel[p] : i), scale);"),
    "bf16 copy cast from the master before the update": (
        "param_bf16[i] = or_bf16_from_f32(p1);", "param_bf16[i] = or_bf16_from_f32(p);"),
    "partition starts the moments at the master": (
        """                m[at] = 0.0f;
                v[at] = 0.0f;""",
        """                m[at] = x;
                v[at] = x * x;"""),
    "gather writes each rank's slice one element late": (
        "memcpy(dst + (size_t)(full_off[p] + i) * elem,",
        "memcpy(dst + (size_t)(full_off[p] + (i + 1 < numel[p] ? i + 1 : i)) * elem,"),
    "accumulate drops the running sum": (
        "out[at] = accumulate ? out[at] + g : g;", "out[at] = g;"),
    "eps inside the square root": (
        "float u = mh / (sqrtf(vh) + k.eps);", "float u = mh / sqrtf(vh + k.eps);"),
    "no first-moment bias correction": ("float mh = m1 * k.rb1;", "float mh = m1;"),
    "wrong sign in the first moment": (
        "float m1 = k.b1 * m[i] + k.c1 * g;", "float m1 = k.b1 * m[i] - k.c1 * g;"),
    "second moment from g, not g*g": (
        "float v1 = k.b2 * v[i] + k.c2 * (g * g);", "float v1 = k.b2 * v[i] + k.c2 * g;"),
    "bf16 by truncation": ("return (uint16_t)(kept + (uint32_t)round_up);",
                           "return (uint16_t)(kept);"),
    "bf16 ties away from zero": ("round_up = (int)(kept & 1u);", "round_up = 1;"),
    "18-byte state accounting": ("*state_bytes_per_rank_16 = (2 + 2 + 4 + 4 + 4) * S;",
                                 "*state_bytes_per_rank_16 = (2 + 4 + 4 + 4 + 4) * S;"),
}

PINS = [
    lambda o: T_red.test_golden_fold_cases(o),
    lambda o: T_red.test_integer_grads_equal_torch_sum(o, 8),
    lambda o: T_red.test_micro_batch_accumulation(o),
    lambda o: T_lay.test_single_param_bruteforce(o, 7),
    lambda o: T_lay.test_allgather_round_trip_and_reshape(o, 7),
    lambda o: T_adam.test_against_torch_adam(o, 0.0),
    lambda o: T_adam.test_against_torch_adam(o, 0.1),
    lambda o: T_adam.test_first_step_closed_form(o),
    lambda o: T_bf16.test_special_values(o),
    lambda o: T_bf16.test_rounding_structured_sample(o),
    lambda o: T_acc.test_worked_7b_example(o),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = orc_mod.source()
    assert src.count(old) == 1, "the mutated snippet must occur exactly once in the oracle"
    lib = orc_mod._bind(ctypes.CDLL(orc_mod.build_variant(src.replace(old, new),
                                                           str(tmp_path))))
    monkeypatch.setattr(orc_mod, "_lib", lib)
    failed = []
    for i, pin in enumerate(PINS):
        try:
            pin(orc_pkg)
        except Exception:  # noqa: BLE001 - a pin that errors out rejects the mutant too
            failed.append(i)
    assert failed, f"no pin catches the mutant '{name}'"
