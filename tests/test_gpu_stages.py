"""Stage 1, stage 2, stage 3 and plain data parallelism on the GPU.

'The ZeRO-3 Diagram Most People Remember Is Wrong', s.4: ZeRO keeps
data-parallel semantics.  From the same parameters and the same per-rank
gradients, one step of every variant leaves the same bf16 parameter replica
and the same fp32 master/moments (bit for bit); the plain DP step itself is
checked against the oracle (all-reduce, then Adam on the whole tensor), and
the new all-reduce and scatter kernels against the oracle directly.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import bits32, f32, u16
from optimizer_state_gb300 import inputs as I

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
LAYOUTS = [([35, 13, 12], 4), ([100003, 7, 1, 0, 4099], 3), ([262147], 64),
           (I.LAYER_D1024.numel, 8)]


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.fail("CUDA is not available: the GPU tests need a GPU")
    from optimizer_state_gb300 import build, schedule, z3
    build.build()
    z3.load()
    return z3, schedule


@pytest.mark.parametrize("numel,n_ranks", LAYOUTS, ids=[f"{len(a)}p-N{b}" for a, b in LAYOUTS])
def test_all_variants_agree_with_dp(mods, orc, numel, n_ranks):
    z3, sch = mods
    dev = torch.device("cuda")
    w = I.Workload("v", tuple((n,) for n in numel), n_ranks, 0.02, 1e-3)
    dp = sch.DPReplica(w, dev, I.make_generator(9, dev))
    units = [sch.Unit(w, dev, I.make_generator(9, dev)) for _ in range(3)]
    L = units[0].L
    O = orc.layout(numel, n_ranks)
    # all-reduce and scatter against the oracle
    gh = u16(dp.grads).reshape(-1)
    want_ar = orc.allreduce(O, gh, w.grad_stride, 1.0 / n_ranks)
    gfull = torch.empty(L.psi, dtype=torch.float32, device=dev)
    gsh = torch.empty(L.psi_padded, dtype=torch.float32, device=dev)
    z3.z3_allreduce(L, dp.grads, w.grad_stride, gfull, 1.0 / n_ranks)
    z3.z3_scatter(L, gfull, gsh)
    torch.cuda.synchronize()
    assert np.array_equal(bits32(f32(gfull)), bits32(want_ar))
    assert np.array_equal(bits32(f32(gsh)), bits32(orc.partition(O, want_ar)[1]))
    # oracle DP step
    p0 = f32(dp.master).copy()
    o_m, o_v = np.zeros_like(p0), np.zeros_like(p0)
    o_bf = np.zeros(p0.size, np.uint16)
    orc.adam(p0, o_m, o_v, want_ar, o_bf, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"],
             HP["weight_decay"], 1)
    # one step of every variant
    dp.step(HP, 1)
    fulls = [torch.empty(L.psi, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    sch.stage1_step(units[0], gfull, gsh, fulls[0], HP, 1)
    sch.stage2_step(units[1], fulls[1], HP, 1)
    z3.z3_step_layer(L, units[2].shards, fulls[2], units[2].grads, w.grad_stride,
                     1.0 / n_ranks, units[2].master, units[2].m, units[2].v, HP, 1)
    z3.z3_allgather(L, units[2].shards, fulls[2])      # the next forward gather
    torch.cuda.synchronize()
    assert np.array_equal(u16(dp.params), o_bf)
    assert np.array_equal(bits32(f32(dp.master)), bits32(p0))
    for u, full in zip(units, fulls):
        assert np.array_equal(u16(full), o_bf)
        for name, want in (("master", p0), ("m", o_m), ("v", o_v)):
            got = orc.allgather_f32(O, f32(getattr(u, name)))
            assert np.array_equal(bits32(got), bits32(want)), name
