"""Plain CPU oracle for the ZeRO-3 sharded model-state path.

TEST INFRASTRUCTURE ONLY.  It is written from the pages' statement of the
method, in plain C loops (``z3_oracle.c``) behind a numpy wrapper
(``oracle.py``).  Only the tests, the smoke check of ``__graft_entry__`` and
the CPU-baseline leg of ``bench.py`` may use it; the CUDA library neither
imports nor links anything here, and this package imports nothing from the
CUDA library.
"""
from .oracle import (  # noqa: F401
    Layout, accounting, adam, adam_constants, allgather, allgather_f32,
    allreduce, bf16_from_f32, build, f32_from_bf16, layout, partition,
    reduce_scatter, step_layer,
)
