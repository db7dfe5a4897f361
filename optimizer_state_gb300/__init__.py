"""ZeRO-3 sharded model-state hot path for one GB300.

The CUDA library (``csrc/``, built in-tree to ``_build/libz3.so`` by
:mod:`optimizer_state_gb300.build`) is reached through the thin ctypes
binding in :mod:`optimizer_state_gb300.z3`; importing this package loads
nothing.  :mod:`optimizer_state_gb300.schedule` drives multi-unit model steps
and the stage variants, :mod:`optimizer_state_gb300.checkpoint` writes and
reads per-rank shard sets, and :mod:`optimizer_state_gb300.inputs` holds the
seeded synthetic workloads.
"""
