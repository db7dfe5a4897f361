"""ZeRO-3 sharded model-state hot path for one GB300.

The CUDA library (``csrc/``, built to ``_lib/libz3.so``) is reached through
the thin ctypes binding in :mod:`optimizer_state_gb300.z3`; importing this
package loads nothing.  :mod:`optimizer_state_gb300.inputs` holds the seeded
synthetic workloads.
"""
