"""Multi-layer ZeRO-3 step: the schedule of "The ZeRO-3 Diagram Most People
Remember Is Wrong", s.3 over a whole model.

Forward: AllGather of every unit (layer, bucket of layers or embedding) in
order.  Backward: for every unit in reverse order, AllGather again, then the
fused reduce-scatter + Adam of that unit ("ZeRO Stage 3: Parameter
Partitioning": the backward pass traverses layers in reverse).  Every gather
lands in one transient buffer sized for the largest unit (same page: the
transient buffer is bounded by the largest single layer); with prefetch
depth D there are D + 1 of them.  A resident unit (persistence threshold) is
never gathered before use: its kept copy is refreshed after its update.

The library schedules the step itself (z3_model_step); the call-by-call form
(``step(..., on_gather=hook)``) issues the same schedule from Python so that
a caller can run its own work where a unit's compute would sit.  Argument
marshalling and launch ordering only; every step runs in the CUDA library
through :mod:`optimizer_state_gb300.z3`.
"""
from __future__ import annotations

import torch

from . import inputs as I
from . import z3


class Unit:
    """Sharded state of one unit (a layer or the embedding)."""

    def __init__(self, w: I.Workload, dev, gen: torch.Generator | None, grads: bool = True,
                 hp: dict | None = None):
        self.w = w
        self.hp = hp                    # this unit's own hyperparameters (None: the step's)
        self.L = z3.Layout(w.numel, w.n_ranks)
        T = self.L.psi_padded
        self.shards = torch.empty(T, dtype=torch.bfloat16, device=dev)
        self.master = torch.empty(T, dtype=torch.float32, device=dev)
        self.m = torch.empty(T, dtype=torch.float32, device=dev)
        self.v = torch.empty(T, dtype=torch.float32, device=dev)
        self.grads = None
        # a resident unit keeps its gathered parameters for the whole run
        self.resident = torch.empty(self.L.psi, dtype=torch.bfloat16, device=dev) \
            if w.resident else None
        if gen is not None:
            full = I.draw_master(w, gen, dev).to(dev)
            self._partition(full)
            del full
            if grads:
                self.grads = I.draw_grads(w, gen, dev).to(dev)

    def _partition(self, full: torch.Tensor):
        z3.z3_partition(self.L, full, self.shards, self.master, self.m, self.v)
        if self.resident is not None:
            z3.z3_allgather(self.L, self.shards, self.resident)

    @classmethod
    def from_full(cls, w: I.Workload, dev, master_full: torch.Tensor, grads_full: torch.Tensor):
        """A unit built from given values: master_full is this unit's fp32
        parameters [Psi_u]; grads_full holds its per-rank gradients as the
        columns of a [N][>= Psi_u] tensor."""
        u = cls(w, dev, None, grads=False)
        u._partition(master_full.contiguous())
        u.grads = torch.zeros((w.n_ranks, w.grad_stride), dtype=torch.bfloat16, device=dev)
        u.grads[:, :w.psi].copy_(grads_full)
        return u

    @property
    def step_bytes(self) -> int:
        st = self.L.stats()
        # a resident unit is gathered once per step instead of twice
        return st["hbm_step_layer"] - (st["hbm_allgather"] if self.resident is not None else 0)


class Model:
    """All units of a model plus the shared transient gathered buffer."""

    def __init__(self, units: list[Unit], dev):
        self.units = units
        self.dev = dev
        self.full = torch.empty(max([u.L.psi for u in units if u.resident is None] or [1]),
                                dtype=torch.bfloat16, device=dev)
        self.t = 0

    @property
    def psi(self) -> int:
        return sum(u.L.psi for u in self.units)

    @property
    def step_bytes(self) -> int:
        return sum(u.step_bytes for u in self.units)

    def launches_per_step(self) -> int:
        n = 0
        for u in self.units:
            tabs = -(-sum(1 for x in u.L.numel if x > 0) // 40)
            n += (2 if u.resident is not None else 3) * tabs
        return n

    def unit_args(self):
        return [(u.L, u.shards, u.master, u.m, u.v, u.grads, u.w.grad_stride,
                 1.0 / u.w.n_ranks, u.resident, u.hp) for u in self.units]

    @staticmethod
    def _update(u: Unit, hp: dict, t: int, stream):
        z3.z3_reduce_scatter_adam(u.L, u.grads, u.w.grad_stride, 1.0 / u.w.n_ranks, None,
                                  u.master, u.m, u.v, u.shards, u.hp or hp, t, stream=stream)
        if u.resident is not None:
            z3.z3_allgather(u.L, u.shards, u.resident, stream=stream)

    def step(self, hp: dict, stream=None, t: int | None = None, on_gather=None):
        """One training step, scheduled by the library (z3_model_step).
        With `on_gather(phase, index)` the same schedule is issued call by
        call from here instead, and the hook is called after each gather is
        enqueued, with the transient buffer holding that unit's parameters
        once the stream reaches it -- the point where the forward or backward
        compute of the unit would run."""
        if t is None:
            self.t += 1
            t = self.t
        if on_gather is None:
            z3.z3_model_step(self.unit_args(), [self.full], hp, t, stream=stream)
            return
        for i, u in enumerate(self.units):            # forward
            if u.resident is None:
                z3.z3_allgather(u.L, u.shards, self.full, stream=stream)
            on_gather("forward", i)
        for i in range(len(self.units) - 1, -1, -1):    # backward, reverse order
            u = self.units[i]
            if u.resident is None:
                z3.z3_allgather(u.L, u.shards, self.full, stream=stream)
            on_gather("backward", i)
            self._update(u, hp, t, stream)


def _torch_stream(stream):
    """A torch stream object for a stream argument (None: the current stream;
    an int: a raw cudaStream_t handle).  Handle 0 is the legacy default
    stream; torch's stream wrapper treats a zero pointer as "none given" and
    hands out a fresh pool stream instead, which would leave the work
    unordered with everything else on the default stream, so 0 maps to
    torch's default stream explicitly."""
    if stream is None:
        return torch.cuda.current_stream()
    if isinstance(stream, int):
        return torch.cuda.default_stream() if stream == 0 else torch.cuda.ExternalStream(stream)
    return stream


class PrefetchModel(Model):
    """The same step with the gather of the next unit prefetched one unit
    ahead on a second stream ("ZeRO Stage 3: Parameter Partitioning": the
    All-Gather for layer l+1 proceeds while layer l computes; "ZeRO Stages:
    ...": prefetched layers occupy memory, so two transient buffers).

    Backward: the gather of unit i-1 runs on the gather stream while unit i's
    fused reduce-scatter + Adam runs on the main stream.  Ordering is by
    events: a unit's update waits for its gather; a gather into a buffer waits
    until the update of the unit that last used that buffer is enqueued after
    it (the point where that unit's backward compute would have finished)."""

    def __init__(self, units: list[Unit], dev, depth: int = 1):
        super().__init__(units, dev)
        self.depth = depth
        self.bufs = [self.full] + [torch.empty_like(self.full) for _ in range(depth)]
        self.gstream = torch.cuda.Stream(device=dev)

    def step(self, hp: dict, stream=None, t: int | None = None, on_gather=None):
        if t is None:
            self.t += 1
            t = self.t
        if on_gather is None:
            z3.z3_model_step(self.unit_args(), self.bufs, hp, t, stream=stream,
                             gather_stream=self.gstream)
            return
        if self.depth != 1:
            raise NotImplementedError("the call-by-call schedule prefetches one unit ahead")
        main = _torch_stream(stream)
        g = self.gstream
        n = len(self.units)
        freed = [torch.cuda.Event(), torch.cuda.Event()]
        g.wait_stream(main)                            # shards updated by the last step
        for i, u in enumerate(self.units):            # forward, back to back on g
            if u.resident is None:
                z3.z3_allgather(u.L, u.shards, self.bufs[i % 2], stream=g.cuda_stream)
            with torch.cuda.stream(g):
                on_gather("forward", i)
        order = list(range(n - 1, -1, -1))
        gathered = {}

        def gather(i):
            u = self.units[i]
            if u.resident is None:
                z3.z3_allgather(u.L, u.shards, self.bufs[i % 2], stream=g.cuda_stream)
            with torch.cuda.stream(g):
                on_gather("backward", i)
            ev = torch.cuda.Event()
            ev.record(g)
            gathered[i] = ev
        gather(order[0])
        for k, i in enumerate(order):
            u = self.units[i]
            if k + 1 < n:
                nxt = order[k + 1]
                if k >= 1:
                    g.wait_event(freed[nxt % 2])       # buffer of unit i+1 is free again
                gather(nxt)                            # prefetch one unit ahead
            main.wait_event(gathered[i])
            self._update(u, hp, t, main.cuda_stream)
            freed[i % 2].record(main)
        main.wait_stream(g)


def full_step_model(dev, seed: int = 0, prefetch: int = 0, bucket_layers: int = 1,
                    persistence_threshold: int = 0) -> Model:
    """The 24-layer d=1024 model with its [50257, 1024] embedding, N_d = 16.

    bucket_layers: the parameter-bucket knob of "The ZeRO-3 Diagram Most
    People Remember Is Wrong", s.8 -- that many consecutive layers form one
    unit (one gather and one fused reduce-scatter + Adam launch each; the
    transient buffer grows to the largest unit).  Every parameter is still
    partitioned on its own, and the update is elementwise, so the result of
    a step does not depend on the bucket size.

    prefetch: how many units ahead the backward gathers run on a second stream
    (0: none; each unit of depth costs one more transient buffer).

    persistence_threshold: the persistence-threshold knob of the same section
    -- parameters of fewer elements are not released after use: they form
    one resident unit whose gathered copy is kept and refreshed once per step
    after its update, instead of being gathered before every use.
    """
    gen = I.make_generator(seed, dev)
    units = [Unit(w, dev, gen) for w in I.full_step_units(bucket_layers, persistence_threshold)]
    return PrefetchModel(units, dev, int(prefetch)) if prefetch else Model(units, dev)



# ---------------------------------------------------------------------------
# The other ZeRO stages and plain data parallelism on the same kernels
# ("ZeRO Stages: Sharding Optimizer State, Gradients, and Parameters";
# "ZeRO Stage 3: Parameter Partitioning", communication list).  Each returns
# the HBM bytes per unpadded element its launches move.
# ---------------------------------------------------------------------------

def stage2_step(u: Unit, full: torch.Tensor, hp: dict, t: int, stream=None) -> int:
    """Stage 2: reduce-scatter the gradients (fused with the shard Adam), then
    one all-gather of the updated parameters into the replica."""
    N = u.w.n_ranks
    z3.z3_reduce_scatter_adam(u.L, u.grads, u.w.grad_stride, 1.0 / N, None, u.master, u.m, u.v,
                              u.shards, hp, t, stream=stream)
    z3.z3_allgather(u.L, u.shards, full, stream=stream)
    return (2 * N + 26) + 4


def stage1_step(u: Unit, grad_full: torch.Tensor, grad_shards: torch.Tensor,
                full: torch.Tensor, hp: dict, t: int, stream=None) -> int:
    """Stage 1: all-reduce the gradients (every rank receives the full sum),
    each rank updates its slice of the optimizer state from its slice of the
    reduced gradient, then an all-gather of the updated parameters."""
    N = u.w.n_ranks
    z3.z3_allreduce(u.L, u.grads, u.w.grad_stride, grad_full, 1.0 / N, stream=stream)
    z3.z3_scatter(u.L, grad_full, grad_shards, stream=stream)
    z3.z3_adam_shard_step(u.L, u.master, u.m, u.v, grad_shards, u.shards, hp, t, stream=stream)
    z3.z3_allgather(u.L, u.shards, full, stream=stream)
    return (2 * N + 4) + 8 + 30 + 4


class DPReplica:
    """Plain data parallelism: every rank holds the whole fp32 master, m, v and
    bf16 parameters; the state is laid out as one rank (N = 1)."""

    def __init__(self, w: I.Workload, dev, gen: torch.Generator):
        self.w = w
        self.L = z3.Layout(w.numel, w.n_ranks)         # the gradient fold over N ranks
        self.L1 = z3.Layout(w.numel, 1)                # unsharded state
        n = self.L1.psi
        self.params = torch.empty(n, dtype=torch.bfloat16, device=dev)
        self.master = torch.empty(n, dtype=torch.float32, device=dev)
        self.m = torch.empty(n, dtype=torch.float32, device=dev)
        self.v = torch.empty(n, dtype=torch.float32, device=dev)
        full = I.draw_master(w, gen, dev).to(dev)
        z3.z3_partition(self.L1, full, self.params, self.master, self.m, self.v)
        self.grads = I.draw_grads(w, gen, dev).to(dev)
        self.grad_full = torch.empty(n, dtype=torch.float32, device=dev)

    def step(self, hp: dict, t: int, stream=None) -> int:
        N = self.w.n_ranks
        z3.z3_allreduce(self.L, self.grads, self.w.grad_stride, self.grad_full, 1.0 / N,
                        stream=stream)
        z3.z3_adam_shard_step(self.L1, self.master, self.m, self.v, self.grad_full, self.params,
                              hp, t, stream=stream)
        return (2 * N + 4) + 30
