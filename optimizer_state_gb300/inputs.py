"""Seeded synthetic inputs for the ZeRO-3 sharded layer step.

This module holds the workload definitions (parameter shapes, rank counts,
value distributions) and the random draws only.  It contains none of the
method's arithmetic -- no layout, gather, reduction or optimizer code -- so
the CUDA library and the CPU oracle can both consume exactly the same input
bytes without sharing any of the computation.

Recipe (every workload):
  * one ``torch.Generator`` seeded with ``seed``; on the CPU for tensors up
    to 256 MB, on the device above that (the oracle always reads back the
    exact bytes, so it never needs to reproduce the generator);
  * master parameters: one draw of Psi values from N(0, param_std) in fp32,
    assigned to the parameters in list order (the bf16 copy is made by the
    partition step, not here);
  * gradients: for every step and every rank k = 0..N-1 in that order, one
    draw of Psi values from N(0, grad_std) in fp32, rounded to bf16 (round
    to nearest even, the torch cast), laid out as rank k's full gradient at
    row k of a [N][grad_stride] buffer; the gap [Psi, grad_stride) is zero.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# Row pitch of the per-rank gradient buffer, in elements.  The library wants
# each rank's row to start on a 16-byte boundary (8 bf16 elements).
GRAD_ROW_ALIGN = 8
_CPU_LIMIT_BYTES = 256 << 20


@dataclass(frozen=True)
class Workload:
    name: str
    shapes: tuple          # parameter shapes, in layer order
    n_ranks: int           # N, the number of logical data-parallel ranks
    param_std: float
    grad_std: float
    hp: dict = field(default_factory=lambda: dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                                  weight_decay=0.0))
    steps: int = 1
    micro_batches: int = 1
    resident: bool = False  # gathered once per step and kept (persistence threshold)

    @property
    def numel(self) -> list[int]:
        return [math.prod(s) for s in self.shapes]

    @property
    def psi(self) -> int:
        return sum(self.numel)

    @property
    def grad_stride(self) -> int:
        return grad_stride(self.psi)


def grad_stride(psi: int) -> int:
    return -(-psi // GRAD_ROW_ALIGN) * GRAD_ROW_ALIGN


def transformer_layer_shapes(d: int, ffn: int, gated: bool) -> tuple:
    """Wqkv, Wo, the FFN matrices (gate+up+down when gated, up+down
    otherwise) and two norm gain vectors, in that order."""
    if gated:
        ffn_shapes = ((ffn, d), (ffn, d), (d, ffn))
    else:
        ffn_shapes = ((ffn, d), (d, ffn))
    return ((3 * d, d), (d, d)) + ffn_shapes + ((d,), (d,))


TINY = Workload("tiny", ((7, 5), (13,), (4, 3)), n_ranks=4, param_std=0.02, grad_std=1.0,
                steps=3)
LAYER_D1024 = Workload("layer_d1024", transformer_layer_shapes(1024, 4096, gated=False),
                       n_ranks=8, param_std=0.02, grad_std=1e-3)


def layer_7b(n_ranks: int) -> Workload:
    return Workload(f"layer_7b_nd{n_ranks}", transformer_layer_shapes(4096, 11008, gated=True),
                    n_ranks=n_ranks, param_std=0.02, grad_std=1e-3)


def layer_primes(n_ranks: int, small: bool = False) -> Workload:
    """A layer of three prime-length parameters: every chunk after the first
    has a different phase between its full-space and shard-space indices,
    so the reduce and gather kernels must shift 16-byte windows.  The small
    variant (13.6 M elements, its gradients still larger than L2) is the
    profiling case of the same kernels."""
    if small:
        return Workload(f"layer_primes_small_nd{n_ranks}", ((8388617,), (4194319,), (1048583,)),
                        n_ranks=n_ranks, param_std=0.02, grad_std=1e-3)
    return Workload(f"layer_primes_nd{n_ranks}", ((67108879,), (33554467,), (1048583,)),
                    n_ranks=n_ranks, param_std=0.02, grad_std=1e-3)


VOCAB = 50257
FULL_STEP_LAYERS = 24


def _full_step_shapes() -> list[tuple]:
    """Every parameter shape of the full-step model in model order: the
    embedding, then the 24 layers' parameters layer by layer."""
    layer = transformer_layer_shapes(1024, 4096, gated=False)
    return [(VOCAB, 1024)] + [sh for _ in range(FULL_STEP_LAYERS) for sh in layer]


def full_step_param_ids(bucket_layers: int = 1, persistence_threshold: int = 0) -> list[tuple]:
    """For each unit of full_step_units(...), the model-order indices of its
    parameters (index 0 is the embedding, then each layer's parameters).

    Unit 0 is the embedding; then buckets of `bucket_layers` consecutive
    layers.  With persistence_threshold > 0 every parameter of fewer than
    that many elements leaves its bucket and joins one resident unit placed
    first: its gathered copy is kept for the whole run (updated once per
    step), and since its gradients are complete only when the backward pass
    has finished, it is updated last (the step runs units in reverse)."""
    shapes = _full_step_shapes()
    per_layer = len(transformer_layer_shapes(1024, 4096, gated=False))
    small = {i for i, sh in enumerate(shapes) if math.prod(sh) < persistence_threshold}
    units = [tuple(i for i in (0,) if i not in small)]
    for l0 in range(0, FULL_STEP_LAYERS, bucket_layers):
        k = min(bucket_layers, FULL_STEP_LAYERS - l0)
        ids = range(1 + l0 * per_layer, 1 + (l0 + k) * per_layer)
        units.append(tuple(i for i in ids if i not in small))
    units = [u for u in units if u]
    if small:
        units.insert(0, tuple(sorted(small)))
    return units


def full_step_units(bucket_layers: int = 1, persistence_threshold: int = 0) -> list[Workload]:
    """24-layer d=1024 model plus the [50257, 1024] embedding, N = 16, as
    units (see full_step_param_ids for which parameters form each unit)."""
    shapes = _full_step_shapes()
    ids = full_step_param_ids(bucket_layers, persistence_threshold)
    resident = persistence_threshold > 0 and \
        all(math.prod(shapes[i]) < persistence_threshold for i in ids[0])
    per_layer = len(transformer_layer_shapes(1024, 4096, gated=False))
    out = []
    for n, u in enumerate(ids):
        is_res = resident and n == 0
        if is_res:
            name = "persistent"
        elif u == (0,):
            name = "embed"
        else:
            name = f"layers{(u[0] - 1) // per_layer}-{(u[-1] - 1) // per_layer}"
        out.append(Workload(name, tuple(shapes[i] for i in u), n_ranks=16, param_std=0.02,
                            grad_std=1e-3, resident=is_res))
    return out


def next_prime(n: int) -> int:
    """Smallest prime >= n (trial division; n < 2**32 here)."""
    def is_prime(x):
        if x < 2:
            return False
        if x % 2 == 0:
            return x == 2
        f = 3
        while f * f <= x:
            if x % f == 0:
                return False
            f += 2
        return True
    while not is_prime(n):
        n += 1
    return n


SWEEP_SIZES = [next_prime(2 ** k + 1) for k in range(18, 31)] + [2 ** 31 - 1]


def sweep(n: int, n_ranks: int) -> Workload:
    """One flattened parameter of prime length n; 4 micro-batches."""
    return Workload(f"sweep_n{n}_nd{n_ranks}", ((n,),), n_ranks=n_ranks, param_std=0.02,
                    grad_std=1e-3, micro_batches=4)


def _device_for(nbytes: int, device) -> torch.device:
    dev = torch.device(device)
    if dev.type == "cuda" or nbytes <= _CPU_LIMIT_BYTES:
        return dev
    raise ValueError(f"{nbytes} bytes is above the CPU-generator limit; draw on the device")


def make_generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def draw_master(w: Workload, gen: torch.Generator, device) -> torch.Tensor:
    """fp32 [Psi]: the full master parameters, N(0, param_std)."""
    dev = _device_for(4 * w.psi, device)
    x = torch.empty(w.psi, dtype=torch.float32, device=dev)
    x.normal_(0.0, w.param_std, generator=gen)
    return x


def draw_grads(w: Workload, gen: torch.Generator, device, out: torch.Tensor | None = None
               ) -> torch.Tensor:
    """bf16 [N, grad_stride]: one step's per-rank full gradients."""
    dev = _device_for(2 * w.n_ranks * w.grad_stride, device)
    if out is None:
        out = torch.zeros((w.n_ranks, w.grad_stride), dtype=torch.bfloat16, device=dev)
    tmp = torch.empty(w.psi, dtype=torch.float32, device=dev)
    for k in range(w.n_ranks):
        tmp.normal_(0.0, w.grad_std, generator=gen)
        out[k, :w.psi].copy_(tmp)
    return out


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """View a bf16 tensor as its uint16 bit patterns (int16 storage)."""
    return t.view(torch.int16)
