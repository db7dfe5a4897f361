"""Shared helpers of the GPU parity tests: guarded device buffers, host
copies as numpy bit patterns, and the tolerance of the Adam outputs."""
import numpy as np
import torch

GUARD = 64                     # guard elements on each side of a buffer
CANARY16 = 0x5A5A
CANARY32 = 0x7FC0DEAD          # a NaN pattern: never produced by the kernels


class Guarded:
    """A device buffer with canary words before and after it."""

    def __init__(self, n: int, dtype: torch.dtype, fill=None):
        self.n = n
        self.dtype = dtype
        self.raw = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        bits = self.raw.view(torch.int16 if dtype.itemsize == 2 else torch.int32)
        canary = CANARY16 if dtype.itemsize == 2 else CANARY32   # both fit the signed type
        bits.fill_(canary)
        self._canary = canary
        self.t = self.raw[GUARD:GUARD + n]
        assert self.t.data_ptr() % 16 == 0
        if fill is not None:
            self.t.copy_(fill)

    def guards_intact(self) -> bool:
        bits = self.raw.view(torch.int16 if self.dtype.itemsize == 2 else torch.int32)
        head, tail = bits[:GUARD], bits[GUARD + self.n:]
        return bool((head == self._canary).all()) and bool((tail == self._canary).all())


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def bits32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def within_adam_tolerance(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """|a - b| <= max(1e-6 |b|, 1e-9): the fp32 master/moment tolerance."""
    g = got.astype(np.float64)
    w = want.astype(np.float64)
    return np.abs(g - w) <= np.maximum(1e-6 * np.abs(w), 1e-9)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps, comparing the patterns as ordered integers."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(ordered(a) - ordered(b))


# ---------------------------------------------------------------------------
# sampled checks at full size: the oracle computes selected outputs one by one
# ---------------------------------------------------------------------------

def sampled_shard_positions(O, n_random: int, seed: int = 0):
    """Shard positions x (int64) covering every rank's first and last owned
    element of every parameter, the element before and after each pad tail,
    and n_random uniform positions."""
    rng = np.random.default_rng(seed)
    xs = []
    for p in range(O.n_params):
        s, o, n = int(O.shard_numel[p]), int(O.shard_off[p]), int(O.numel[p])
        if s == 0:
            continue
        for r in range(O.n_ranks):
            base = r * O.S + o
            valid = max(0, min(s, n - r * s))
            xs += [base, base + s - 1]
            if 0 < valid < s:
                xs += [base + valid - 1, base + valid]
    if O.psi_padded:
        xs += list(rng.integers(0, O.psi_padded, size=n_random))
    return np.unique(np.asarray(xs, np.int64))


def shard_to_full(O, xs: np.ndarray):
    """For shard positions xs: (full index e, valid mask); e is -1 in the pad."""
    r = xs // O.S
    y = xs - r * O.S
    p = np.searchsorted(O.shard_off, y, side="right") - 1
    # skip parameters with s_p = 0 that share an offset with the next one
    s = O.shard_numel[p]
    while np.any(s == 0):
        bad = s == 0
        p[bad] += 1
        s = O.shard_numel[p]
    j = y - O.shard_off[p]
    i = r * s + j
    valid = i < O.numel[p]
    e = np.where(valid, O.full_off[p] + i, -1)
    return e, valid


def gather_rows(t: torch.Tensor, rows: int, stride: int, cols: np.ndarray) -> np.ndarray:
    """t viewed as [rows][stride]: the uint16 bits at the given columns,
    as a C-contiguous [rows][len(cols)] array."""
    idx = torch.from_numpy(cols).to(t.device)
    sub = t.view(rows, stride).index_select(1, idx)
    return u16(sub).reshape(rows, len(cols))


def pick(t: torch.Tensor, idx: np.ndarray) -> torch.Tensor:
    return t.index_select(0, torch.from_numpy(idx).to(t.device))
