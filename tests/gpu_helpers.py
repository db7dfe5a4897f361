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
