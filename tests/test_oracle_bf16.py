"""Oracle pin: the fp32 -> bf16 round-to-nearest-even and bf16 -> fp32
widening, against torch's CPU casts (an independent implementation)."""
import numpy as np
import pytest
import torch


def _torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _compare(orc, bits: np.ndarray):
    x = bits.view(np.float32)
    got = orc.bf16_from_f32(x)
    want = _torch_bf16_bits(x)
    nan = np.isnan(x)
    # NaN stays NaN (any quiet payload); everything else bit-exact
    gn = got[nan]
    assert np.all((gn & 0x7f80) == 0x7f80) and np.all((gn & 0x007f) != 0)
    assert np.all((gn & 0x0040) != 0)
    bad = np.flatnonzero((got != want) & ~nan)
    assert bad.size == 0, [hex(int(bits[i])) for i in bad[:8]]


def test_special_values(orc):
    cases = {
        0x00000000: 0x0000, 0x80000000: 0x8000,   # +-0
        0x7f800000: 0x7f80, 0xff800000: 0xff80,   # +-inf
        0x7f7fffff: 0x7f80,                       # max finite rounds up to inf
        0x3f808000: 0x3f80,                       # tie, even neighbour below
        0x3f818000: 0x3f82,                       # tie, even neighbour above
        0x3f808001: 0x3f81,                       # just above the tie
        0x00000001: 0x0000,                       # smallest subnormal
        0x00008000: 0x0000,                       # subnormal tie to even (0)
        0x00018000: 0x0002,                       # subnormal tie to even (2)
    }
    for src, dst in cases.items():
        x = np.array([src], np.uint32).view(np.float32)
        assert int(orc.bf16_from_f32(x)[0]) == dst, hex(src)


def test_widening_exhaustive(orc):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = orc.f32_from_bf16(h)
    want = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_rounding_structured_sample(orc):
    """Every exponent, both signs, all 2^16 low halves for a spread of upper
    mantissa bits: covers every rounding case of every binade."""
    hi = np.arange(0, 1 << 16, 97, dtype=np.uint32)          # sign|exp|mant7 patterns
    lo = np.array([0, 1, 0x7fff, 0x8000, 0x8001, 0xffff], np.uint32)
    bits = (hi[:, None] << 16 | lo[None, :]).reshape(-1)
    _compare(orc, bits)
    rng = np.random.default_rng(5)
    _compare(orc, rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32))


@pytest.mark.slow
def test_rounding_exhaustive(orc):
    """All 2^32 binary32 patterns, in chunks."""
    chunk = 1 << 26
    for c in range((1 << 32) // chunk):
        bits = np.arange(c * chunk, (c + 1) * chunk, dtype=np.uint64).astype(np.uint32)
        _compare(orc, bits)
