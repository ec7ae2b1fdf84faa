"""Pins of the oracle's bf16 -> float64 widening.

bfloat16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent
bits (bias 127), 7 mantissa bits.  The values below follow from that format
alone; the second test compares against torch's own bfloat16 type, an
independent implementation of the same format.
"""
import numpy as np
import pytest

from oracle.bf16 import widen

# (bits, value fixed by the format)
CASES = [
    (0x0000, 0.0),
    (0x3F80, 1.0),                          # sign 0, exponent 127, mantissa 0
    (0xC000, -2.0),                         # sign 1, exponent 128
    (0x3FC0, 1.5),                          # mantissa 0b1000000 = 1/2
    (0x4049, 3.140625),                     # 2 * (1 + 73/128)
    (0x0001, 2.0 ** -133),                  # smallest subnormal: 2^-126 * 2^-7
    (0x0080, 2.0 ** -126),                  # smallest normal
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),   # largest finite
    (0xFF80, -np.inf),
    (0x7F80, np.inf),
]


@pytest.mark.parametrize("bits,value", CASES)
def test_explicit_bit_patterns(bits, value):
    got = widen(np.array([bits], dtype=np.uint16))
    assert got.dtype == np.float64
    assert got[0] == value


def test_negative_zero_keeps_its_sign():
    got = widen(np.array([0x8000], dtype=np.uint16))[0]
    assert got == 0.0 and np.signbit(got)


def test_nan_patterns_stay_nan():
    got = widen(np.array([0x7FC0, 0xFFC1], dtype=np.uint16))
    assert np.isnan(got).all()


def test_matches_torch_bfloat16_on_random_patterns():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=200_000, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = widen(bits)
    both_nan = np.isnan(want) & np.isnan(got)
    assert np.array_equal(np.where(both_nan, 0.0, got), np.where(both_nan, 0.0, want))
    # signed zeros match too
    assert np.array_equal(np.signbit(got[~both_nan]), np.signbit(want[~both_nan]))


def test_shape_is_kept():
    bits = np.arange(24, dtype=np.uint16).reshape(2, 3, 4) + 0x3F80
    assert widen(bits).shape == (2, 3, 4)
