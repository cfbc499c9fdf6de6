"""Pins of the oracle's bf16 decoding against what the bfloat16 format fixes.

Every input the tests generate and every result read back from the GPU reaches
the oracle through `bf16_to_f64`, so a wrong shift, sign or byte order there
would be blamed on the kernels.  bfloat16 is the top half of an IEEE-754
binary32: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.  The
checks below use that definition directly, not the oracle's widening.
"""
import math
import struct

import numpy as np
import pytest

from oracle import lora_oracle as O

# NaN patterns raise numpy's cast warning when widened; they are checked below
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

# bit pattern -> value, each worked out by hand from sign / exponent / fraction
KNOWN = [
    (0x0000, 0.0),
    (0x3F80, 1.0),                            # exponent 127, fraction 0
    (0xBF80, -1.0),
    (0x4000, 2.0),
    (0xC000, -2.0),
    (0x3F00, 0.5),
    (0x4049, 3.140625),                       # 2 * (1 + 73/128)
    (0x4120, 10.0),                           # 8 * (1 + 32/128)
    (0x3DCD, 0.10009765625),                  # 2^-4 * (1 + 77/128)
    (0x0080, 2.0 ** -126),                    # smallest normal
    (0x0001, 2.0 ** -133),                    # smallest subnormal: 1/128 * 2^-126
    (0x007F, 127 * 2.0 ** -133),              # largest subnormal
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),  # largest finite
    (0xFF7F, -(2.0 - 2.0 ** -7) * 2.0 ** 127),
]


@pytest.mark.parametrize("bits,value", KNOWN)
def test_known_patterns(bits, value):
    got = O.bf16_to_f64(np.array([bits], dtype=np.uint16))[0]
    assert got == value, (hex(bits), got, value)


def test_signed_zero_and_infinities_and_nan():
    v = O.bf16_to_f64(np.array([0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1], dtype=np.uint16))
    assert v[0] == 0.0 and math.copysign(1.0, v[0]) == -1.0
    assert v[1] == math.inf and v[2] == -math.inf
    assert math.isnan(v[3]) and math.isnan(v[4])


def _decode_by_fields(b: int) -> float:
    """Value of one bf16 pattern from its sign, exponent and fraction fields."""
    sign = -1.0 if b >> 15 else 1.0
    e = (b >> 7) & 0xFF
    f = b & 0x7F
    if e == 0xFF:
        return sign * math.inf if f == 0 else math.nan
    if e == 0:
        return sign * f * 2.0 ** -133
    return sign * (1.0 + f / 128.0) * 2.0 ** (e - 127)


def test_every_pattern_against_the_field_definition():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = O.bf16_to_f64(bits)
    want = np.array([_decode_by_fields(int(b)) for b in range(65536)])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # sign bit kept on zeros too
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_every_pattern_against_a_big_endian_binary32():
    # the pattern is the high two bytes of a binary32; decode those four bytes
    # with the struct module (its own IEEE decoder, not numpy's view)
    for b in range(0, 65536, 7):
        ref = struct.unpack(">f", bytes([b >> 8, b & 0xFF, 0, 0]))[0]
        got = O.bf16_to_f64(np.array([b], dtype=np.uint16))[0]
        if math.isnan(ref):
            assert math.isnan(got)
        else:
            assert got == ref, hex(b)


def test_shape_and_dtype_kept():
    bits = np.array([[0x3F80, 0x4000], [0xBF80, 0x0000]], dtype=np.uint16)
    v = O.bf16_to_f64(bits)
    assert v.dtype == np.float64 and v.shape == (2, 2)
    assert v.tolist() == [[1.0, 2.0], [-1.0, 0.0]]
