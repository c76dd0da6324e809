"""Pins of the oracle's number formats (E2M1, E4M3, bf16) against their definitions.

The values come from the format definitions (hand-written golden tables), not from the oracle.
"""
import math
import struct

import numpy as np
import pytest

import oracle
from conftest import read_table


def f32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0]


def f32_next(v, direction):
    """Next binary32 after v towards +inf (direction > 0) or towards 0 (direction < 0)."""
    return float(np.nextafter(np.float32(v), np.float32(np.inf if direction > 0 else 0.0)))


# ---------------------------------------------------------------------------------------
# E2M1
# ---------------------------------------------------------------------------------------
def test_e2m1_decode_table():
    for code, val in read_table("e2m1_values.txt"):
        got = oracle.e2m1_decode(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e2m1_encode_representable():
    for code, val in read_table("e2m1_values.txt"):
        assert oracle.e2m1_encode(val) == code, (code, val)


@pytest.mark.parametrize("mid,lo,hi", [(0.25, 0x0, 0x1), (0.75, 0x1, 0x2), (1.25, 0x2, 0x3),
                                       (1.75, 0x3, 0x4), (2.5, 0x4, 0x5), (3.5, 0x5, 0x6),
                                       (5.0, 0x6, 0x7)])
def test_e2m1_rounding_at_midpoints(mid, lo, hi):
    even = lo if lo % 2 == 0 else hi
    assert oracle.e2m1_encode(mid) == even
    assert oracle.e2m1_encode(-mid) == (even | 0x8)
    assert oracle.e2m1_encode(f32_next(mid, -1)) == lo
    assert oracle.e2m1_encode(f32_next(mid, +1)) == hi
    assert oracle.e2m1_encode(-f32_next(mid, +1)) == (hi | 0x8)


def test_e2m1_saturation_and_sign():
    assert oracle.e2m1_encode(6.0) == 0x7
    assert oracle.e2m1_encode(6.5) == 0x7
    assert oracle.e2m1_encode(1e30) == 0x7
    assert oracle.e2m1_encode(math.inf) == 0x7
    assert oracle.e2m1_encode(-7.0) == 0xF
    assert oracle.e2m1_encode(-math.inf) == 0xF
    assert oracle.e2m1_encode(0.0) == 0x0
    assert oracle.e2m1_encode(-0.0) == 0x8
    assert oracle.e2m1_encode(-1e-30) == 0x8
    assert oracle.e2m1_encode(1e-30) == 0x0


def test_e2m1_monotone_dense_sweep():
    """Encoding is monotone in the input and every code is the nearest grid value."""
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    xs = np.linspace(0, 7, 2801)
    prev = 0
    for x in xs:
        c = oracle.e2m1_encode(x)
        assert c >= prev
        prev = c
        d = np.abs(grid - f32(x))
        assert d[c] == d.min()


# ---------------------------------------------------------------------------------------
# E4M3
# ---------------------------------------------------------------------------------------
def test_e4m3_decode_table():
    for code, val in read_table("e4m3_values.txt"):
        got = oracle.e4m3_decode(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e4m3_all_finite_codes_roundtrip_and_monotone():
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
    assert vals[0x7E] == 448.0 and vals[1] == 2.0 ** -9
    for c in range(0x7F):
        assert oracle.e4m3_encode(vals[c]) == c
        if c:
            assert oracle.e4m3_encode(-vals[c]) == (0x80 | c)


def test_e4m3_midpoints_tie_to_even():
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    for c in range(0x7E):
        mid = 0.5 * (vals[c] + vals[c + 1])
        assert f32(mid) == mid
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even, (c, mid)
        assert oracle.e4m3_encode(f32_next(mid, -1)) == c
        assert oracle.e4m3_encode(f32_next(mid, +1)) == c + 1


def test_e4m3_saturation_subnormal_and_zero():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E          # beyond the largest finite: saturate
    assert oracle.e4m3_encode(1e9) == 0x7E
    assert oracle.e4m3_encode(math.inf) == 0x7E
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00     # tie between 0 and 2^-9 -> even (0)
    assert oracle.e4m3_encode(f32_next(2.0 ** -10, +1)) == 0x01
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02  # tie between 1 and 2 (x 2^-9) -> 2
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80


# ---------------------------------------------------------------------------------------
# bf16
# ---------------------------------------------------------------------------------------
@pytest.mark.parametrize("v,bits", [
    (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
    (1 + 2 ** -8, 0x3F80),            # tie -> even mantissa (0)
    (1 + 3 * 2 ** -8, 0x3F82),        # tie between ...81 and ...82 -> even
    (1 + 2 ** -8 + 2 ** -30, 0x3F81), # just past the tie
    (1.0 / 672.0, 0x3AC3),            # hand-computed: 195/128 * 2^-10
    (255.0 / 128.0 * 2.0 ** 127, 0x7F7F),  # largest finite bf16
    (2.0 ** 128, 0x7F80),             # overflow -> +inf
    (2.0 ** -133, 0x0001),            # smallest subnormal
    (2.0 ** -134, 0x0000),            # tie between 0 and the smallest subnormal -> 0
    (3 * 2.0 ** -134, 0x0002),        # tie between 1 and 2 subnormal quanta -> 2
])
def test_bf16_from_double(v, bits):
    assert oracle.bf16_from_double(v) == bits


def test_bf16_roundtrip_all_finite_patterns():
    for b in list(range(0, 0x7F80, 7)) + [0x7F7F, 0x0001, 0x8001, 0xFF7F]:
        assert oracle.bf16_from_double(oracle.bf16_to_double(b)) == b


def test_array_encoders_match_scalar():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 4,
                        np.array([0.0, -0.0, 0.25, 0.75, 5.0, 448.0, 1e-9, -1e30], np.float32)])
    assert oracle.e2m1_encode_array(v).tolist() == [oracle.e2m1_encode(float(x)) for x in v]
    w = np.abs(v) * 60
    assert oracle.e4m3_encode_array(w).tolist() == [oracle.e4m3_encode(float(x)) for x in w]


def test_encoders_terminate_outside_the_domain():
    # NaN is outside the method's domain (never produced from finite inputs); the oracle must
    # still return instead of searching forever.
    assert oracle.e2m1_encode(float("nan")) in range(16)
    assert oracle.e4m3_encode(float("nan")) in range(256)


def test_every_finite_e4m3_value_is_an_f16_value():
    """The dispatch kernels decode an E4M3 block scale through the hardware E4M3 -> f16 -> fp32
    conversions, which is exact only if every finite E4M3 value (448 down to the subnormal
    2^-9) is an f16 value.  f16 has 11 significant bits and normal exponents down to 2^-14, so
    the subnormals need the f16 subnormals (down to 2^-24)."""
    vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)], dtype=np.float64)
    assert vals[0] == 0.0 and vals.max() == 448.0 and vals[1] == 2.0 ** -9
    assert np.array_equal(vals.astype(np.float16).astype(np.float64), vals)
