"""The encoder's scale quotient amax / c (c = 127 for q8_0, 7 for q4s) is formed without a
division: q0 = fp32(amax * r) with r = fp32(1 / c), e = fma(-q0, c, amax), q1 = fma(e, r, q0).
The codec contract wants the correctly rounded fp32 quotient, so this checks, with exact
rational arithmetic, that q1 equals it for every positive finite bf16 amax (the only values
amax takes: the maximum magnitude of bf16 inputs)."""

import struct
from fractions import Fraction

import pytest


def rn32(x: Fraction) -> Fraction:
    """x rounded to the nearest fp32 value (ties to even), normal and subnormal range."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    if Fraction(2) ** (e + 1) <= x:
        e += 1
    e = max(e, -126)
    scale = Fraction(2) ** (e - 23)
    m = x / scale
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * scale


def bf16_value(bits: int) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<I", bits << 16))[0])


@pytest.mark.parametrize("c", [127, 7])
def test_fma_corrected_quotient_is_correctly_rounded(c):
    r = rn32(Fraction(1, c))
    mismatches = []
    for bits in range(1, 0x7F80):                 # every positive finite bf16 value
        a = bf16_value(bits)
        q0 = rn32(a * r)
        e = rn32(a - q0 * c)                      # fma(-q0, c, a)
        q1 = rn32(q0 + e * r)                     # fma(e, r, q0)
        if q1 != rn32(a / c):
            mismatches.append(bits)
    assert not mismatches, [hex(b) for b in mismatches[:5]]


def test_rn32_rounds_ties_to_even():
    # 1 + 2^-24 is halfway between 1 and the next fp32: ties to the even one (1); 1 + 3 * 2^-24
    # is halfway between 1 + 2^-23 (odd) and 1 + 2^-22 (even)
    assert rn32(1 + Fraction(1, 2 ** 24)) == 1
    assert rn32(1 + Fraction(3, 2 ** 24)) == 1 + Fraction(1, 2 ** 22)
    assert rn32(Fraction(1, 2 ** 149)) == Fraction(1, 2 ** 149)            # smallest subnormal
    assert rn32(Fraction(1, 2 ** 150)) == 0                               # halfway to it: even (0)
