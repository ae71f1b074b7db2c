"""Exact rational helpers used by the oracle pins (independent of numpy's
floating point): correct rounding of a rational to fp32 / BF16 and ulp sizes.
"""
from fractions import Fraction
import math
import struct


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def ulp_f32(q: Fraction) -> Fraction:
    """Spacing of fp32 numbers at |q| (normal range)."""
    a = abs(q)
    if a == 0:
        return Fraction(1, 2 ** 149)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # fix possible off-by-one of the float log
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return Fraction(2) ** (e - 23)


def round_to_f32(q: Fraction) -> Fraction:
    """Nearest fp32 value to the rational q, ties to even (normal range)."""
    if q == 0:
        return Fraction(0)
    u = ulp_f32(q)
    n = q / u                       # integer part is the significand count
    fl = math.floor(n)
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl * u


def round_to_bf16(q: Fraction) -> Fraction:
    """Nearest BF16 value to the rational q, ties to even (normal range):
    8 significant bits, spacing 2^(e-7) on [2^e, 2^(e+1))."""
    if q == 0:
        return Fraction(0)
    u = ulp_f32(q) * 2 ** 16
    n = q / u
    fl = math.floor(n)
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl * u
