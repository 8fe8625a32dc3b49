"""Exact binary-float rounding in pure Python (fractions), for pinning the oracle.

Independent of numpy: these helpers decide IEEE round-to-nearest-even by exact
rational arithmetic, so they can check numpy's float32 / float16 conversions and
the oracle's rounding decisions.
"""
from fractions import Fraction
import math
import struct


def round_binary(v: Fraction, mant_bits: int, min_exp: int, max_finite: Fraction) -> Fraction:
    """Round v to the nearest value of a binary format with `mant_bits` stored
    fraction bits and minimum normal exponent `min_exp`; ties to even.
    Returns +-inf (as float) on overflow."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # fix possible off-by-one of the float log2
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, min_exp)
    ulp = Fraction(2) ** (e - mant_bits)
    q = a / ulp
    fl = math.floor(q)
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * ulp
    # overflow threshold: halfway between max_finite and the next step
    if r > max_finite:
        return sign * float("inf")
    return sign * r


F16_MAX = Fraction(65504)
F32_MAX = Fraction(struct.unpack("<f", b"\xff\xff\x7f\x7f")[0])


def fl16(v: Fraction) -> Fraction:
    return round_binary(v, 10, -14, F16_MAX)


def fl32(v: Fraction) -> Fraction:
    return round_binary(v, 23, -126, F32_MAX)


def round_half_even(v: Fraction) -> int:
    fl = math.floor(v)
    rem = v - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return int(fl)
