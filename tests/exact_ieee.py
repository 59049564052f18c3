"""Exact IEEE-754 rounding from rational arithmetic (test helper).

An independent model of binary32 / bf16 arithmetic: every operation is done
exactly on Fractions and then rounded to the nearest representable value,
ties to even, following the IEEE-754 definition (normal and subnormal
ranges; overflow is not needed by the tests and raises).  It shares nothing
with the oracle or the CUDA library, so agreement with it is a real check.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def _round_to_format(q: Fraction, mant_bits: int, emin: int, emax: int) -> Fraction:
    """Round q to a binary format with `mant_bits` significand bits (incl. the
    implicit one), minimum normal exponent emin, maximum exponent emax."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = -q if q < 0 else q
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)  # subnormal range shares the spacing of the smallest normal binade
    spacing = Fraction(2) ** (e - (mant_bits - 1))
    m = a / spacing
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    r = lo * spacing
    if r >= Fraction(2) ** (emax + 1):
        raise OverflowError("result overflows the format")
    return sign * r


def rn_f32(q: Fraction) -> Fraction:
    return _round_to_format(Fraction(q), 24, -126, 127)


def rn_bf16(q: Fraction) -> Fraction:
    return _round_to_format(Fraction(q), 8, -126, 127)


def frac(x) -> Fraction:
    """Exact value of a float32 / float64 / int."""
    return Fraction(float(x)) if not isinstance(x, Fraction) else x


def to_f32(q: Fraction) -> np.float32:
    v = np.float32(float(q))
    assert Fraction(float(v)) == q, "value is not a binary32 number"
    return v


def add(a, b):
    return rn_f32(frac(a) + frac(b))


def sub(a, b):
    return rn_f32(frac(a) - frac(b))


def mul(a, b):
    return rn_f32(frac(a) * frac(b))


def div(a, b):
    return rn_f32(frac(a) / frac(b))


def bf16_bits(q: Fraction) -> int:
    """bf16 bit pattern of a value that is exactly a bf16 number."""
    v = np.array([float(q)], dtype=np.float32).view(np.uint32)[0]
    assert v & 0xFFFF == 0, "value is not a bf16 number"
    return int(v >> 16)


def bf16_value(bits: int) -> Fraction:
    return Fraction(float(np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0]))
