"""Exact-arithmetic helpers for pinning the oracle (tests only).

Rational arithmetic with ``fractions.Fraction`` plus a round-to-nearest-even
to binary32 written from the IEEE-754 definition.  Independent of the oracle's
C code: nothing here is shared with it.
"""
from fractions import Fraction
import math

import numpy as np


def f32_to_frac(x) -> Fraction:
    return Fraction(float(np.float32(x)))  # every fp32 value is exact in fp64


def _rn_int_even(q: Fraction) -> int:
    # Python's round() on a Fraction rounds halves to even
    return round(q)


def rn_binary(q: Fraction, mant_bits: int, emin: int, emax: int) -> float:
    """Round rational q to the nearest value of a binary format with
    ``mant_bits`` significand bits (incl. the implicit one), minimum normal
    exponent ``emin`` and maximum exponent ``emax``; ties to even."""
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(q)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - (mant_bits - 1))
    n = _rn_int_even(a / ulp)
    v = n * ulp
    if v >= Fraction(2) ** (emax + 1):
        return sign * math.inf
    return sign * float(v)


def rn_f32(q: Fraction) -> np.float32:
    return np.float32(rn_binary(q, 24, -126, 127))


def rn_bf16(q: Fraction) -> np.float32:
    return np.float32(rn_binary(q, 8, -126, 127))
