"""Exact rational arithmetic with IEEE round-to-nearest-even into a binary
format, used by the tests as a brute-force reference that shares nothing with
the oracle's numpy/bit-trick arithmetic.

A binary format with p significand bits and minimum normal exponent emin
represents values m * 2**(e - p + 1), |m| < 2**p, e >= emin (subnormals at
e = emin).  round_to() returns the nearest such value to a Fraction, ties to the
even significand, and +-inf past the largest finite value (IEEE 754 section 4.3.1,
roundTiesToEven).
"""
from fractions import Fraction  # noqa: F401  (re-exported for tests)
import math
import struct

import numpy as np

INF = float("inf")


def _floor_log2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_to(q, p: int, emin: int, emax: int):
    """Round Fraction q to the binary format (p, emin, emax); returns a
    Fraction or +-inf (a float)."""
    if isinstance(q, float):
        return q
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = max(_floor_log2(a), emin)
    ulp = Fraction(2) ** (e - p + 1)
    m = a / ulp
    n = math.floor(m)
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * ulp
    # the largest finite value is (2 - 2**(1-p)) * 2**emax; anything that
    # rounds past it is an overflow
    if r >= Fraction(2) ** (emax + 1):
        return sign * INF
    return sign * r


def f32(q):
    return round_to(q, 24, -126, 127)


def bf16(q):
    return round_to(q, 8, -126, 127)


def add(a, b):
    """Exact sum of two values that may be +-inf (inf + -inf is not used)."""
    if isinstance(a, float) or isinstance(b, float):
        return a if isinstance(a, float) else b
    return a + b


def mul(a, b):
    if isinstance(a, float) or isinstance(b, float):
        return math.copysign(INF, (a if isinstance(a, float) else float(a)) *
                             (b if isinstance(b, float) else float(b)))
    return a * b


def of_f32(x) -> Fraction:
    v = float(np.float32(x))
    return v if math.isinf(v) else Fraction(v)


def of_bf16_bits(b: int):
    v = struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]
    return v if math.isinf(v) else Fraction(v)


def same(a, b) -> bool:
    if isinstance(a, float) or isinstance(b, float):
        return float(a) == float(b)
    return a == b
