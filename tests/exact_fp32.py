"""Exact IEEE binary32 rounding of rational numbers, for pinning the oracle.

The oracle takes its fp32 steps with numpy float32 arithmetic. The pins in
tests/ recompute the same quantities from their definitions with exact
rationals (``fractions.Fraction``) and an independent round-to-nearest-even
to binary32 written here from the format's definition: a 24-bit significand,
normal exponents down to 2**-126, subnormal spacing 2**-149. Nothing here is
shared with the oracle or the CUDA library.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

_MIN_EXP = -149          # spacing of binary32 subnormals
_MAX_FINITE = Fraction((1 << 24) - 1) * Fraction(2) ** 104


def _pow2(e: int) -> Fraction:
    return Fraction(1 << e) if e >= 0 else Fraction(1, 1 << -e)


def floor_log2(a: Fraction) -> int:
    """e with 2**e <= a < 2**(e+1), for a > 0."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if _pow2(e) > a:
        e -= 1
    elif _pow2(e + 1) <= a:
        e += 1
    return e


def rne32(x) -> Fraction:
    """x (any rational) rounded to the nearest binary32 value, ties to the
    even significand. Raises on overflow, which no caller here reaches."""
    x = Fraction(x)
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = -x if x < 0 else x
    q = max(floor_log2(a) - 23, _MIN_EXP)        # exponent of one unit in the last place
    scaled = a / _pow2(q)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = Fraction(n) * _pow2(q)
    if r > _MAX_FINITE:
        raise OverflowError("beyond binary32")
    return sign * r


def rne_int(x: Fraction) -> int:
    """Nearest integer, ties to even."""
    n = x.numerator // x.denominator
    rem = x - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n


def f32(v) -> Fraction:
    """The exact value of a float32 (or a Python float that is one)."""
    return Fraction(float(np.float32(v)))


def as_f32(x: Fraction) -> np.float32:
    """A rational that is a binary32 value, as np.float32 (checked)."""
    v = np.float32(float(x))
    assert Fraction(float(v)) == x, "not a binary32 value"
    return v
