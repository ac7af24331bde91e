"""Exact (rational) helpers used to pin the oracle.  Nothing here is shared with
the oracle or the CUDA path: bf16 rounding is done by brute force against the
sorted table of every finite bf16 value, sums are ``fractions.Fraction``, and
square roots are ``decimal`` at 60 digits.
"""
from __future__ import annotations

import decimal
from fractions import Fraction

import numpy as np

_ALL = np.arange(1 << 16, dtype=np.uint32)
with np.errstate(invalid="ignore"):
    _VALS = (_ALL << np.uint32(16)).view(np.float32).astype(np.float64)
_FINITE = np.isfinite(_VALS)
# non-negative finite bf16 values, ascending, with their bit patterns
_POS_BITS = np.arange(0x0000, 0x7F80, dtype=np.uint32)  # +0 .. largest finite
_POS_VALS = (_POS_BITS << np.uint32(16)).view(np.float32).astype(np.float64)
BF16_MAX = float(_POS_VALS[-1])


def bf16_value(bits: int) -> float:
    return float(_VALS[int(bits)])


def bf16_round_exact(v) -> tuple[int, bool]:
    """Round an exact value (Fraction/int/float) to bf16, ties to even.

    Returns (bits, near_tie) where near_tie says the value is within 1e-12
    (relative) of the midpoint between its two bf16 neighbours, so a binary64
    computation may legitimately land on either side.
    """
    f = Fraction(v)
    sign = 0x8000 if f < 0 else 0
    a = -f if f < 0 else f
    if a == 0:
        return sign, False
    af = float(a)
    i = int(np.searchsorted(_POS_VALS, af, side="right")) - 1
    i = max(0, min(i, _POS_VALS.size - 1))
    # adjust so that lo <= a < hi exactly
    while i > 0 and Fraction(_POS_VALS[i]) > a:
        i -= 1
    while i + 1 < _POS_VALS.size and Fraction(_POS_VALS[i + 1]) <= a:
        i += 1
    lo = Fraction(_POS_VALS[i])
    if i + 1 >= _POS_VALS.size:
        # above the largest finite value: overflow threshold is max + half ulp
        half_ulp = (lo - Fraction(_POS_VALS[i - 1])) / 2
        if a >= lo + half_ulp:
            return sign | 0x7F80, False
        return sign | int(_POS_BITS[i]), False
    hi = Fraction(_POS_VALS[i + 1])
    if a == lo:
        return sign | int(_POS_BITS[i]), False
    d_lo, d_hi = a - lo, hi - a
    mid = (lo + hi) / 2
    near = abs(a - mid) <= mid * Fraction(1, 10**12)
    if d_lo < d_hi:
        return sign | int(_POS_BITS[i]), near
    if d_hi < d_lo:
        return sign | int(_POS_BITS[i + 1]), near
    even = i if (int(_POS_BITS[i]) & 1) == 0 else i + 1
    return sign | int(_POS_BITS[even]), True


def dec_sqrt_recip(x: Fraction, digits: int = 60) -> Fraction:
    """1/sqrt(x) to about ``digits`` significant digits, as a Fraction."""
    with decimal.localcontext() as ctx:
        ctx.prec = digits
        d = decimal.Decimal(x.numerator) / decimal.Decimal(x.denominator)
        return Fraction(decimal.Decimal(1) / d.sqrt())


def rel_close(a: float, b: Fraction | float, rel: float) -> bool:
    b = float(b)
    return abs(a - b) <= rel * max(abs(b), 1e-300)


def f32_round_exact(v) -> Fraction:
    """Round an exact value to IEEE binary32, ties to even, by integer
    arithmetic on the Fraction (normal and subnormal range; no overflow
    handling: the callers stay far below 2^128)."""
    f = Fraction(v)
    if f == 0:
        return Fraction(0)
    sign = -1 if f < 0 else 1
    a = -f if f < 0 else f
    # e = floor(log2 a)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    m = a / ulp
    r = m.numerator // m.denominator
    rem = m - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    return sign * r * ulp


def f32_sqrt_exact(v: Fraction, digits: int = 60) -> Fraction:
    """The binary32 rounding of sqrt(v) (v >= 0), from a 60-digit decimal
    square root (a square root is never exactly halfway between two binary32
    values, so the decimal precision decides every case)."""
    with decimal.localcontext() as ctx:
        ctx.prec = digits
        d = decimal.Decimal(v.numerator) / decimal.Decimal(v.denominator)
        return f32_round_exact(Fraction(d.sqrt()))
