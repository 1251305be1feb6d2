"""Exact-arithmetic helpers for pinning the oracle (tests only).

Written independently of the oracle's C code: rational arithmetic
(``fractions.Fraction``) and 60-digit ``decimal`` square roots, so that a slip
in the oracle's fp64 loop or its encoders shows up as a mismatch here.
"""
from __future__ import annotations

import decimal
from fractions import Fraction

# (fraction bits, minimum normal exponent, bias, all-ones exponent field)
FORMATS = {"bf16": (7, -126, 127, 0xFF), "fp16": (10, -14, 15, 0x1F),
           "fp32": (23, -126, 127, 0xFF)}
# Position of the sign bit.
SIGN_BIT = {"bf16": 15, "fp16": 15, "fp32": 31}

_CTX = decimal.Context(prec=60)


def decode_exact(dtype: str, bits: int) -> Fraction | None:
    """Bit pattern -> exact rational value (None for inf/NaN)."""
    mbits, emin, bias, emax_field = FORMATS[dtype]
    sign = -1 if bits >> SIGN_BIT[dtype] else 1
    field = (bits >> mbits) & emax_field
    frac = bits & ((1 << mbits) - 1)
    if field == emax_field:
        return None
    if field == 0:
        mag = Fraction(frac, 1) * Fraction(2) ** (emin - mbits)
    else:
        mag = Fraction((1 << mbits) + frac) * Fraction(2) ** (field - bias - mbits)
    return sign * mag


def round_exact(dtype: str, v: Fraction, negative_zero: bool = False) -> int:
    """Nearest representable value of ``dtype`` to the rational ``v``, ties to even."""
    mbits, emin, bias, emax_field = FORMATS[dtype]
    sign = (1 << SIGN_BIT[dtype]) if (v < 0 or (v == 0 and negative_zero)) else 0
    a = abs(v)
    if a == 0:
        return sign
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    units = a / Fraction(2) ** (e - mbits)
    n = units.numerator // units.denominator
    rem = units - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    hidden = 1 << mbits
    if n == 0:
        return sign
    if n >= 2 * hidden:
        n >>= 1
        e += 1
    if n < hidden:
        field = 0
    else:
        field = e + bias
        n -= hidden
    if field >= emax_field:
        return sign | (emax_field << mbits)
    return sign | (field << mbits) | n


def rmsnorm_row_exact(x: list[Fraction], w: list[Fraction], eps: Fraction, offset: Fraction):
    """One row: returns (r, [y_j]) as Fractions, exact or to 60 significant digits."""
    n = len(x)
    s = sum((xi * xi for xi in x), Fraction(0))
    ms_eps = s / n + eps
    d = _CTX.divide(decimal.Decimal(ms_eps.numerator), decimal.Decimal(ms_eps.denominator))
    if d == 0:
        return None, None
    root = _CTX.sqrt(d)
    # r is exact when ms_eps is a rational square; otherwise 60 significant digits.
    r_num, r_den = _sqrt_rational(ms_eps)
    if r_num is not None:
        r = Fraction(r_den, r_num)
    else:
        r = Fraction(_CTX.divide(decimal.Decimal(1), root))
    return r, [xi * r * (offset + wj) for xi, wj in zip(x, w)]


def _isqrt_exact(k: int):
    import math
    s = math.isqrt(k)
    return s if s * s == k else None


def _sqrt_rational(q: Fraction):
    a = _isqrt_exact(q.numerator)
    b = _isqrt_exact(q.denominator)
    if a is None or b is None:
        return None, None
    return a, b
