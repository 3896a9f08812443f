"""Exact IEEE 754 binary32 arithmetic on rationals, for pinning the oracle by brute force.

Independent of the oracle: it does not call fmaf or any float32 hardware operation. A float32 value is turned into
an exact Fraction, the operation is carried out exactly, and the result is rounded to binary32 by our own
round-to-nearest-ties-to-even (normal and subnormal ranges, overflow to infinity), with IEEE 754-2008 rules for
signed zeros, infinities and NaN (clauses 6.1-6.3 and 7.2: 0 * inf and inf - inf are invalid and give NaN; an exact
zero sum of operands of opposite sign is +0 under round-to-nearest).
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

_EMIN = -126
_P = 24
_MAX_EXP = 127


def f32_to_frac(v) -> Fraction:
    return Fraction(float(np.float32(v)))


def _sign(v) -> int:
    return -1 if math.copysign(1.0, float(v)) < 0 else 1


def round_f32(q: Fraction, zero_sign: int = 1) -> np.float32:
    """Round the exact rational q to binary32 (round to nearest, ties to even). zero_sign is used when q == 0."""
    if q == 0:
        return np.float32(0.0) if zero_sign > 0 else np.float32(-0.0)
    s = -1 if q < 0 else 1
    a = -q if q < 0 else q
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, _EMIN)
    quantum = Fraction(2) ** (e - (_P - 1))
    m = a / quantum
    fl = m.numerator // m.denominator
    r = m - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * quantum
    if val >= Fraction(2) ** (_MAX_EXP + 1):
        return np.float32(np.inf) if s > 0 else np.float32(-np.inf)
    if val == 0:   # underflow of a nonzero value: a zero with the value's sign
        return np.float32(0.0) if s > 0 else np.float32(-0.0)
    f = float(val) * s          # val has <= 24 significant bits and is in float32 range: exact as a float64
    return np.float32(f)


def fma32(a, b, c) -> np.float32:
    """IEEE binary32 fused multiply-add a*b + c with a single rounding."""
    a, b, c = float(np.float32(a)), float(np.float32(b)), float(np.float32(c))
    if math.isnan(a) or math.isnan(b) or math.isnan(c):
        return np.float32(np.nan)
    if (math.isinf(a) and b == 0) or (math.isinf(b) and a == 0):
        return np.float32(np.nan)
    psign = _sign(a) * _sign(b)
    pinf = math.isinf(a) or math.isinf(b)
    if pinf and math.isinf(c):
        if psign != _sign(c):
            return np.float32(np.nan)
        return np.float32(np.inf * psign)
    if pinf:
        return np.float32(np.inf * psign)
    if math.isinf(c):
        return np.float32(c)
    prod = f32_to_frac(a) * f32_to_frac(b)
    tot = prod + f32_to_frac(c)
    if tot == 0:
        # exact zero: the sign of two zero addends of the same sign, else +0 (round to nearest)
        if prod == 0 and c == 0 and psign == _sign(c):
            return round_f32(Fraction(0), psign)
        return round_f32(Fraction(0), 1)
    return round_f32(tot)


def add32(a, b) -> np.float32:
    """IEEE binary32 a + b, one rounding (a*1 + b fused is the same operation)."""
    return fma32(a, np.float32(1.0), b)


def chain_element(xcol, dcol, u) -> np.float32:
    """The step update of one element written with exact arithmetic: acc = +0; acc = fma(x_j, d_j, acc) for j in
    order; result = u + acc."""
    acc = np.float32(0.0)
    for a, b in zip(xcol, dcol):
        acc = fma32(a, b, acc)
    return add32(u, acc)
