"""Exact rational arithmetic with IEEE-754 binary32 round-to-nearest-even.

Used to pin the oracle's floating point independently of any C compiler or
FPU: every value is a Python Fraction and the rounding to float32 is done
with integer arithmetic written here.
"""
from fractions import Fraction

import numpy as np

_EMIN = -126          # smallest normal exponent of binary32
_P = 24               # significand bits of binary32


def round_f32(x: Fraction) -> np.float32:
    """Round a rational to the nearest binary32 value, ties to even."""
    if x == 0:
        return np.float32(0.0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    q_exp = max(e, _EMIN) - (_P - 1)          # exponent of one unit in the last place
    quantum = Fraction(2) ** q_exp
    t = a / quantum
    n = t.numerator // t.denominator
    rem = t - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    value = n * quantum
    if value >= Fraction(2) ** 128:
        return np.float32(sign * np.inf)
    return np.float32(sign * float(value))   # exact: n < 2^25, power of two scale


def F(v) -> Fraction:
    """Exact rational value of a float32 (or float) number."""
    return Fraction(float(np.float32(v)))


def s32_exact(q, x) -> np.float32:
    """((dx*dx + dy*dy) + dz*dz) with one binary32 rounding per operation."""
    d = [round_f32(F(q[i]) - F(x[i])) for i in range(3)]
    sq = [round_f32(F(v) * F(v)) for v in d]
    sxy = round_f32(F(sq[0]) + F(sq[1]))
    return round_f32(F(sxy) + F(sq[2]))


def s32_fma_variant(q, x) -> np.float32:
    """The same sum contracted to fma(dz, dz, fma(dy, dy, dx*dx)) (a wrong reading)."""
    d = [round_f32(F(q[i]) - F(x[i])) for i in range(3)]
    xx = round_f32(F(d[0]) * F(d[0]))
    t = round_f32(F(d[1]) * F(d[1]) + F(xx))
    return round_f32(F(d[2]) * F(d[2]) + F(t))


def s_real(q, x) -> Fraction:
    """The real squared distance of the float32 inputs, exactly."""
    return sum((F(q[i]) - F(x[i])) ** 2 for i in range(3))


def sd_exact(q, x) -> np.float32:
    """Dimension-by-dimension sum of squared differences, accumulated in
    increasing dimension, one binary32 rounding per operation."""
    s = np.float32(0.0)
    for i in range(len(q)):
        t = round_f32(F(q[i]) - F(x[i]))
        t2 = round_f32(F(t) * F(t))
        s = round_f32(F(s) + F(t2))
    return s


def fma_exact(a, b, c) -> np.float32:
    """fl32(a*b + c) with a single rounding (the FMA instruction), exactly."""
    return round_f32(F(a) * F(b) + F(c))


def fma_f32(a, b, c) -> np.ndarray:
    """Vectorised fl32(a*b + c) with one rounding, for float32 arrays.

    a*b is exact in float64 (48 significant bits, and every float32 product
    lies inside float64's normal range).  A two-sum gives the exact sum as
    hi + lo with hi = fl64(a*b + c).  Rounding hi to float32 then gives the
    correctly rounded result except when hi sits exactly on a midpoint of two
    float32 neighbours while lo != 0: a float64 value strictly between the
    exact sum and hi would be nearer the sum than hi is.  That case is
    decided by the sign of lo.  Checked against ``fma_exact`` in the tests.
    """
    a = np.asarray(a, np.float32).astype(np.float64)
    b = np.asarray(b, np.float32).astype(np.float64)
    c = np.asarray(c, np.float32).astype(np.float64)
    p = a * b
    with np.errstate(invalid="ignore", over="ignore"):
        hi = p + c
        bb = hi - p
        lo = (p - (hi - bb)) + (c - bb)
        r = hi.astype(np.float32)
        r64 = r.astype(np.float64)
        toward = np.where(hi > r64, np.inf, -np.inf).astype(np.float32)
        other = np.nextafter(r, toward)
        mid = (r64 + other.astype(np.float64)) * 0.5
        fix = np.isfinite(hi) & (r64 != hi) & (hi == mid) & (lo != 0)
    if fix.any():
        up = lo > 0
        hi_side = np.where(r64 > other.astype(np.float64), r, other)
        lo_side = np.where(r64 > other.astype(np.float64), other, r)
        r = np.where(fix, np.where(up, hi_side, lo_side), r)
    return r.astype(np.float32)
