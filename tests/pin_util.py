"""Exact-arithmetic helpers for the oracle pins (independent of the oracle).

Everything here works on Python ``fractions.Fraction`` values, so a pin
computed with these helpers does not share any floating-point step with the
oracle it checks.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def f32_round(fr: Fraction) -> np.float32:
    """Round an exact rational to the nearest float32, ties to even."""
    c = np.float32(float(fr))  # within one float32 step of the answer
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        if not np.isfinite(cand):
            continue
        err = abs(Fraction(float(cand)) - fr)
        key = (err, int(np.array(cand, np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def round_half_even(fr: Fraction) -> int:
    """Python's round() on a Fraction rounds half to even."""
    return round(fr)


def e4m3_finite_values():
    """All finite non-negative e4m3fn values with their codes, from the
    golden table's format definition (bias 7, 3 mantissa bits, subnormals
    m * 2^-9, top code 0x7F is NaN)."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        v = Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        vals.append((v, code))
    return vals


_E4M3 = e4m3_finite_values()


def e4m3_round_bruteforce(x: float) -> int:
    """Encode x as e4m3fn by exhaustive search: the nearest finite value,
    ties to the even code, magnitudes past 448 saturating to 448."""
    fr = Fraction(float(x))
    sign = 0x80 if math.copysign(1.0, float(x)) < 0 else 0
    a = abs(fr)
    if a >= 448:
        return sign | 0x7E
    best = None
    for v, code in _E4M3:
        key = (abs(v - a), code & 1)
        if best is None or key < best[0]:
            best = (key, code)
    return sign | best[1]
