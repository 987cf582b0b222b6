"""Exact-rational helpers for the oracle pins (test-only).

Independent of the oracle: rounding is done from the definition (nearest
representable value, ties to the even significand) on ``fractions.Fraction``,
not by numpy arithmetic.
"""

from fractions import Fraction

import numpy as np


def f32_rn(x: Fraction) -> np.float32:
    """Round an exact rational to the nearest binary32 (ties to even)."""
    if x == 0:
        return np.float32(0.0)
    c = np.float32(float(x))  # within one ulp of the answer
    cands = {c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))}
    best = None
    for v in cands:
        if not np.isfinite(v):
            continue
        d = abs(Fraction(float(v)) - x)
        key = (d, int(np.array(v, dtype=np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, v)
    return np.float32(best[1])


def bf16_rn_bits(x: np.float32) -> int:
    """Round a binary32 value to bf16 (8-bit significand), ties to even; returns bits."""
    b = int(np.array(x, dtype=np.float32).view(np.uint32))
    lo = b & 0xFFFF0000  # truncation toward zero
    hi = lo + 0x10000  # next bf16 away from zero
    xv = Fraction(float(x))
    vlo = Fraction(float(np.array(lo, dtype=np.uint32).view(np.float32)))
    vhi = Fraction(float(np.array(hi & 0xFFFFFFFF, dtype=np.uint32).view(np.float32)))
    dlo, dhi = abs(xv - vlo), abs(vhi - xv)
    if dlo < dhi or (dlo == dhi and ((lo >> 16) & 1) == 0):
        return lo >> 16
    return (hi >> 16) & 0xFFFF


def e4m3_values():
    """{code: Fraction} for the 127 non-negative finite codes, from the closed form."""
    out = {}
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        out[c] = Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return out


_E4M3 = e4m3_values()


def e4m3_nearest(y: Fraction, negative: bool) -> int:
    """Nearest e4m3 code by exhaustive search, ties to even, saturating at 448."""
    mag = abs(y)
    best = None
    for c, v in _E4M3.items():
        d = abs(mag - v)
        if best is None or (d, c % 2) < best[0]:
            best = ((d, c % 2), c)
    return best[1] | (0x80 if negative else 0)


def e4m3_value(code: int) -> Fraction:
    v = _E4M3[code & 0x7F]
    return -v if code & 0x80 else v
