"""e5m2 codec (oracle; test infrastructure only).

[WT] sec. 2.1 (format table) and [PT] "E4M3 vs E5M2": e5m2 has 1 sign, 5 exponent and 2
mantissa bits, reaches about 57344 and is the format kept for gradients (wider range, less
precision).  With exponent bias 15 the largest finite value 1.75 * 2^15 = 57344 is S.11110.11,
so the top exponent 11111 holds no finite values: like IEEE binary formats it encodes
infinities (mantissa 0) and NaN (mantissa 1..3).  That is the OCP "E5M2" format:

    code (s, E, m):  E == 0         -> (-1)^s * m * 2^-16              (subnormal)
                     E == 31, m == 0 -> (-1)^s * inf
                     E == 31, m != 0 -> NaN
                     otherwise      -> (-1)^s * (1 + m/4) * 2^(E-15)

Encoding follows the e4m3 rules (e4m3.py): the nearest finite value, ties to the even code,
magnitudes above 57344 saturate to 57344 (satfinite), the sign is kept, NaN maps to 0x7F.
"""

from __future__ import annotations

import numpy as np

E5M2_MAX = 57344.0


def _code_value(code: int) -> float:
    s = (code >> 7) & 1
    e = (code >> 2) & 0x1F
    m = code & 0x3
    sign = -1.0 if s else 1.0
    if e == 0x1F:
        return sign * float("inf") if m == 0 else float("nan")
    if e == 0:
        return sign * m * 2.0 ** -16
    return sign * (1.0 + m / 4.0) * 2.0 ** (e - 15)


def e5m2_decode_table() -> np.ndarray:
    """float64 [256]: value of every code."""
    return np.array([_code_value(c) for c in range(256)], dtype=np.float64)


_TABLE = e5m2_decode_table()
_POS = _TABLE[:0x7C].copy()  # non-negative finite magnitudes, codes 0x00..0x7B, strictly increasing


def e5m2_decode(codes: np.ndarray) -> np.ndarray:
    """uint8 codes -> float64 values."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def e5m2_encode(v: np.ndarray) -> np.ndarray:
    """float32/float64 values -> uint8 e5m2 codes (RN ties-to-even, satfinite)."""
    v = np.asarray(v, dtype=np.float64)
    nan = np.isnan(v)
    mag = np.where(nan, 0.0, np.abs(v))
    hi = np.minimum(np.searchsorted(_POS, mag, side="left"), 0x7B)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = mag - _POS[lo], _POS[hi] - mag
    code = np.where((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)), hi, lo)
    code = np.where(mag >= _POS[0x7B], 0x7B, code)  # satfinite
    out = (code | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), out).astype(np.uint8)
