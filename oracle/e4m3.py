"""e4m3 codec and bf16 rounding (oracle; test infrastructure only).

[WT] sec. 2.1 (format table): e4m3 has 1 sign, 4 exponent and 3 mantissa bits
and a largest finite value of about 448.  [PT] "E4M3 vs E5M2" section: the
e4m3 range is +-448.  Those two facts fix the variant: with exponent bias 7 the
code S.1111.111 cannot be finite (it would be 480), so the top exponent keeps
finite values for mantissas 0..6 and only S.1111.111 is NaN; there are no
infinities.  That is the OCP "e4m3fn" format:

    code (s, E, m):  E == 0          -> (-1)^s * m * 2^-9           (subnormal)
                     E == 15, m == 7 -> NaN
                     otherwise       -> (-1)^s * (1 + m/8) * 2^(E-7)

Encoding rounds to the nearest representable value ([EX] sec. 5.1: the default
rounding is round-to-nearest; the pages leave the tie rule open and the oracle
takes ties-to-even, the IEEE default), saturates magnitudes above 448 to 448
(satfinite: [WT] sec. 2.1 and 5.2 warn that unscaled overflow gives NaN; with
amax scaling only the rounding edge can exceed 448), keeps the sign (so -0.0 and
negative values that round to zero give 0x80) and maps NaN to 0x7F.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _code_value(code: int) -> float:
    """Value of one e4m3 code, from the closed form above."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    sign = -1.0 if s else 1.0
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_decode_table() -> np.ndarray:
    """float64 [256]: value of every code."""
    return np.array([_code_value(c) for c in range(256)], dtype=np.float64)


_TABLE = e4m3_decode_table()
# Non-negative finite magnitudes, indexed by code 0x00..0x7E.  They increase
# strictly with the code, so a position in this array is the code itself.
_POS = _TABLE[:0x7F].copy()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """uint8 codes -> float64 values."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float32/float64 values -> uint8 e4m3 codes (RN ties-to-even, satfinite).

    Nearest-value search over the 127 non-negative finite codes (a sorted-table
    search), the tie between two neighbours going to the even code (the even
    mantissa), then the sign bit.
    """
    v = np.asarray(v, dtype=np.float64)
    mag = np.abs(v)
    nan = np.isnan(v)
    mag = np.where(nan, 0.0, mag)
    hi = np.searchsorted(_POS, mag, side="left")  # first code with value >= mag
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _POS[lo]
    d_hi = _POS[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= _POS[0x7E], 0x7E, code)  # satfinite
    sign = np.signbit(v)
    out = (code | (sign.astype(np.int64) << 7)).astype(np.uint8)
    out = np.where(nan, np.uint8(0x7F), out).astype(np.uint8)
    return out


def bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even.

    bf16 keeps the top 16 bits of the binary32 encoding; rounding adds half an
    ulp of the kept part (0x7FFF plus the kept LSB for the even tie) to the
    discarded 16 bits.  Finite inputs only (out of contract otherwise).
    """
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = (b + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
