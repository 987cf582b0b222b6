"""Pins for the oracle's e4m3 codec and bf16 rounding (CPU only).

Pinned against: the values the pages print (tests/golden/e4m3_format.txt), the
format's closed form at hand-picked codes, a library routine (torch's
float8_e4m3fn and bfloat16 casts), and a pure-Python exhaustive nearest-value
search.  A planted mistake (ties away from zero) must fail the tie pin.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import e4m3 as E

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = line.split()[:2]
                out[k] = float(v)
    return out


def test_max_finite_is_the_pages_448():
    g = _golden("e4m3_format.txt")
    tab = E.e4m3_decode_table()
    finite = tab[np.isfinite(tab)]
    assert finite.max() == g["max_finite"] == E.E4M3_MAX
    # 3 mantissa bits: 8 codes per binade; 4 exponent bits: 16 exponent fields
    assert g["mantissa_bits"] == 3 and g["exponent_bits"] == 4
    assert sum(1 for c in range(0x7F) if (c >> 3) == 7) == 2 ** g["mantissa_bits"]


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x77, 240.0),
    (0x78, 256.0), (0x7D, 416.0), (0x7E, 448.0), (0x80, -0.0), (0xB8, -1.0), (0xFE, -448.0),
])
def test_decode_hand_values(code, value):
    v = E.e4m3_decode(np.array([code], dtype=np.uint8))[0]
    assert v == value and math.copysign(1, v) == math.copysign(1, value)


def test_decode_nan_codes_only_all_ones():
    tab = E.e4m3_decode_table()
    nan_codes = [c for c in range(256) if np.isnan(tab[c])]
    assert nan_codes == [0x7F, 0xFF]
    assert not np.isinf(tab).any()


def test_decode_matches_torch_float8_e4m3fn_all_256():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = E.e4m3_decode(codes.numpy())
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(ours[ok]))


def test_decode_strictly_monotone_positive_codes():
    tab = E.e4m3_decode_table()[:0x7F]
    assert np.all(np.diff(tab) > 0)


def test_encode_roundtrip_every_finite_code():
    tab = E.e4m3_decode_table()
    codes = np.array([c for c in range(256) if not np.isnan(tab[c])], dtype=np.uint8)
    assert np.array_equal(E.e4m3_encode(tab[codes]), codes)


def _tie_pin(encode):
    """Midpoints between neighbouring codes go to the even code."""
    tab = E.e4m3_decode_table()
    bad = []
    for c in range(0x7E):
        mid = (tab[c] + tab[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        for sgn in (1.0, -1.0):
            got = int(encode(np.array([sgn * mid], dtype=np.float32))[0])
            if got != (want | (0x80 if sgn < 0 else 0)):
                bad.append((c, sgn, got))
    return bad


def test_encode_ties_to_even():
    assert _tie_pin(E.e4m3_encode) == []


def test_planted_ties_away_mistake_is_caught():
    def ties_away(v):
        v = np.asarray(v, dtype=np.float64)
        mag = np.abs(v)
        pos = E.e4m3_decode_table()[:0x7F]
        hi = np.minimum(np.searchsorted(pos, mag), 0x7E)
        lo = np.maximum(hi - 1, 0)
        code = np.where(pos[hi] - mag <= mag - pos[lo], hi, lo)  # ties up
        return (code | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)
    assert _tie_pin(ties_away) != []


def test_encode_neighbours_of_midpoints():
    tab = E.e4m3_decode_table()
    for c in range(0x7E):
        mid = np.float32((tab[c] + tab[c + 1]) / 2)
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1e9))
        assert E.e4m3_encode(np.array([below]))[0] == c
        assert E.e4m3_encode(np.array([above]))[0] == c + 1


def test_encode_matches_torch_on_dense_sweep():
    g = torch.Generator().manual_seed(123)
    # log-uniform magnitudes across the whole e4m3 range incl. subnormals, random signs
    mag = torch.exp2(torch.rand(400_000, generator=g, dtype=torch.float64) * 19 - 11)
    mag = mag.clamp(max=463.0)
    sgn = torch.where(torch.rand(400_000, generator=g) < 0.5, -1.0, 1.0).double()
    v = (mag * sgn).float()
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = E.e4m3_encode(v.numpy())
    assert np.array_equal(ref, ours)


def test_encode_saturates_and_keeps_sign():
    v = np.array([448.0, 449.0, 463.9, 464.0, 1e6, 3e38, -449.0, -3e38], dtype=np.float32)
    assert list(E.e4m3_encode(v)) == [0x7E] * 6 + [0xFE] * 2
    z = np.array([0.0, -0.0, 1e-10, -1e-10, 2.0 ** -10, -(2.0 ** -10)], dtype=np.float32)
    # 2^-10 is the midpoint between 0 and 2^-9: ties to the even code 0
    assert list(E.e4m3_encode(z)) == [0x00, 0x80, 0x00, 0x80, 0x00, 0x80]
    assert E.e4m3_encode(np.array([np.nan], dtype=np.float32))[0] == 0x7F


def test_encode_matches_pure_python_exhaustive_search():
    tab = E.e4m3_decode_table()
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.uniform(-470, 470, 300), rng.uniform(-0.05, 0.05, 300)]).astype(np.float32)
    for v in vals:
        best, best_d = None, None
        for c in range(0x7F):  # every non-negative finite code
            d = abs(abs(float(v)) - tab[c])
            if best is None or d < best_d or (d == best_d and c % 2 == 0):
                best, best_d = c, d
        want = best | (0x80 if np.signbit(v) else 0)
        assert E.e4m3_encode(np.array([v]))[0] == want, v


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(200_000, generator=g) * torch.exp2(torch.randint(-30, 30, (200_000,), generator=g).float())
    ours = E.bf16_round_bits(x.numpy())
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8)], dtype=np.float32)
    got = E.bf16_bits_to_f32(E.bf16_round_bits(x))
    assert list(got) == [1.0, 1 + 2.0 ** -6, -1.0]
