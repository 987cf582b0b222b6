"""Pins for the oracle's 1x128 and 128x128 quantisation (CPU only).

Pinned against: a hand-worked example of the scale rule amax/448 (the divisor
the pages print, tests/golden/e4m3_format.txt), an exact-rational brute force
that rounds from the definition, the power-of-two invariance, the zero block,
and the relation between the two block shapes.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import e4m3_decode, quantize_1x128, quantize_128x128
from tests.exact import e4m3_nearest, f32_rn


def _brute_quantize_block(vals):
    """vals: float32 list of one block -> (codes, scale) from exact rationals."""
    amax = max(abs(Fraction(float(v))) for v in vals)
    s = f32_rn(amax / 448)
    if s == 0:
        return [0] * len(vals), s
    codes = []
    for v in vals:
        y = f32_rn(Fraction(float(v)) / Fraction(float(s)))
        codes.append(e4m3_nearest(Fraction(float(y)), bool(np.signbit(v)) or (y == 0 and np.signbit(y))))
    return codes, s


def _bf16_values(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    # keep bf16 values only (truncate the low 16 bits: still a valid bf16 draw)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)


def test_worked_example_scale_two():
    # amax = 896 -> s = 896/448 = 2 exactly; every x/2 below is an e4m3 value.
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, :6] = [896.0, -896.0, 1.0, -3.0, 0.0, 2.0 ** -8]
    q, s = quantize_1x128(x)
    assert s[0, 0] == 2.0
    assert list(q[0, :6]) == [0x7E, 0xFE, 0x30, 0xBC, 0x00, 0x01]
    # 0x30 = 0.5, 0xBC = -1.5, 0x01 = 2^-9
    assert list(e4m3_decode(q[0, :6])) == [448.0, -448.0, 0.5, -1.5, 0.0, 2.0 ** -9]


def test_scale_rule_is_amax_over_448():
    rng = np.random.default_rng(1)
    x = _bf16_values(rng, (16, 512), 3.0)
    q, s = quantize_1x128(x)
    for m in range(16):
        for kb in range(4):
            amax = Fraction(float(np.abs(x[m, kb * 128:(kb + 1) * 128]).max()))
            assert s[m, kb] == f32_rn(amax / 448)


def test_1x128_matches_exact_rational_brute_force():
    rng = np.random.default_rng(2)
    x = _bf16_values(rng, (3, 256))
    x[1, :128] *= 1e-30  # tiny block: subnormal-range quotients
    x[2, 128:] = 0.0
    x[2, 130] = -0.0
    q, s = quantize_1x128(x)
    for m in range(3):
        for kb in range(2):
            codes, sc = _brute_quantize_block(list(x[m, kb * 128:(kb + 1) * 128]))
            assert s[m, kb] == sc
            assert list(q[m, kb * 128:(kb + 1) * 128]) == codes, (m, kb)


def test_zero_block_gives_zero_scale_and_zero_codes():
    x = np.zeros((2, 256), dtype=np.float32)
    x[0, 5] = -0.0
    x[1, 200] = 1.5
    q, s = quantize_1x128(x)
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0
    assert not q[0].any() and not q[1, :128].any()
    assert s[1, 1] == np.float32(1.5) / np.float32(448)


@pytest.mark.parametrize("k", [-20, -3, 1, 7, 30])
def test_power_of_two_invariance(k):
    rng = np.random.default_rng(3)
    x = _bf16_values(rng, (8, 384))
    q0, s0 = quantize_1x128(x)
    q1, s1 = quantize_1x128((x * np.float32(2.0 ** k)).astype(np.float32))
    assert np.array_equal(q0, q1)
    assert np.array_equal(s1, (s0 * np.float32(2.0 ** k)).astype(np.float32))


def test_block_max_maps_to_448_and_error_bound():
    rng = np.random.default_rng(4)
    x = _bf16_values(rng, (32, 1024), 10.0)
    q, s = quantize_1x128(x)
    xb = x.reshape(32, 8, 128)
    qb = q.reshape(32, 8, 128)
    i = np.abs(xb).argmax(axis=2)
    top = np.take_along_axis(qb, i[..., None], 2)[..., 0] & 0x7F
    assert np.all(top == 0x7E)
    # relative dequantisation error of a normal e4m3 value is at most 2^-4
    deq = e4m3_decode(qb) * s[:, :, None]
    big = np.abs(xb) >= s[:, :, None] * 2.0 ** -6
    err = np.abs(deq - xb)[big] / np.abs(xb)[big]
    assert err.max() <= 2.0 ** -4 + 1e-6


def test_128x128_brute_force_with_ragged_tail():
    rng = np.random.default_rng(5)
    N, K = 200, 256  # second row block has 72 rows
    w = _bf16_values(rng, (N, K), 0.05)
    q, s = quantize_128x128(w)
    assert s.shape == (2, 2)
    for nb in range(2):
        r0, r1 = nb * 128, min(N, nb * 128 + 128)
        for kb in range(2):
            blk = w[r0:r1, kb * 128:(kb + 1) * 128]
            amax = Fraction(float(np.abs(blk).max()))
            sc = f32_rn(amax / 448)
            assert s[nb, kb] == sc
            # spot rows: full brute force is slow in pure Python
            for r in (r0, r0 + 1, r1 - 1):
                for c in range(kb * 128, kb * 128 + 128, 7):
                    y = f32_rn(Fraction(float(w[r, c])) / Fraction(float(sc)))
                    want = e4m3_nearest(Fraction(float(y)), bool(np.signbit(w[r, c])))
                    assert q[r, c] == want


def test_128x128_scale_is_max_of_row_scales():
    # amax/448 rounds monotonically, so the block scale is the largest 1x128 scale of its rows
    rng = np.random.default_rng(6)
    w = _bf16_values(rng, (256, 512))
    _, s_blk = quantize_128x128(w)
    _, s_row = quantize_1x128(w)
    assert np.array_equal(s_blk, s_row.reshape(2, 128, 4).max(axis=1))
