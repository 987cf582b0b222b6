"""Pins for the oracle's e5m2 codec, gradient quantisation and backward GEMMs (CPU only).

Pinned against: the closed form and the values the pages print (57344, the e5m2 maximum),
torch's float8_e5m2 casts (library routines), an exhaustive nearest-value search on exact
rationals with the tie rule (a planted ties-away encoder must fail), exact-rational brute force
of quantisation and of the whole promotion chain, the dequantised definition within its
rounding bound (planted mistakes must fail it), the integer block sums past 2^53, token-order
invariance inside a block, and the reduction of the K-grouped weight gradient to the
block-scaled form when its column scales are constant per 128 rows.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import bf16_bits_to_f32, e4m3_decode, quantize_128x128, quantize_1x128
from oracle.backward import (block_products, gemm_nt_dgrad, quantize_1x128_e5m2, wgrad_k_grouped)
from oracle.e5m2 import E5M2_MAX, e5m2_decode, e5m2_decode_table, e5m2_encode
from tests.exact import bf16_rn_bits, f32_rn


def _bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)


def _e5m2_values():
    out = {}
    for c in range(0x7C):
        e, m = c >> 2, c & 3
        out[c] = Fraction(m, 1 << 16) if e == 0 else (1 + Fraction(m, 4)) * Fraction(2) ** (e - 15)
    return out


_E5 = _e5m2_values()


def _nearest(y: Fraction, negative: bool) -> int:
    best = None
    for c, v in _E5.items():
        key = (abs(abs(y) - v), c % 2)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1] | (0x80 if negative else 0)


# ------------------------------------------------------------------ codec

def test_decode_closed_form_and_printed_maximum():
    t = e5m2_decode_table()
    assert t[0x7B] == 57344.0 == E5M2_MAX  # the maximum the pages print
    assert t[0x01] == 2.0 ** -16 and t[0x04] == 2.0 ** -14 and t[0x3C] == 1.0 and t[0x3E] == 1.5
    assert np.isinf(t[0x7C]) and t[0xFC] == -np.inf and np.all(np.isnan(t[[0x7D, 0x7E, 0x7F, 0xFF]]))
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    fin = np.isfinite(t)
    assert np.array_equal(t[fin], lib[fin]) and np.array_equal(np.isnan(t), np.isnan(lib))


def test_encode_matches_exhaustive_nearest_with_ties_to_even():
    rng = np.random.default_rng(201)
    vals = np.concatenate([rng.standard_normal(300) * 10.0 ** rng.integers(-6, 5, 300),
                           [0.0, -0.0, 2.0 ** -17, 3 * 2.0 ** -18, 1.125, 1.375, 57344.0, 60000.0, 61440.0,
                            -1e9, 2.0 ** -16 * 1.5]]).astype(np.float32)
    got = e5m2_encode(vals)
    for v, c in zip(vals, got):
        want = 0x7B | (0x80 if np.signbit(v) else 0) if abs(float(v)) >= 57344 else \
            _nearest(Fraction(float(v)), bool(np.signbit(v)))
        assert c == want, (v, hex(c), hex(want))
    # ties: 1.125 lies between 1.0 (0x3C) and 1.25 (0x3D) -> even code 0x3C; 1.375 -> 1.5 (0x3E)
    assert got[list(vals).index(np.float32(1.125))] == 0x3C
    assert got[list(vals).index(np.float32(1.375))] == 0x3E


def test_encode_matches_the_library_cast_in_range():
    rng = np.random.default_rng(202)
    v = (rng.standard_normal(20000) * 10.0 ** rng.integers(-5, 4, 20000)).astype(np.float32)
    v = v[np.abs(v) < 57344]
    lib = torch.from_numpy(v).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(e5m2_encode(v), lib)


def test_planted_ties_away_encoder_fails_the_tie_pin():
    def ties_away(x):
        lo = e5m2_encode(x)
        up = e5m2_encode(np.nextafter(np.float32(x), np.float32(np.inf)))
        return np.where(e5m2_decode(up) - x == x - e5m2_decode(lo), up, lo)
    x = np.float32(1.125)
    assert e5m2_encode(x) == 0x3C and ties_away(x) != 0x3C


# ------------------------------------------------------------------ gradient quantisation

def test_quantize_e5m2_matches_exact_rational_brute_force():
    rng = np.random.default_rng(203)
    x = _bf16(rng, (3, 256), 1e-3)
    x[1, :128] *= 1e-30
    x[2, 128:] = 0.0
    q, s = quantize_1x128_e5m2(x)
    for m in range(3):
        for kb in range(2):
            blk = x[m, kb * 128:(kb + 1) * 128]
            amax = max(abs(Fraction(float(v))) for v in blk)
            sc = f32_rn(amax / 57344)
            assert s[m, kb] == sc
            if sc == 0:
                assert not q[m, kb * 128:(kb + 1) * 128].any()
                continue
            for j, v in enumerate(blk):
                y = f32_rn(Fraction(float(v)) / Fraction(float(sc)))
                want = _nearest(Fraction(float(y)), bool(np.signbit(v)) or (y == 0 and np.signbit(y)))
                assert q[m, kb * 128 + j] == want, (m, kb, j)


@pytest.mark.parametrize("k", [-12, 9])
def test_quantize_e5m2_power_of_two_invariance_and_amax_code(k):
    rng = np.random.default_rng(204)
    x = _bf16(rng, (4, 384))
    q0, s0 = quantize_1x128_e5m2(x)
    q1, s1 = quantize_1x128_e5m2((x * np.float32(2.0 ** k)).astype(np.float32))
    assert np.array_equal(q0, q1) and np.array_equal((s0 * np.float32(2.0 ** k)).astype(np.float32), s1)
    j = np.abs(x[0, :128]).argmax()
    assert (q0[0, j] & 0x7F) == 0x7B


# ------------------------------------------------------------------ block sums

def test_block_products_are_exact_then_rounded_once():
    rng = np.random.default_rng(205)
    qa = rng.integers(0, 256, (3, 256)).astype(np.uint8)
    qa[(qa & 0x7C) == 0x7C] = 0x11  # finite e5m2 codes only
    qb = rng.integers(0, 256, (4, 256)).astype(np.uint8)
    qb[(qb & 0x7F) == 0x7F] = 0x22
    P = block_products(qa, "e5m2", qb, "e4m3")
    A, B = e5m2_decode(qa), e4m3_decode(qb)
    for kb in range(2):
        for m in range(3):
            for n in range(4):
                exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in
                            zip(A[m, kb * 128:(kb + 1) * 128], B[n, kb * 128:(kb + 1) * 128]))
                assert P[kb, m, n] == f32_rn(exact), (kb, m, n)


def test_block_sum_past_2_to_53_units_rounds_correctly():
    # 128 products of the largest codes: 57344 * 448 * 128 needs 57 bits in units of 2^-25;
    # one small term makes the float64 conversion inexact, the integer rounding must not care
    qa = np.full((1, 128), 0x7B, np.uint8)
    qb = np.full((2, 128), 0x7E, np.uint8)
    qb[1, 5] = 0x01  # 2^-9 instead of 448 in one product
    P = block_products(qa, "e5m2", qb, "e4m3")
    for n in range(2):
        exact = sum(Fraction(57344) * Fraction(float(b)) for b in e4m3_decode(qb[n]))
        assert P[0, 0, n] == f32_rn(exact)


# ------------------------------------------------------------------ backward GEMMs

def _dgrad_problem(rng, M, N, K):
    qa, sa = quantize_1x128_e5m2(_bf16(rng, (M, K), 1e-4))  # gradients: small values
    qb, sb = quantize_128x128(_bf16(rng, (N, K), 0.05))
    return qa, sa, qb, sb


def _dgrad_definition_ok(gemm, qa, sa, qb, sb):
    M, K = qa.shape
    N = qb.shape[0]
    A = e5m2_decode(qa) * np.repeat(sa.astype(np.float64), 128, axis=1)
    sbe = np.repeat(np.repeat(sb.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
    B = e4m3_decode(qb) * sbe
    R, mag = A @ B.T, np.abs(A) @ np.abs(B).T
    D = bf16_bits_to_f32(gemm(qa, sa, qb, sb)).astype(np.float64)
    return np.all(np.abs(D - R) <= 2.0 ** -8 * np.abs(R) + (K // 128 + 2) * 2.0 ** -22 * mag + 1e-300)


def test_dgrad_matches_exact_rational_promotion_chain():
    rng = np.random.default_rng(206)
    qa, sa, qb, sb = _dgrad_problem(rng, 2, 130, 256)
    d = gemm_nt_dgrad(qa, sa, qb, sb)
    A, B = e5m2_decode(qa), e4m3_decode(qb)
    for m in range(2):
        for n in (0, 127, 128, 129):
            acc = np.float32(0)
            for kb in range(2):
                p = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in
                        zip(A[m, kb * 128:(kb + 1) * 128], B[n, kb * 128:(kb + 1) * 128]))
                s = f32_rn(Fraction(float(sa[m, kb])) * Fraction(float(sb[n // 128, kb])))
                t = f32_rn(Fraction(float(f32_rn(p))) * Fraction(float(s)))
                acc = f32_rn(Fraction(float(acc)) + Fraction(float(t)))
            assert d[m, n] == bf16_rn_bits(acc), (m, n)


def test_dgrad_definition_and_planted_mistakes():
    rng = np.random.default_rng(207)
    qa, sa, qb, sb = _dgrad_problem(rng, 16, 300, 512)
    sb[1] *= 8
    sa[:, 2] *= 4
    assert _dgrad_definition_ok(gemm_nt_dgrad, qa, sa, qb, sb)

    def a_read_as_e4m3(qa, sa, qb, sb):
        P = block_products(qa, "e4m3", qb, "e4m3")
        from oracle.backward import _promote
        return _promote(P, sa, sb[np.arange(qb.shape[0]) // 128])

    def b_scale_per_row_index(qa, sa, qb, sb):  # n % 128 instead of n // 128
        from oracle.backward import _promote
        P = block_products(qa, "e5m2", qb, "e4m3")
        return _promote(P, sa, sb[np.arange(qb.shape[0]) % sb.shape[0]])

    def dropped_block(qa, sa, qb, sb):
        sa2 = sa.copy()
        sa2[:, 0] = 0
        return gemm_nt_dgrad(qa, sa2, qb, sb)

    for bad in (a_read_as_e4m3, b_scale_per_row_index, dropped_block):
        assert not _dgrad_definition_ok(bad, qa, sa, qb, sb), bad.__name__


def _wgrad_problem(rng, N, K, T):
    qa, sa = quantize_1x128_e5m2(_bf16(rng, (N, T), 1e-4))  # dY^T
    qb, sb = quantize_1x128(_bf16(rng, (K, T)))              # X^T
    return qa, sa, qb, sb


def test_wgrad_per_expert_definition_and_empty_expert():
    rng = np.random.default_rng(208)
    N, K, T = 24, 40, 640
    qa, sa, qb, sb = _wgrad_problem(rng, N, K, T)
    off = np.array([0, 256, 256, 512], np.int32)  # expert 1 empty; tokens 512.. in no expert
    d = wgrad_k_grouped(qa, sa, qb, sb, off)
    assert d.shape == (3, N, K) and not d[1].any()
    for e in (0, 2):
        t0, t1 = off[e], off[e + 1]
        A = e5m2_decode(qa[:, t0:t1]) * np.repeat(sa[:, t0 // 128:t1 // 128].astype(np.float64), 128, axis=1)
        B = e4m3_decode(qb[:, t0:t1]) * np.repeat(sb[:, t0 // 128:t1 // 128].astype(np.float64), 128, axis=1)
        R, mag = A @ B.T, np.abs(A) @ np.abs(B).T
        D = bf16_bits_to_f32(d[e]).astype(np.float64)
        assert np.all(np.abs(D - R) <= 2.0 ** -8 * np.abs(R) + 6 * 2.0 ** -22 * mag + 1e-300), e
    # planted: expert 0 also summing expert 2's tokens fails its definition
    leak = wgrad_k_grouped(qa, sa, qb, sb, np.array([0, 512, 512, 512], np.int32))[0]
    assert not np.array_equal(leak, d[0])


def test_wgrad_token_order_inside_a_block_does_not_matter():
    rng = np.random.default_rng(209)
    qa, sa, qb, sb = _wgrad_problem(rng, 8, 16, 256)
    off = np.array([0, 256], np.int32)
    perm = np.concatenate([rng.permutation(128), 128 + rng.permutation(128)])
    assert np.array_equal(wgrad_k_grouped(qa, sa, qb, sb, off),
                          wgrad_k_grouped(qa[:, perm], sa, qb[:, perm], sb, off))


def test_wgrad_reduces_to_the_block_scaled_form():
    # column scales constant over each 128 rows of X^T: the K-grouped weight gradient of one
    # expert is the data-gradient form with 128x128 scales on B
    rng = np.random.default_rng(210)
    N, K, T = 16, 256, 384
    qa, sa, qb, _ = _wgrad_problem(rng, N, K, T)
    sblk = rng.uniform(0.5, 2.0, (K // 128, T // 128)).astype(np.float32)
    sb_rows = np.repeat(sblk, 128, axis=0)
    d = wgrad_k_grouped(qa, sa, qb, sb_rows, np.array([0, T], np.int32))[0]
    assert np.array_equal(d, gemm_nt_dgrad(qa, sa, qb, sblk))
