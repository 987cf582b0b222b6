"""Pins for the oracle's per-tensor / per-channel scaled GEMM and its quantisers (CPU only).

Pinned against: an exact-rational brute force of quantisation and of the epilogue chain
(exact sum, one fp32 rounding, fp32 scale product, fp32 product, bf16), the plain
definition computed another way (dequantise both operands in fp64, one matmul) within
the rounding bound, the block-scaled oracle (itself pinned) where the two coincide --
one 128-wide K block for the quantisers, constant scales and exactly representable sums
for the GEMM (the per-tensor formula of the Triton listing on "Production FP8 GEMM
alignment and Tensor Core peak tuning") --, power-of-two invariances, and grouped ==
per-group dense.  Planted mistakes (scales indexed by the wrong operand, a sign flip, a
dropped K block) must fail the definition pin.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import (bf16_bits_to_f32, e4m3_decode, gemm_nt, quantize_1x128)
from oracle.scaled import (gemm_nt_scaled, grouped_contiguous_scaled, grouped_masked_scaled,
                           quantize_per_row, quantize_per_tensor)
from tests.exact import bf16_rn_bits, e4m3_nearest, f32_rn


def _bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)


def _brute_quantize_group(vals):
    amax = max(abs(Fraction(float(v))) for v in vals)
    s = f32_rn(amax / 448)
    if s == 0:
        return [0] * len(vals), s
    codes = []
    for v in vals:
        y = f32_rn(Fraction(float(v)) / Fraction(float(s)))
        codes.append(e4m3_nearest(Fraction(float(y)), bool(np.signbit(v)) or (y == 0 and np.signbit(y))))
    return codes, s


# ------------------------------------------------------------------ quantisers

def test_per_row_matches_exact_rational_brute_force():
    rng = np.random.default_rng(101)
    x = _bf16(rng, (3, 384), 2.0)
    x[1] *= 1e-30  # subnormal-range quotients
    x[2] = 0.0
    x[2, 7] = -0.0
    q, s = quantize_per_row(x)
    for m in range(3):
        codes, sc = _brute_quantize_group(list(x[m]))
        assert s[m] == sc
        assert list(q[m]) == codes, m


def test_per_tensor_matches_exact_rational_brute_force():
    rng = np.random.default_rng(102)
    x = _bf16(rng, (3, 256), 0.5)
    x[2, 5] = 37.25  # the tensor's amax sits in one row
    q, s = quantize_per_tensor(x)
    codes, sc = _brute_quantize_group(list(x.reshape(-1)))
    assert s.shape == (1,) and s[0] == sc
    assert list(q.reshape(-1)) == codes


def test_single_block_reduces_to_the_1x128_quantiser():
    rng = np.random.default_rng(103)
    x = _bf16(rng, (17, 128), 4.0)
    q1, s1 = quantize_1x128(x)
    qr, sr = quantize_per_row(x)
    assert np.array_equal(q1, qr) and np.array_equal(s1[:, 0], sr)
    qt, st = quantize_per_tensor(x[5:6])
    assert np.array_equal(qt, q1[5:6]) and st[0] == s1[5, 0]


def test_per_tensor_equals_per_row_when_every_row_holds_the_amax():
    rng = np.random.default_rng(104)
    x = _bf16(rng, (8, 512))
    x[:, 3] = -9.5  # larger than every normal draw here
    qr, sr = quantize_per_row(x)
    qt, st = quantize_per_tensor(x)
    assert np.all(sr == st[0]) and np.array_equal(qr, qt)


def test_group_amax_maps_to_448():
    rng = np.random.default_rng(105)
    x = _bf16(rng, (6, 256), 3.0)
    q, s = quantize_per_row(x)
    for m in range(6):
        j = int(np.argmax(np.abs(x[m])))
        assert (q[m, j] & 0x7F) == 0x7E  # +-448


@pytest.mark.parametrize("k", [-20, 7])
def test_quantisers_scale_with_powers_of_two(k):
    rng = np.random.default_rng(106)
    x = _bf16(rng, (5, 256))
    f = np.float32(2.0 ** k)
    for quant in (quantize_per_row, quantize_per_tensor):
        q0, s0 = quant(x)
        q1, s1 = quant((x * f).astype(np.float32))
        assert np.array_equal(q0, q1) and np.array_equal((s0 * f).astype(np.float32), s1)


def test_zero_groups():
    x = np.zeros((3, 256), np.float32)
    x[1, 9] = 2.0
    q, s = quantize_per_row(x)
    assert s[0] == 0 and s[2] == 0 and not q[0].any() and not q[2].any()
    qt, st = quantize_per_tensor(np.zeros((2, 128), np.float32))
    assert st[0] == 0 and not qt.any()


# ------------------------------------------------------------------ GEMM

def _problem(rng, M, N, K, per_row=True, per_col=True, a_scale=1.0, b_scale=0.05):
    xa, xb = _bf16(rng, (M, K), a_scale), _bf16(rng, (N, K), b_scale)
    qa, sa = quantize_per_row(xa) if per_row else quantize_per_tensor(xa)
    qb, sb = quantize_per_row(xb) if per_col else quantize_per_tensor(xb)
    return qa, sa, qb, sb


def _definition_pin(gemm, qa, sa, qb, sb):
    """|D - R| <= 2^-8 |R| + 2^-21 sum|a b|: the fp32 rounding of the sum, of the scale
    product and of the scaled value, then one bf16 rounding."""
    M, N = qa.shape[0], qb.shape[0]
    sa_ = np.broadcast_to(np.asarray(sa, np.float64).reshape(-1), (M,))
    sb_ = np.broadcast_to(np.asarray(sb, np.float64).reshape(-1), (N,))
    A = e4m3_decode(qa) * sa_[:, None]
    B = e4m3_decode(qb) * sb_[:, None]
    R = A @ B.T
    mag = np.abs(A) @ np.abs(B).T
    D = bf16_bits_to_f32(gemm(qa, sa, qb, sb)).astype(np.float64)
    return np.all(np.abs(D - R) <= 2.0 ** -8 * np.abs(R) + 2.0 ** -21 * mag + 1e-30)


def test_matches_exact_rational_epilogue_chain():
    rng = np.random.default_rng(111)
    qa, sa, qb, sb = _problem(rng, 3, 5, 384, a_scale=3.0)
    d = gemm_nt_scaled(qa, sa, qb, sb)
    A = [[Fraction(float(v)) for v in row] for row in e4m3_decode(qa)]
    B = [[Fraction(float(v)) for v in row] for row in e4m3_decode(qb)]
    for m in range(3):
        for n in range(5):
            acc = f32_rn(sum(a * b for a, b in zip(A[m], B[n])))
            s = f32_rn(Fraction(float(sa[m])) * Fraction(float(sb[n])))
            assert d[m, n] == bf16_rn_bits(f32_rn(Fraction(float(acc)) * Fraction(float(s)))), (m, n)


@pytest.mark.parametrize("per_row,per_col", [(True, True), (False, False), (True, False), (False, True)])
def test_matches_definition_within_rounding_bound(per_row, per_col):
    rng = np.random.default_rng(112)
    qa, sa, qb, sb = _problem(rng, 24, 200, 640, per_row, per_col, a_scale=3.0)
    assert _definition_pin(gemm_nt_scaled, qa, sa, qb, sb)


def test_planted_mistakes_fail_the_definition_pin():
    rng = np.random.default_rng(113)
    qa, sa, qb, sb = _problem(rng, 16, 16, 512)
    sa = (sa * np.float32(2.0) ** np.arange(16, dtype=np.float32)).astype(np.float32)  # rows differ

    def swapped_scales(qa, sa, qb, sb):  # A's scale taken per column, B's per row
        return gemm_nt_scaled(qa, sb, qb, sa)

    def sign_flip(qa, sa, qb, sb):
        return gemm_nt_scaled(qa, -sa, qb, sb)

    def dropped_block(qa, sa, qb, sb):
        qa2 = qa.copy()
        qa2[:, -128:] = 0
        return gemm_nt_scaled(qa2, sa, qb, sb)

    def transposed_result(qa, sa, qb, sb):
        return gemm_nt_scaled(qa, sa, qb, sb).T.copy()

    assert _definition_pin(gemm_nt_scaled, qa, sa, qb, sb)
    for bad in (swapped_scales, sign_flip, dropped_block, transposed_result):
        assert not _definition_pin(bad, qa, sa, qb, sb), bad.__name__


def test_per_tensor_equals_block_scaled_with_constant_scales():
    # small integer codes: every partial sum is exact in fp32, so per-block promotion with equal
    # block scales and the single epilogue multiplication give the same bits
    rng = np.random.default_rng(114)
    M, N, K = 8, 256, 512
    codes = np.array([0x00, 0x38, 0xB8, 0x40, 0xC0, 0x30], dtype=np.uint8)  # 0, +-1, +-2, 0.5
    qa = rng.choice(codes, (M, K))
    qb = rng.choice(codes, (N, K))
    alpha, beta = np.float32(0.375), np.float32(0.0078125)
    d_block = gemm_nt(qa, np.full((M, K // 128), alpha, np.float32), qb,
                      np.full((N // 128, K // 128), beta, np.float32))
    d_tensor = gemm_nt_scaled(qa, np.array([alpha]), qb, np.array([beta]))
    assert np.array_equal(d_block, d_tensor)


def test_power_of_two_row_and_column_scales():
    rng = np.random.default_rng(115)
    qa, sa, qb, sb = _problem(rng, 6, 9, 256)
    d0 = gemm_nt_scaled(qa, sa, qb, sb)
    ka = np.array([3, -2, 0, 5, -7, 1], np.float32)
    kb = np.array([-3, 2, 0, -5, 7, -1, 4, -4, 0], np.float32)
    d1 = gemm_nt_scaled(qa, (sa * 2.0 ** ka).astype(np.float32), qb, (sb * 2.0 ** kb).astype(np.float32))
    want = bf16_bits_to_f32(d0).astype(np.float64) * 2.0 ** ka[:, None] * 2.0 ** kb[None, :]
    assert np.array_equal(bf16_bits_to_f32(d1).astype(np.float64), want)


def test_grouped_contiguous_equals_concatenated_dense():
    rng = np.random.default_rng(116)
    E, N, K = 3, 144, 256
    off = np.array([0, 128, 128, 384], np.int32)  # expert 1 empty; rows 384.. in no group
    M_total = 512
    qa, sa = quantize_per_row(_bf16(rng, (M_total, K)))
    qw, sw = quantize_per_row(_bf16(rng, (E * N, K), 0.05))
    qb, sb = qw.reshape(E, N, K), sw.reshape(E, N)
    init = np.full((M_total, N), 0xFFFF, np.uint16)
    d = grouped_contiguous_scaled(qa, sa, qb, sb, off, init)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            assert np.array_equal(d[r0:r1], gemm_nt_scaled(qa[r0:r1], sa[r0:r1], qb[e], sb[e]))
    assert np.all(d[384:] == 0xFFFF)
    # one scale per expert for B and one for all of A
    sbt = np.array([[0.5], [0.25], [2.0]], np.float32)
    d2 = grouped_contiguous_scaled(qa, np.array([0.125], np.float32), qb, sbt, off, init)
    for e in (0, 2):
        r0, r1 = off[e], off[e + 1]
        assert np.array_equal(d2[r0:r1], gemm_nt_scaled(qa[r0:r1], np.array([0.125]), qb[e], sbt[e]))


def test_grouped_masked_leaves_rows_past_the_count():
    rng = np.random.default_rng(117)
    E, cap, N, K = 3, 32, 48, 128
    qa, sa = quantize_per_row(_bf16(rng, (E * cap, K)))
    qw, sw = quantize_per_row(_bf16(rng, (E * N, K), 0.05))
    masked = np.array([5, 0, 32], np.int32)
    init = np.full((E, cap, N), 0xFFFF, np.uint16)
    d = grouped_masked_scaled(qa.reshape(E, cap, K), sa, qw.reshape(E, N, K), sw.reshape(E, N), masked, init)
    for e in range(E):
        m = masked[e]
        rows = slice(e * cap, e * cap + m)
        if m:
            assert np.array_equal(d[e, :m], gemm_nt_scaled(qa[rows], sa[rows], qw[e * N:(e + 1) * N],
                                                            sw[e * N:(e + 1) * N]))
        assert np.all(d[e, m:] == 0xFFFF)
