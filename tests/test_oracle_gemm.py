"""Pins for the oracle's block-scaled GEMM and its grouped forms (CPU only).

Pinned against: an exact-rational brute force of the whole promotion chain,
the plain definition computed another way (dequantise both operands in fp64,
then one matmul) within the rounding bound, power-of-two invariances, the
per-tensor special case (the epilogue formula of the Triton listing on
"Production FP8 GEMM alignment and Tensor Core peak tuning"), the single-block
case, and grouped == per-group dense.  Planted mistakes (transposed B-scale
index, a dropped K block, a sign flip) must fail the definition pin.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import (bf16_bits_to_f32, e4m3_decode, gemm_nt, grouped_contiguous, grouped_masked,
                    quantize_1x128, quantize_128x128)
from tests.exact import bf16_rn_bits, f32_rn


def _bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) & 0xFFFF0000).view(np.float32)


def _problem(rng, M, N, K, a_scale=1.0, b_scale=0.05):
    qa, sa = quantize_1x128(_bf16(rng, (M, K), a_scale))
    qb, sb = quantize_128x128(_bf16(rng, (N, K), b_scale))
    return qa, sa, qb, sb


def _definition(qa, sa, qb, sb):
    """Dequantise each operand in fp64 (scale per element), then one matmul.

    Returns the exact real result R and the magnitude sum used in the bound.
    """
    M, K = qa.shape
    N = qb.shape[0]
    A = e4m3_decode(qa) * np.repeat(sa.astype(np.float64), 128, axis=1)
    sbe = np.repeat(np.repeat(sb.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
    B = e4m3_decode(qb) * sbe
    R = A @ B.T
    mag = np.abs(A) @ np.abs(B).T
    return R, mag


def _definition_pin(gemm, qa, sa, qb, sb):
    """|D - R| <= 2^-8 |R| + (KB + 2) 2^-22 sum|a b|  (fp32 promotion + one bf16 rounding)."""
    D = bf16_bits_to_f32(gemm(qa, sa, qb, sb)).astype(np.float64)
    R, mag = _definition(qa, sa, qb, sb)
    KB = qa.shape[1] // 128
    bound = 2.0 ** -8 * np.abs(R) + (KB + 2) * 2.0 ** -22 * mag + 1e-30
    return np.all(np.abs(D - R) <= bound)


def test_matches_exact_rational_promotion_chain():
    rng = np.random.default_rng(11)
    qa, sa, qb, sb = _problem(rng, 3, 130, 256)
    cols = np.array([0, 1, 127, 128, 129])
    d = gemm_nt(qa, sa, qb[cols], sb, n_index=cols)
    A = [[Fraction(float(v)) for v in row] for row in e4m3_decode(qa)]
    B = [[Fraction(float(v)) for v in e4m3_decode(qb[c])] for c in cols]
    for m in range(3):
        for j, c in enumerate(cols):
            acc = np.float32(0)
            for kb in range(2):
                p = sum(A[m][k] * B[j][k] for k in range(kb * 128, kb * 128 + 128))
                s = f32_rn(Fraction(float(sa[m, kb])) * Fraction(float(sb[c // 128, kb])))
                t = f32_rn(Fraction(float(f32_rn(p))) * Fraction(float(s)))
                acc = f32_rn(Fraction(float(acc)) + Fraction(float(t)))
            assert d[m, j] == bf16_rn_bits(acc), (m, c)


def test_matches_definition_within_rounding_bound():
    rng = np.random.default_rng(12)
    qa, sa, qb, sb = _problem(rng, 40, 300, 640, a_scale=3.0)
    # non-uniform B scales across row blocks make the n // 128 index matter
    sb[1] *= 8
    sb[2] /= 4
    assert _definition_pin(gemm_nt, qa, sa, qb, sb)


def test_planted_mistakes_fail_the_definition_pin():
    rng = np.random.default_rng(13)
    qa, sa, qb, sb = _problem(rng, 16, 300, 512)
    sb[1] *= 8
    sb[2] /= 4
    sa[:, 2] *= 16

    def wrong_b_index(qa, sa, qb, sb):  # n % 128 instead of n // 128 (clipped to the table)
        return gemm_nt(qa, sa, qb, sb, n_index=(np.arange(qb.shape[0]) % 128) * 128 % (sb.shape[0] * 128))

    def dropped_block(qa, sa, qb, sb):
        sa2 = sa.copy()
        sa2[:, -1] = 0
        return gemm_nt(qa, sa2, qb, sb)

    def sign_flip(qa, sa, qb, sb):
        return gemm_nt(qa, -sa, qb, sb)

    def transposed_scales(qa, sa, qb, sb):  # A's scales taken in reverse K-block order
        return gemm_nt(qa, sa[:, ::-1].copy(), qb, sb)

    assert _definition_pin(gemm_nt, qa, sa, qb, sb)
    for bad in (wrong_b_index, dropped_block, sign_flip, transposed_scales):
        assert not _definition_pin(bad, qa, sa, qb, sb), bad.__name__


@pytest.mark.parametrize("k", [-9, 5])
def test_scale_power_of_two_invariance(k):
    rng = np.random.default_rng(14)
    qa, sa, qb, sb = _problem(rng, 8, 256, 384)
    d0 = gemm_nt(qa, sa, qb, sb)
    sa2, sb2 = sa.copy(), sb.copy()
    sa2[:, 1] *= np.float32(2.0 ** k)
    sb2[:, 1] *= np.float32(2.0 ** -k)
    assert np.array_equal(d0, gemm_nt(qa, sa2, qb, sb2))


def test_code_exponent_shift_invariance():
    # doubling every A value of one K block (code exponent +1) with its scale halved
    rng = np.random.default_rng(15)
    qa, sa, qb, sb = _problem(rng, 8, 128, 256)
    blk = qa[:, :128]
    e = (blk >> 3) & 0xF
    ok = (e >= 1) & (e <= 13)  # normal codes that stay finite after +1
    qa2 = qa.copy()
    qa2[:, :128] = np.where(ok, blk + 8, 0)
    qa_ref = qa.copy()
    qa_ref[:, :128] = np.where(ok, blk, 0)
    sa2 = sa.copy()
    sa2[:, 0] /= 2
    assert np.array_equal(gemm_nt(qa_ref, sa, qb, sb), gemm_nt(qa2, sa2, qb, sb))


def test_per_tensor_special_case_is_the_listing_epilogue():
    # all block scales equal and small integer codes: every partial sum is exact in fp32,
    # so per-block promotion equals acc * (scale_a * scale_b) applied once at the end.
    rng = np.random.default_rng(16)
    M, N, K = 8, 256, 512
    codes = np.array([0x00, 0x38, 0xB8, 0x40, 0xC0, 0x30], dtype=np.uint8)  # 0, +-1, +-2, 0.5
    qa = rng.choice(codes, (M, K))
    qb = rng.choice(codes, (N, K))
    alpha, beta = np.float32(0.375), np.float32(0.0078125)
    sa = np.full((M, K // 128), alpha, np.float32)
    sb = np.full((N // 128, K // 128), beta, np.float32)
    d = gemm_nt(qa, sa, qb, sb)
    acc = e4m3_decode(qa) @ e4m3_decode(qb).T
    want = (acc.astype(np.float32) * (alpha * beta)).astype(np.float32)
    want_bits = torch.from_numpy(want).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(d, want_bits)


def test_single_k_block_closed_form():
    rng = np.random.default_rng(17)
    qa, sa, qb, sb = _problem(rng, 5, 7, 128)
    d = gemm_nt(qa, sa, qb, sb)
    A, B = e4m3_decode(qa), e4m3_decode(qb)
    for m in range(5):
        for n in range(7):
            p = np.float32(sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(A[m], B[n])))
            want = bf16_rn_bits(f32_rn(Fraction(float(p)) * Fraction(float(f32_rn(
                Fraction(float(sa[m, 0])) * Fraction(float(sb[0, 0])))))))
            assert d[m, n] == want


def test_pages_64x64_case():
    # "DeepGEMM explainer" sec. 4.2: check a 64x64 product against a CPU reference first
    rng = np.random.default_rng(18)
    qa, sa, qb, sb = _problem(rng, 64, 64, 128)
    assert _definition_pin(gemm_nt, qa, sa, qb, sb)


def test_grouped_contiguous_equals_concatenated_dense():
    rng = np.random.default_rng(19)
    E, N, K = 3, 192, 256
    off = np.array([0, 128, 128, 384], np.int32)  # expert 1 empty
    M_total = 512  # rows 384.. belong to no group and must stay untouched
    qa, sa = quantize_1x128(_bf16(rng, (M_total, K)))
    qbs, sbs = zip(*(quantize_128x128(_bf16(rng, (N, K), 0.05)) for _ in range(E)))
    qb, sb = np.stack(qbs), np.stack(sbs)
    init = np.full((M_total, N), 0xFFFF, np.uint16)
    d = grouped_contiguous(qa, sa, qb, sb, off, init)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            assert np.array_equal(d[r0:r1], gemm_nt(qa[r0:r1], sa[r0:r1], qb[e], sb[e]))
    assert np.all(d[384:] == 0xFFFF)


def test_pages_two_experts_eight_tokens():
    # "DeepGEMM FP8 walk-through" sec. 5.3: a fixed grouping of 2 experts x 8 tokens first.
    rng = np.random.default_rng(20)
    K, N = 256, 128
    x = _bf16(rng, (16, K))
    qx, sx = quantize_1x128(x)
    qa = np.zeros((256, K), np.uint8)
    sa = np.zeros((256, K // 128), np.float32)
    qa[0:8], sa[0:8] = qx[:8], sx[:8]  # expert 0: tokens 0..7, padded to 128 rows
    qa[128:136], sa[128:136] = qx[8:], sx[8:]
    qbs, sbs = zip(*(quantize_128x128(_bf16(rng, (N, K), 0.05)) for _ in range(2)))
    qb, sb = np.stack(qbs), np.stack(sbs)
    d = grouped_contiguous(qa, sa, qb, sb, np.array([0, 128, 256]), np.zeros((256, N), np.uint16))
    assert np.array_equal(d[0:8], gemm_nt(qx[:8], sx[:8], qb[0], sb[0]))
    assert np.array_equal(d[128:136], gemm_nt(qx[8:], sx[8:], qb[1], sb[1]))
    assert not d[8:128].any()  # zero padding rows: s = 0, codes 0 -> exact zeros


def test_grouped_masked_per_expert_and_untouched_rows():
    rng = np.random.default_rng(21)
    E, cap, N, K = 4, 160, 128, 256
    masked = np.array([0, 1, 160, 37])
    qa, sa = quantize_1x128(_bf16(rng, (E * cap, K)))
    qa, sa = qa.reshape(E, cap, K), sa.reshape(E, cap, K // 128)
    qbs, sbs = zip(*(quantize_128x128(_bf16(rng, (N, K), 0.05)) for _ in range(E)))
    qb, sb = np.stack(qbs), np.stack(sbs)
    init = np.full((E, cap, N), 0xABCD, np.uint16)
    d = grouped_masked(qa, sa, qb, sb, masked, init)
    for e in range(E):
        m = masked[e]
        if m:
            assert np.array_equal(d[e, :m], gemm_nt(qa[e, :m], sa[e, :m], qb[e], sb[e]))
        assert np.all(d[e, m:] == 0xABCD)
