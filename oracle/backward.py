"""Gradient (backward) GEMMs with e5m2 gradients (oracle; test infrastructure only).

[WT] sec. 2.1 and [PT] "E4M3 vs E5M2": gradients use e5m2 (range to 57344), activations and
weights e4m3.  The pages name the backward GEMMs but give no layout; the readings here:

  * quantisation of a gradient: the 1x128 rule of quantize.py with the e5m2 maximum,
        s = fp32(amax / 57344),  q = e5m2_encode(fp32(x / s));
  * data gradient dX = dY * W as an NT GEMM: A = dY [M, N] (e5m2, 1x128 scales along N),
    B = W^T [K, N] (e4m3, 128x128 block scales); the promotion chain of gemm.py;
  * weight gradient of a grouped MoE layer, dW[e] = dY_e^T * X_e, summed over the tokens of
    expert e: an NT GEMM whose contraction runs over tokens and is grouped by expert
    ("K-grouped"): A = dY^T [N, T] (e5m2) and B = X^T [K, T] (e4m3), both with one scale per
    row and 128-token block; expert e owns tokens offsets[e] .. offsets[e+1]-1, each a multiple
    of 128, so no token block spans two experts.  Both scales vary along the contraction, so
    each block's partial sum takes the product of its row's and its column's scale:
        acc[m, n] = sum over the expert's blocks kb of  P_kb[m, n] * (sA[m, kb] * sB[n, kb])
    with the fp32 rounding of gemm.py; an expert with no tokens gets dW = 0.

Block sums of e5m2 x e4m3 products are not always exact in float64 (the values span
2^-16 .. 2^15.8 and 2^-9 .. 2^8.8, so a sum of 128 products can need 57 bits).  They are
computed exactly in int64 (codes as integers in units of 2^-16 and 2^-9) and rounded once to
fp32: exactly through float64 when below 2^53 units, else by integer round-to-nearest-even.
"""

from __future__ import annotations

import numpy as np

from .e4m3 import bf16_round_bits, e4m3_decode
from .e5m2 import E5M2_MAX, e5m2_decode, e5m2_encode

BLOCK = 128
_UNIT = {"e4m3": 9, "e5m2": 16}  # values are integers in units of 2^-UNIT
_DEC = {"e4m3": e4m3_decode, "e5m2": e5m2_decode}


def quantize_1x128_e5m2(x: np.ndarray):
    """x float32 [M, K] (bf16 values), K % 128 == 0 -> (q uint8 [M, K] e5m2, s float32 [M, K/128])."""
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % BLOCK == 0
    xb = x.reshape(M, K // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=2, initial=np.float32(0.0)).astype(np.float32)
    s = (amax / np.float32(E5M2_MAX)).astype(np.float32)
    zero = s == 0
    y = (xb / np.where(zero, np.float32(1.0), s)[:, :, None]).astype(np.float32)
    q = np.where(zero[:, :, None], np.uint8(0), e5m2_encode(y)).astype(np.uint8)
    return q.reshape(M, K), s


def _as_int(codes: np.ndarray, fmt: str) -> np.ndarray:
    v = _DEC[fmt](codes) * 2.0 ** _UNIT[fmt]
    assert np.all(np.isfinite(v)), "non-finite code"
    return v.astype(np.int64)  # exact: integers below 2^32


def _round_int_f32(v: np.ndarray, unit: int) -> np.ndarray:
    """Exact integers v (int64) times 2^-unit -> float32, rounded once to nearest-even."""
    out = (v.astype(np.float64) * 2.0 ** -unit).astype(np.float32)  # exact float64 below 2^53
    for idx in zip(*np.nonzero(np.abs(v) >= (1 << 53))):
        a = int(v[idx])
        mag = abs(a)
        sh = mag.bit_length() - 24
        q, r = divmod(mag, 1 << sh)
        half = 1 << (sh - 1)
        if r > half or (r == half and q & 1):
            q += 1
        out[idx] = np.float32((-1 if a < 0 else 1) * float(q << sh) * 2.0 ** -unit)
    return out


def block_products(qa, a_fmt, qb, b_fmt):
    """P [KB, M, N] float32: each 128-wide K block's exact dot products, rounded once to fp32."""
    A, B = _as_int(qa, a_fmt), _as_int(qb, b_fmt)
    M, K = A.shape
    KB = K // BLOCK
    unit = _UNIT[a_fmt] + _UNIT[b_fmt]
    P = np.empty((KB, M, B.shape[0]), dtype=np.float32)
    for kb in range(KB):
        cols = slice(kb * BLOCK, (kb + 1) * BLOCK)
        P[kb] = _round_int_f32(A[:, cols] @ B[:, cols].T, unit)
    return P


def _promote(P, sa, sb_cols):
    """acc = fp32(acc + fp32(P_kb * fp32(sa[m, kb] * sb_cols[n, kb]))), kb ascending; bf16 bits."""
    KB, M, N = P.shape
    acc = np.zeros((M, N), dtype=np.float32)
    for kb in range(KB):
        s = (sa[:, kb][:, None] * sb_cols[:, kb][None, :]).astype(np.float32)
        acc = (acc + (P[kb] * s).astype(np.float32)).astype(np.float32)
    return bf16_round_bits(acc)


def gemm_nt_dgrad(qa, sa, qb, sb):
    """Data gradient: qa e5m2 [M, K] with sa [M, K/128]; qb e4m3 [N, K] with 128x128 scales
    sb [ceil(N/128), K/128].  Returns bf16 bits [M, N]."""
    P = block_products(qa, "e5m2", qb, "e4m3")
    sb = np.asarray(sb, np.float32)
    return _promote(P, np.asarray(sa, np.float32), sb[np.arange(qb.shape[0]) // BLOCK])


def wgrad_k_grouped(qa, sa, qb, sb, offsets):
    """Weight gradient over experts: qa e5m2 [N, T] with sa [N, T/128]; qb e4m3 [K, T] with
    sb [K, T/128]; offsets int [E+1] (multiples of 128, non-decreasing, offsets[E] <= T).
    Returns bf16 bits [E, N, K]."""
    N, K = qa.shape[0], qb.shape[0]
    off = [int(v) for v in offsets]
    E = len(off) - 1
    out = np.zeros((E, N, K), dtype=np.uint16)
    sa, sb = np.asarray(sa, np.float32), np.asarray(sb, np.float32)
    for e in range(E):
        t0, t1 = off[e], off[e + 1]
        if t1 > t0:
            b0, b1 = t0 // BLOCK, t1 // BLOCK
            P = block_products(qa[:, t0:t1], "e5m2", qb[:, t0:t1], "e4m3")
            out[e] = _promote(P, sa[:, b0:b1], sb[:, b0:b1])
    return out
