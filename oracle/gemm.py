"""Blockwise-dequantised FP8 GEMM and its grouped MoE forms (oracle; test infrastructure only).

What is computed ("NT": A [M,K] and B [N,K] both K-contiguous, [EX] sec. 3.3):

    D[m, n] = bf16( sum over kb of  P_kb[m, n] * (sA[m, kb] * sB[n // 128, kb]) )
    P_kb[m, n] = sum over k in block kb of  dec(A[m, k]) * dec(B[n, k])

[WT] sec. 2.3: accumulation stays FP32 across the whole K and the result is
rounded to the output type only when written.  [WT] sec. 2.2 and [PT] (Triton
listing, fused epilogue): the scales are applied inside the GEMM, not by a
separate dequantisation pass.  The listing on [PT] multiplies the accumulator
by one scalar pair at the end, which is only right for per-tensor scales; with a
scale per 128-wide K block the only consistent reading is to scale each
block's partial sum before adding it (per-block promotion).  Oracle steps:

    P_kb   in float64 -- exact: every e4m3 value is an integer multiple of 2^-9
           below 2^9, so products are integers below 2^36 in units of 2^-18 and a
           sum of 128 of them stays below 2^43 < 2^53, in any order;
    s      = fp32(sA * sB);  t = fp32(fp32(P_kb) * s);  acc = fp32(acc + t),
           kb ascending from acc = 0;
    D      = bf16 round-to-nearest-even of acc.

Grouped forms ([EX] sec. 3.2, [WT] sec. 1.2 and 5.3): several experts with
different token counts in one call.  Contiguous: each expert's rows are one
contiguous, 128-aligned range of A given by group offsets; the result is the
per-expert dense GEMM on those rows.  Masked: A is [E, cap, K] and only the first
masked_m[e] rows of expert e are computed; the other rows of D are left as
they were.
"""

from __future__ import annotations

import numpy as np

from .e4m3 import bf16_round_bits, e4m3_decode

BLOCK = 128


def gemm_nt(qa, sa, qb, sb, n_index=None, return_acc=False):
    """qa uint8 [M,K], sa float32 [M,K/128], qb uint8 [N,K], sb float32 [ceil(N/128),K/128].

    ``n_index`` (int [N]) gives the original column number of each row of qb
    when qb is a subset of a weight matrix (its scale row is sb[n_index // 128]);
    default 0..N-1.  Returns bf16 bits uint16 [M, N] (and the fp32 accumulator).
    """
    qa = np.asarray(qa, dtype=np.uint8)
    qb = np.asarray(qb, dtype=np.uint8)
    M, K = qa.shape
    N = qb.shape[0]
    assert qb.shape[1] == K and K % BLOCK == 0
    if n_index is None:
        n_index = np.arange(N)
    n_block = np.asarray(n_index) // BLOCK
    sa = np.asarray(sa, dtype=np.float32)
    sb = np.asarray(sb, dtype=np.float32)
    A = e4m3_decode(qa)  # float64
    B = e4m3_decode(qb)
    acc = np.zeros((M, N), dtype=np.float32)
    for kb in range(K // BLOCK):
        cols = slice(kb * BLOCK, (kb + 1) * BLOCK)
        p = A[:, cols] @ B[:, cols].T  # float64, exact
        s = (sa[:, kb][:, None] * sb[n_block, kb][None, :]).astype(np.float32)
        t = (p.astype(np.float32) * s).astype(np.float32)
        acc = (acc + t).astype(np.float32)
    d = bf16_round_bits(acc)
    return (d, acc) if return_acc else d


def grouped_contiguous(qa, sa, qb, sb, group_offsets, d_init):
    """Contiguous grouped GEMM.

    qa [M_total,K], sa [M_total,K/128], qb [E,N,K], sb [E,ceil(N/128),K/128],
    group_offsets int [E+1] (non-decreasing, multiples of 128), d_init uint16
    [M_total,N] (bf16 bits).  Rows of expert e are offsets[e] .. offsets[e+1]-1;
    rows outside every group keep d_init.  Returns uint16 [M_total, N].
    """
    d = np.array(d_init, dtype=np.uint16, copy=True)
    off = [int(v) for v in group_offsets]
    for e in range(len(off) - 1):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            d[r0:r1] = gemm_nt(qa[r0:r1], sa[r0:r1], qb[e], sb[e])
    return d


def grouped_masked(qa, sa, qb, sb, masked_m, d_init):
    """Masked grouped GEMM.

    qa [E,cap,K], sa [E,cap,K/128], qb [E,N,K], sb [E,ceil(N/128),K/128],
    masked_m int [E] (0 <= masked_m[e] <= cap), d_init uint16 [E,cap,N].
    Rows m < masked_m[e] of expert e get that expert's GEMM; the others keep
    d_init.  Returns uint16 [E, cap, N].
    """
    d = np.array(d_init, dtype=np.uint16, copy=True)
    for e in range(qa.shape[0]):
        m = int(masked_m[e])
        if m > 0:
            d[e, :m] = gemm_nt(qa[e, :m], sa[e, :m], qb[e], sb[e])
    return d
