"""Per-tensor and per-channel scaled FP8 GEMM (oracle; test infrastructure only).

"DeepGEMM FP8 walk-through" sec. 2.2: the coarsest choice is one scale for a whole tensor
(per-tensor); finer ones scale the activations A per token (one scale per row of A) and
the weights B per channel (one scale per output channel, a row of B [N, K]).
"Production FP8 GEMM alignment and Tensor Core peak tuning" (Triton listing, fused
epilogue): the FP32 accumulator of the whole K is multiplied once, in registers, by
scale_a * scale_b and converted to BF16.

Quantisation follows the same rules as ``quantize.py``, with the scaling group a whole
row or the whole tensor:
    amax = max |x| over the group        (exact in fp32)
    s    = fp32(amax / 448)              (a zero group: s = 0, codes 0x00)
    q    = e4m3_encode(fp32(x / s))

GEMM ("NT": A [M, K], B [N, K]):
    acc[m, n] = sum over k of dec(A[m, k]) * dec(B[n, k])   in float64, exact: the
                products are integers below 2^36 in units of 2^-18, so a sum of K of them
                stays below 2^53 for K < 2^17, in any order;
    D[m, n]   = bf16( fp32( fp32(acc) * fp32(sa[m] * sb[n]) ) )
with sa one value (per-tensor) or one per row of A (per-token), and sb one value or one per
row of B (per-channel).

Grouped forms as in ``gemm.py``: contiguous (expert e owns rows offsets[e] .. offsets[e+1]-1)
and masked (A [E, cap, K], the first masked_m[e] rows of expert e).  A's scales are indexed
by the row of the whole A (M_total or E * cap rows), or are one value; B's are [E, N] or
[E, 1] (one per expert).
"""

from __future__ import annotations

import numpy as np

from .e4m3 import E4M3_MAX, bf16_round_bits, e4m3_decode, e4m3_encode


def _quantize_group(x: np.ndarray, amax: np.ndarray):
    """x float32, amax float32 broadcastable to x."""
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    zero = s == 0
    y = (x / np.where(zero, np.float32(1.0), s)).astype(np.float32)
    q = np.where(zero, np.uint8(0), e4m3_encode(y)).astype(np.uint8)
    return q, s


def quantize_per_row(x: np.ndarray):
    """x float32 [M, K] (bf16 values).  Returns (q uint8 [M, K], s float32 [M])."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1, initial=np.float32(0.0)).astype(np.float32)
    q, s = _quantize_group(x, amax[:, None])
    return q, s[:, 0]


def quantize_per_tensor(x: np.ndarray):
    """x float32 [..., K] (bf16 values), one tensor.  Returns (q uint8, s float32 [1])."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.abs(x).max(initial=np.float32(0.0)))
    q, s = _quantize_group(x, np.full((1,) * x.ndim, amax, np.float32))
    return q, s.reshape(1)


def _col(v: np.ndarray, n: int) -> np.ndarray:
    v = np.asarray(v, dtype=np.float32).reshape(-1)
    assert v.size in (1, n), (v.size, n)
    return np.broadcast_to(v, (n,))


def gemm_nt_scaled(qa, sa, qb, sb, return_acc=False):
    """qa uint8 [M, K], sa float32 [M] or [1], qb uint8 [N, K], sb float32 [N] or [1].

    Returns bf16 bits uint16 [M, N] (and the fp32 accumulator before scaling).
    """
    qa = np.asarray(qa, dtype=np.uint8)
    qb = np.asarray(qb, dtype=np.uint8)
    M, K = qa.shape
    N = qb.shape[0]
    assert qb.shape[1] == K
    acc = (e4m3_decode(qa) @ e4m3_decode(qb).T).astype(np.float32)  # exact float64, one rounding
    s = (_col(sa, M)[:, None] * _col(sb, N)[None, :]).astype(np.float32)
    d = bf16_round_bits((acc * s).astype(np.float32))
    return (d, acc) if return_acc else d


def _expert_scales(sb: np.ndarray, E: int, N: int) -> np.ndarray:
    sb = np.asarray(sb, dtype=np.float32)
    assert sb.shape in ((E, N), (E, 1), (E,)), sb.shape
    return sb.reshape(E, -1)


def grouped_contiguous_scaled(qa, sa, qb, sb, group_offsets, d_init):
    """qa [M_total, K], sa [M_total] or [1], qb [E, N, K], sb [E, N] or [E, 1],
    group_offsets int [E+1] (non-decreasing, multiples of 128), d_init uint16 [M_total, N]."""
    d = np.array(d_init, dtype=np.uint16, copy=True)
    E, N = qb.shape[0], qb.shape[1]
    sa = _col(sa, qa.shape[0])
    sbe = _expert_scales(sb, E, N)
    off = [int(v) for v in group_offsets]
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            d[r0:r1] = gemm_nt_scaled(qa[r0:r1], sa[r0:r1], qb[e], sbe[e])
    return d


def grouped_masked_scaled(qa, sa, qb, sb, masked_m, d_init):
    """qa [E, cap, K], sa [E * cap] or [1], qb [E, N, K], sb [E, N] or [E, 1],
    masked_m int [E], d_init uint16 [E, cap, N].  Rows m >= masked_m[e] keep d_init."""
    d = np.array(d_init, dtype=np.uint16, copy=True)
    E, cap = qa.shape[0], qa.shape[1]
    N = qb.shape[1]
    sa = _col(sa, E * cap).reshape(E, cap)
    sbe = _expert_scales(sb, E, N)
    for e in range(E):
        m = int(masked_m[e])
        if m > 0:
            d[e, :m] = gemm_nt_scaled(qa[e, :m], sa[e, :m], qb[e], sbe[e])
    return d
