"""Block quantisation to e4m3 (oracle; test infrastructure only).

[EX] sec. 3.1: the matrix is cut into blocks, each with its own scale; with amax
the block's largest magnitude the scale is amax divided by the largest FP8 value;
quantising divides each element by the scale, dequantising multiplies it back.
[WT] sec. 5.2 gives the same scale, max_val / 448.  [WT] sec. 2.2: activations
A are grouped per token, weights B per channel, with K cut into blocks; the
block edges here are 1x128 for A (one scale per row and 128-wide K block) and
128x128 for B.

All arithmetic is IEEE binary32 with round-to-nearest-even and subnormals kept:
    amax = max |x| over the block        (exact: bf16 values are exact in fp32)
    s    = fp32(amax / 448)
    q_i  = e4m3_encode(fp32(x_i / s))
A block whose amax is 0 (for example a zero padding row) has s = 0 and all codes
0x00: the quotient 0/0 is not formed.  Inputs must be finite.
"""

from __future__ import annotations

import numpy as np

from .e4m3 import E4M3_MAX, e4m3_encode

BLOCK = 128


def _quantize_blocks(xb: np.ndarray, amax: np.ndarray):
    """xb: float32 [..., blocks..., elements]; amax broadcastable float32."""
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    zero = s == 0
    safe = np.where(zero, np.float32(1.0), s).astype(np.float32)
    y = (xb / safe).astype(np.float32)
    q = e4m3_encode(y)
    q = np.where(zero, np.uint8(0), q).astype(np.uint8)
    return q, s


def quantize_1x128(x: np.ndarray):
    """x: float32 [M, K] (bf16 values), K % 128 == 0.

    Returns (q uint8 [M, K], s float32 [M, K/128]); s[m, kb] is the scale of
    row m, columns kb*128 .. kb*128+127.
    """
    x = np.asarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % BLOCK == 0
    xb = x.reshape(M, K // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=2, initial=np.float32(0.0)).astype(np.float32)
    q, s = _quantize_blocks(xb, amax[:, :, None])
    return q.reshape(M, K), s[:, :, 0]


def quantize_128x128(w: np.ndarray):
    """w: float32 [N, K] (bf16 values), K % 128 == 0, any N.

    Returns (q uint8 [N, K], s float32 [ceil(N/128), K/128]); s[nb, kb] is the
    scale of rows nb*128 .. nb*128+127 (those that exist) and columns
    kb*128 .. kb*128+127.
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % BLOCK == 0
    NB, KB = -(-N // BLOCK), K // BLOCK
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty((NB, KB), dtype=np.float32)
    for nb in range(NB):
        rows = w[nb * BLOCK:(nb + 1) * BLOCK]  # the rows of this block that exist
        rb = rows.reshape(rows.shape[0], KB, BLOCK)
        amax = np.abs(rb).max(axis=(0, 2), initial=np.float32(0.0)).astype(np.float32)
        qb, sb = _quantize_blocks(rb, amax[None, :, None])
        q[nb * BLOCK:(nb + 1) * BLOCK] = qb.reshape(rows.shape[0], K)
        s[nb] = sb[0, :, 0]
    return q, s
