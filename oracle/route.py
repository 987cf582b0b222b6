"""Route-gather-quantize: the contiguous grouped layout built from routed tokens -- TEST
INFRASTRUCTURE ONLY (see the package docstring).

Pages: [EX] "DeepGEMM explainer" sec. 3.2 (the MoE grouped GEMM takes experts with different token
counts in one call) and sec. 4.2 (the call takes the group sizes); [WT] "DeepGEMM FP8 walk-through"
sec. 5.3 (pass each group's id and its token offset; keep each expert's rows contiguous and
block-loadable).  The layout is the one the contiguous grouped GEMM reads: expert e owns rows
offsets[e] .. offsets[e+1]-1, holding its routed tokens in ascending order, then zero rows up to
a multiple of 128.  Those rows are then quantised exactly like any activation rows (quantize.py).

Readings where the pages are silent: a token whose top-k list names the same expert twice gets
one row per entry, entries ordered by (token, slot); rows past offsets[E] up to the caller's
capacity are zero rows with token -1; expert ids outside [0, E) are out of contract (rejected
here; the library drops them and raises its device-assert status).
"""

from __future__ import annotations

import numpy as np

from .quantize import quantize_1x128

GROUP = 128


def route_layout(topk_ids: np.ndarray, E: int, m_cap: int | None = None):
    """(group_offsets int32 [E+1], row_token int32 [m_cap]) for expert choices topk_ids [T, k]."""
    ids = np.asarray(topk_ids)
    T, k = ids.shape
    if ids.size and (ids.min() < 0 or ids.max() >= E):
        raise ValueError("expert id out of range")
    members = [[] for _ in range(E)]  # per expert: its tokens, in (token, slot) order
    for t in range(T):
        for j in range(k):
            members[int(ids[t, j])].append(t)
    offsets = [0]
    for e in range(E):
        n = len(members[e])
        offsets.append(offsets[-1] + (n + GROUP - 1) // GROUP * GROUP)
    m_cap = offsets[E] if m_cap is None else m_cap
    if m_cap < offsets[E]:
        raise ValueError("capacity below the padded row count")
    row_token = np.full(m_cap, -1, dtype=np.int32)
    for e in range(E):
        for i, t in enumerate(members[e]):
            row_token[offsets[e] + i] = t
    return np.array(offsets, dtype=np.int32), row_token


def route_gather_quantize(x: np.ndarray, topk_ids: np.ndarray, E: int, m_cap: int | None = None):
    """Tokens x [T, K] (bf16 values as float32) and their expert choices topk_ids [T, k] ->
    (q uint8 [m_cap, K], sA float32 [m_cap, K/128], group_offsets, row_token): the gathered rows in
    the contiguous grouped layout, quantised 1x128 (zero rows: scale 0, codes 0)."""
    x = np.asarray(x, dtype=np.float32)
    offsets, row_token = route_layout(topk_ids, E, m_cap)
    gathered = np.zeros((row_token.size, x.shape[1]), dtype=np.float32)
    used = row_token >= 0
    gathered[used] = x[row_token[used]]
    q, sA = quantize_1x128(gathered)
    return q, sA, offsets, row_token
