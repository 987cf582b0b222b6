"""Pins of the oracle's route-gather-quantize (oracle/route.py) without a GPU.

Pinned against: the input generator's own, separately written layout builder
(moe_grouped_gemm_block_gb300.workloads.contiguous_layout, used to make the contiguous GEMM's
inputs), the layout's invariants on random routings, a small case worked by hand (two experts,
eight tokens: "DeepGEMM walk-through" sec. 5.3 names such a case), and the 1x128 quantiser on the
gathered rows."""

import numpy as np
import pytest
import torch

from moe_grouped_gemm_block_gb300.workloads import contiguous_layout, route_top2
from oracle import quantize_1x128, route_gather_quantize, route_layout


def _routing(T, E, k, seed):
    gen = torch.Generator().manual_seed(seed)
    logits = torch.randn((T, E), generator=gen)
    experts, _ = route_top2(logits, k)
    return experts.reshape(T, k).numpy().astype(np.int32)


@pytest.mark.parametrize("T,E,k,seed", [(300, 8, 2, 1), (4096, 8, 2, 4), (50, 64, 4, 2), (7, 3, 1, 3)])
def test_layout_matches_the_input_generators_layout(T, E, k, seed):
    ids = _routing(T, E, k, seed)
    offs, rows = route_layout(ids, E)
    tok = torch.arange(T).unsqueeze(1).expand(T, k).reshape(-1)
    ref_rows, ref_offs = contiguous_layout(torch.from_numpy(ids).reshape(-1).long(), tok, E)
    assert np.array_equal(offs, ref_offs.numpy())
    assert np.array_equal(rows, ref_rows.numpy().astype(np.int32))


@pytest.mark.parametrize("seed", range(5))
def test_layout_invariants(seed):
    rng = np.random.default_rng(seed)
    T, E, k = int(rng.integers(1, 400)), int(rng.integers(1, 40)), int(rng.integers(1, 5))
    ids = np.stack([rng.choice(E, size=min(k, E), replace=False) for _ in range(T)]).astype(np.int32)
    k = ids.shape[1]
    cap = ((T * k + E * 127 + 127) // 128) * 128
    offs, rows = route_layout(ids, E, cap)
    assert offs[0] == 0 and np.all(np.diff(offs) >= 0) and np.all(offs % 128 == 0)
    counts = np.bincount(ids.ravel(), minlength=E)
    assert np.array_equal(np.diff(offs), (counts + 127) // 128 * 128)
    assert rows.size == cap and np.all(rows[offs[E]:] == -1)
    for e in range(E):
        seg = rows[offs[e]:offs[e + 1]]
        toks = seg[:counts[e]]
        assert np.all(seg[counts[e]:] == -1)
        assert np.all(np.diff(toks) > 0)  # ascending tokens
        assert np.array_equal(np.sort(toks), np.sort(np.nonzero((ids == e).any(axis=1))[0]))


def test_two_experts_eight_tokens_by_hand():
    ids = np.array([[1], [0], [0], [1], [1], [0], [1], [1]], dtype=np.int32)
    offs, rows = route_layout(ids, 2)
    assert offs.tolist() == [0, 128, 256]
    assert rows[:4].tolist() == [1, 2, 5, -1] and np.all(rows[3:128] == -1)
    assert rows[128:134].tolist() == [0, 3, 4, 6, 7, -1] and np.all(rows[133:] == -1)


def test_gathered_rows_quantise_like_their_tokens():
    gen = torch.Generator().manual_seed(9)
    x = (torch.randn((40, 512), generator=gen) * 3).to(torch.bfloat16).float().numpy()
    ids = _routing(40, 5, 2, 9)
    q, sA, offs, rows = route_gather_quantize(x, ids, 5, m_cap=640)
    q_tok, s_tok = quantize_1x128(x)
    for r in range(640):
        t = rows[r]
        if t >= 0:
            assert np.array_equal(q[r], q_tok[t]) and np.array_equal(sA[r], s_tok[t])
        else:
            assert not q[r].any() and not sA[r].any()  # zero rows: scale 0, codes 0


def test_out_of_contract_inputs_are_rejected():
    with pytest.raises(ValueError):
        route_layout(np.array([[0], [3]], dtype=np.int32), 3)
    with pytest.raises(ValueError):
        route_layout(np.array([[0], [1]], dtype=np.int32), 2, m_cap=128)
