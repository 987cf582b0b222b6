"""GPU parity of route-gather-quantize (the contiguous grouped layout built on the device from
routed tokens) against the oracle: group offsets, row->token map, e4m3 codes and scales, all
bit-exact."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from moe_grouped_gemm_block_gb300.workloads import WORKLOADS, make_inputs, route_top2
from oracle import quantize_1x128, route_gather_quantize, route_layout
from tests.gpu_util import check_status, need_gpu, sa_from_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    need_gpu()


def _tokens(T, K, seed):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn((T, K), generator=gen) * 2).to(torch.bfloat16)


def _run(x, ids, E, m_cap=None):
    q, sA, offs, rows, ent = g.route_gather_quantize_1x128(x.cuda(), torch.from_numpy(ids).cuda(), E, m_cap)
    torch.cuda.synchronize()
    return (q.cpu().numpy(), sa_from_device(sA, q.shape[0]), offs.cpu().numpy(), rows.cpu().numpy(),
            ent.cpu().numpy())


def _entry_rows(ids, offs, E):
    """The row of each (token, slot) entry under the layout rule: an expert's rows start at its
    offset and are handed out in (token, slot) order; -1 for an id outside [0, E)."""
    ent = np.full(ids.shape, -1, np.int32)
    nxt = [int(o) for o in offs[:E]]
    for t in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            if 0 <= e < E:
                ent[t, j] = nxt[e]
                nxt[e] += 1
    return ent


def _check_entries(ent, ids, offs_r, rows_r, E):
    want = _entry_rows(ids, offs_r, E)
    valid = want >= 0
    # the rule agrees with the oracle's row -> token map, and the library's map is that rule's
    assert np.array_equal(rows_r[want[valid]], np.nonzero(valid)[0])
    assert np.array_equal(ent, want)


def _check(x, ids, E, m_cap=None):
    q, sA, offs, rows, ent = _run(x, ids, E, m_cap)
    check_status()
    q_r, s_r, offs_r, rows_r = route_gather_quantize(x.float().numpy(), ids, E, q.shape[0])
    assert np.array_equal(offs, offs_r)
    assert np.array_equal(rows, rows_r)
    _check_entries(ent, ids, offs_r, rows_r, E)
    assert np.array_equal(q, q_r)
    assert np.array_equal(sA.view(np.uint32), s_r.view(np.uint32))


def _routing(T, E, k, seed):
    gen = torch.Generator().manual_seed(seed)
    experts, _ = route_top2(torch.randn((T, E), generator=gen), k)
    return experts.reshape(T, k).numpy().astype(np.int32)


@pytest.mark.parametrize("T,E,k,K", [(300, 8, 2, 512), (1, 1, 1, 128), (5, 64, 4, 256), (1000, 3, 1, 384),
                                     (700, 256, 2, 128)])
def test_route_gather_quantize_small(T, E, k, K):
    _check(_tokens(T, K, T + E), _routing(T, E, k, T * E), E)


@pytest.mark.parametrize("E", [8, 300])
def test_many_entries(E):
    # 66000 entries: 2063 per warp of the layout kernel for up to 256 experts, past the 512 ids it
    # keeps in registers; 300 experts take the kernel for more
    T, k, K = 33000, 2, 128
    _check(_tokens(T, K, 77), _routing(T, E, k, 78 + E), E)


def test_many_empty_experts_and_a_larger_capacity():
    ids = np.array([[2047], [5], [5], [2047], [0]], dtype=np.int32)
    _check(_tokens(5, 256, 3), ids, 2048, m_cap=g.route_capacity(5, 1, 2048) + 256)


def test_a_token_naming_one_expert_twice_gets_two_rows():
    ids = np.array([[1, 1], [0, 1], [1, 0]], dtype=np.int32)
    _check(_tokens(3, 128, 4), ids, 2)


def test_no_tokens():
    x = torch.empty((0, 256), dtype=torch.bfloat16)
    ids = np.zeros((0, 2), dtype=np.int32)
    q, sA, offs, rows, ent = _run(x, ids, 4)
    check_status()
    assert not offs.any() and np.all(rows == -1) and not q.any() and not sA.any() and ent.size == 0


def test_ids_out_of_range_are_dropped_and_flagged():
    x = _tokens(6, 128, 5)
    ids = np.array([[0, 7], [1, -1], [0, 1], [3, 2], [2, 0], [9, 1]], dtype=np.int32)
    q, sA, offs, rows, ent = _run(x, ids, 4)
    assert g.fp8g_get_status() == 6  # FP8G_ERR_DEVICE_ASSERT
    # the layout of the valid entries alone (out-of-range entries replaced by a fifth expert)
    ids5 = np.where((ids >= 0) & (ids < 4), ids, 4)
    offs5, rows5 = route_layout(ids5, 5)
    assert np.array_equal(offs, offs5[:5])
    assert np.array_equal(rows[:offs5[4]], rows5[:offs5[4]]) and np.all(rows[offs5[4]:] == -1)
    assert np.array_equal(ent, _entry_rows(ids, offs5, 4))  # dropped entries: -1


@pytest.mark.parametrize("T,E,k", [(1111, 8, 2), (1500, 32, 2), (4097, 5, 1), (2048, 1, 1)])
def test_layout_over_several_ctas(T, E, k):
    # 2048 entries or more of at most 32 experts: the layout kernel over several CTAs (uneven
    # ranges and warp slices of fewer than 32 entries included); the same layout as the oracle's
    _check(_tokens(T, 128, T + 11 * E), _routing(T, E, k, 5 * T + E), E)


def test_layout_over_several_ctas_drops_ids_out_of_range():
    T, E = 1200, 6
    ids = _routing(T, E, 2, 99)
    ids[7, 1], ids[400, 0], ids[1199, 1], ids[0, 0] = -3, 6, 1000, -1
    x = _tokens(T, 128, 12)
    q, sA, offs, rows, ent = _run(x, ids, E)
    assert g.fp8g_get_status() == 6  # FP8G_ERR_DEVICE_ASSERT
    ids7 = np.where((ids >= 0) & (ids < E), ids, E)
    offs7, rows7 = route_layout(ids7, E + 1)
    assert np.array_equal(offs, offs7[:E + 1])
    assert np.array_equal(rows[:offs7[E]], rows7[:offs7[E]]) and np.all(rows[offs7[E]:] == -1)
    assert np.array_equal(ent, _entry_rows(ids, offs7, E))


def test_full_size_moe_contiguous_layout():
    w = WORKLOADS["moe_contiguous"]
    inp = make_inputs(w, "cuda")
    ids = inp["topk_ids"].numpy()
    q, sA, offs, rows, ent = g.route_gather_quantize_1x128(inp["tokens"], inp["topk_ids"].cuda(), w.E)
    torch.cuda.synchronize()
    check_status()
    offs_r, rows_r = route_layout(ids, w.E, q.shape[0])
    assert np.array_equal(offs.cpu().numpy(), offs_r) and np.array_equal(rows.cpu().numpy(), rows_r)
    _check_entries(ent.cpu().numpy(), ids, offs_r, rows_r, w.E)
    # the rows equal the quantisation of the generator's gathered A, row for row
    m_total = inp["A"].shape[0]
    assert int(offs_r[-1]) == m_total
    q_a, s_a = g.quantize_1x128(inp["A"])
    torch.cuda.synchronize()
    assert torch.equal(q[:m_total], q_a)
    assert torch.equal(sA[:, :m_total], s_a[:, :m_total])
    assert not q[m_total:].any() and not sA[:, m_total:].any()
    # and sampled rows agree with the oracle
    rng = np.random.default_rng(0)
    sample = rng.choice(m_total, 96, replace=False)
    tok = rows_r[sample]
    xs = inp["tokens"].float().cpu().numpy()
    gathered = np.where((tok >= 0)[:, None], xs[np.maximum(tok, 0)], 0.0).astype(np.float32)
    q_o, s_o = quantize_1x128(gathered)
    assert np.array_equal(q[sample].cpu().numpy(), q_o)
    assert np.array_equal(sa_from_device(sA, q.shape[0])[sample], s_o)


def test_routed_layout_feeds_the_contiguous_gemm():
    # route-gather-quantize, then the grouped GEMM with M_total = capacity: the routed rows match
    # the GEMM of the generator's layout, and rows past the last group are left untouched
    w = WORKLOADS["moe_contiguous"]
    T, E, k, N, K = 260, 4, 2, 256, 512
    x = _tokens(T, K, 11)
    ids = _routing(T, E, k, 11)
    q, sA, offs, rows, _ = g.route_gather_quantize_1x128(x.cuda(), torch.from_numpy(ids).cuda(), E)
    gen = torch.Generator().manual_seed(12)
    Bq, sB = g.quantize_128x128((torch.randn((E, N, K), generator=gen) / np.sqrt(K)).to(torch.bfloat16).cuda())
    m_cap = q.shape[0]
    D = torch.full((m_cap, N), 7.0, dtype=torch.bfloat16, device="cuda")
    g.fp8_grouped_gemm_contiguous(q, sA, Bq, sB, D, offs)
    torch.cuda.synchronize()
    check_status()
    m_total = int(offs[-1])
    # the same GEMM on the rows the layout produced, compacted to exactly m_total rows
    D2 = torch.empty((m_total, N), dtype=torch.bfloat16, device="cuda")
    sA2 = sA[:, :m_total].contiguous()
    g.fp8_grouped_gemm_contiguous(q[:m_total].contiguous(), sA2, Bq, sB, D2, offs)
    torch.cuda.synchronize()
    check_status()
    assert torch.equal(D[:m_total], D2)
    assert torch.all(D[m_total:] == 7.0)
