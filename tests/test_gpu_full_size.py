"""Every output element of the full-size workloads against the oracle.

For each workload the GPU quantises the bf16 activations (1x128) and weights (128x128) and runs
the GEMM in the configuration the benchmark times.  On the host the oracle quantises the same bf16
inputs (they must give the GPU's codes and scales bit for bit) and computes the blockwise-
dequantised GEMM from its own codes, so no oracle input comes from the CUDA path.  The whole of D
is then compared at the GEMM tolerance (per element and relative Frobenius); in the masked form
every row past an expert's count must still hold the sentinel.  The oracle runs in a pool of
spawned worker processes, split by rows, weight blocks and experts.
"""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from moe_grouped_gemm_block_gb300.workloads import WORKLOADS, make_inputs
from tests import oracle_jobs
from tests.gpu_util import assert_gemm_close, bf16_to_np, check_status, env_var, need_gpu, sa_from_device

pytestmark = pytest.mark.gpu
SENTINEL = 0x7FC1  # a bf16 NaN bit pattern no GEMM produces


@pytest.fixture(scope="module")
def ex():
    with oracle_jobs.pool() as p:
        yield p


def _chunks(n, parts, unit=1):
    """Boundaries splitting range(n) into about `parts` pieces, each a multiple of `unit`."""
    step = max(unit, -(-n // parts) // unit * unit)
    return [(a, min(n, a + step)) for a in range(0, n, step)]


def _oracle_acts(ex, A_np):
    """Oracle 1x128 codes and scales [rows, K/128] of A, computed in row chunks."""
    futs = [ex.submit(oracle_jobs.quantize_rows, A_np[a:b]) for a, b in _chunks(A_np.shape[0], 16)]
    parts = [f.result() for f in futs]
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def _oracle_weights(ex, B_np):
    """Oracle 128x128 codes and scales of one weight matrix [N, K], in chunks of 128-row blocks."""
    futs = [ex.submit(oracle_jobs.quantize_weights, B_np[a:b]) for a, b in _chunks(B_np.shape[0], 16, 128)]
    parts = [f.result() for f in futs]
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def _oracle_gemm(ex, qa, sa, qb, sb, parts=16):
    futs = [ex.submit(oracle_jobs.gemm, qa[a:b], sa[a:b], qb, sb) for a, b in _chunks(qa.shape[0], parts)]
    return np.concatenate([f.result() for f in futs])


def _assert_codes(q_gpu, s_gpu, q_ref, s_ref, what):
    assert np.array_equal(q_gpu, q_ref), f"{what}: codes differ from the oracle"
    assert np.array_equal(s_gpu.view(np.uint32), s_ref.view(np.uint32)), f"{what}: scales differ from the oracle"


@pytest.mark.parametrize("name,ck", [("decode", None), ("decode", "4"), ("large_4096", None),
                                     ("large_4096x8192", None)])
def test_dense_full_size_every_element(ex, name, ck):
    # ck: the cluster K split (FP8G_CLUSTER_K), 28 tiles of 256 columns x 4 ranks on the decode shape
    need_gpu()
    w = WORKLOADS[name]
    inp = make_inputs(w, "cuda")
    A, B = inp["A"], inp["B"]
    qA, sA = g.quantize_1x128(A)
    qB, sB = g.quantize_128x128(B)
    D = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
    with env_var("FP8G_CLUSTER_K", ck):
        g.fp8_gemm_nt(qA, sA, qB, sB, D)
        torch.cuda.synchronize()
        assert g.fp8g_last_config()["cluster_k"] == (int(ck) if ck else 0)
    check_status()
    qa, sa = _oracle_acts(ex, A.float().cpu().numpy())
    qb, sb = _oracle_weights(ex, B.float().cpu().numpy())
    _assert_codes(qA.cpu().numpy(), sa_from_device(sA, w.M), qa, sa, f"{name} A")
    _assert_codes(qB.cpu().numpy(), sB.cpu().numpy(), qb, sb, f"{name} B")
    ref = _oracle_gemm(ex, qa, sa, qb, sb)
    assert_gemm_close(bf16_to_np(D), ref, f"{name}: all {w.M}x{w.N} elements")


def test_contiguous_full_size_every_element(ex):
    need_gpu()
    w = WORKLOADS["moe_contiguous"]
    inp = make_inputs(w, "cuda")
    A, B, offs = inp["A"], inp["B"], inp["group_offsets"]
    qA, sA = g.quantize_1x128(A)
    qB, sB = g.quantize_128x128(B)
    M_total = A.shape[0]
    D = torch.empty((M_total, w.N), dtype=torch.bfloat16, device="cuda")
    g.fp8_grouped_gemm_contiguous(qA, sA, qB, sB, D, offs.cuda())
    torch.cuda.synchronize()
    check_status()
    qa, sa = _oracle_acts(ex, A.float().cpu().numpy())
    _assert_codes(qA.cpu().numpy(), sa_from_device(sA, M_total), qa, sa, "moe_contiguous A")
    B_np = B.float().cpu().numpy()
    got = bf16_to_np(D)
    offs = [int(v) for v in offs]
    assert offs[-1] == M_total
    for e in range(w.E):
        qb, sb = _oracle_weights(ex, B_np[e])
        _assert_codes(qB[e].cpu().numpy(), sB[e].cpu().numpy(), qb, sb, f"moe_contiguous B[{e}]")
        r0, r1 = offs[e], offs[e + 1]
        if r1 > r0:
            ref = _oracle_gemm(ex, qa[r0:r1], sa[r0:r1], qb, sb)
            assert_gemm_close(got[r0:r1], ref, f"moe_contiguous expert {e}: all {r1 - r0}x{w.N} elements")


def test_masked_full_size_every_element(ex):
    need_gpu()
    w = WORKLOADS["moe_masked"]
    inp = make_inputs(w, "cuda")
    A, B, masked = inp["A"], inp["B"], inp["masked_m"]
    rows = w.E * w.cap
    qA, sA = g.quantize_1x128(A.reshape(rows, w.K))
    qB, sB = g.quantize_128x128(B)
    D = torch.full((w.E, w.cap, w.N), 0, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    g.fp8_grouped_gemm_masked(qA.view(w.E, w.cap, w.K), sA, qB, sB, D, masked.cuda())
    torch.cuda.synchronize()
    check_status()
    qa, sa = _oracle_acts(ex, A.reshape(rows, w.K).float().cpu().numpy())
    _assert_codes(qA.cpu().numpy(), sa_from_device(sA, rows), qa, sa, "moe_masked A")
    B_np = B.float().cpu().numpy()
    bits = D.view(torch.int16).cpu().numpy().view(np.uint16)
    got = bf16_to_np(D)
    ms = [int(v) for v in masked]
    # one expert's weights per task (32 experts spread over the pool), then its valid rows
    wfuts = {e: ex.submit(oracle_jobs.quantize_weights, B_np[e]) for e in range(w.E) if ms[e] > 0}
    gfuts = {}
    for e, f in wfuts.items():
        qb, sb = f.result()
        _assert_codes(qB[e].cpu().numpy(), sB[e].cpu().numpy(), qb, sb, f"moe_masked B[{e}]")
        r0 = e * w.cap
        gfuts[e] = ex.submit(oracle_jobs.gemm, qa[r0:r0 + ms[e]], sa[r0:r0 + ms[e]], qb, sb)
    for e in range(w.E):
        assert np.all(bits[e, ms[e]:] == SENTINEL), f"expert {e}: rows past its count were written"
        if ms[e] > 0:
            assert_gemm_close(got[e, :ms[e]], gfuts[e].result(), f"moe_masked expert {e}: all {ms[e]}x{w.N} elements")
