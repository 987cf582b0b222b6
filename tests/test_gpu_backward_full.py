"""The backward GEMMs at the MoE contiguous layer's full size (8 experts, 4096 outputs, 7168 inputs,
8576 padded tokens), as the benchmark runs them: the GPU quantises a seeded synthetic gradient and the
layer's activations, its codes on sampled rows must equal the oracle's bit for bit, and then sampled
entries of dX and of one expert's dW are compared with the oracle."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from moe_grouped_gemm_block_gb300.workloads import WORKLOADS, make_inputs
from oracle import quantize_128x128, quantize_1x128
from oracle.backward import gemm_nt_dgrad, quantize_1x128_e5m2, wgrad_k_grouped
from tests.gpu_util import assert_gemm_close, bf16_to_np, check_status, need_gpu, sa_from_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    need_gpu()
    w = WORKLOADS["moe_contiguous"]
    inp = make_inputs(w, "cuda")
    A, B = inp["A"], inp["B"]  # [M_total, K] activations, [E, N, K] weights
    valid = (inp["row_token"] >= 0).cuda()
    gen = torch.Generator(device="cuda").manual_seed(77)
    dY = (torch.randn((A.shape[0], B.shape[1]), generator=gen, device="cuda") * 1e-3 * valid[:, None]).to(torch.bfloat16)
    return A, B, dY, inp["group_offsets"].cuda()


def test_full_size_grouped_dgrad(layer):
    A, B, dY, offs = layer
    E, N, K = B.shape
    qdy, sdy = g.quantize_1x128_e5m2(dY)
    WT = B.transpose(1, 2).contiguous()  # [E, K, N]
    qwt, swt = g.quantize_128x128(WT)
    dX = torch.empty((A.shape[0], K), dtype=torch.bfloat16, device="cuda")
    g.fp8_grouped_gemm_contiguous_dgrad(qdy, sdy, qwt, swt, dX, offs)
    torch.cuda.synchronize()
    check_status()
    o = offs.cpu().numpy()
    e = 5
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(np.arange(o[e], o[e + 1]), 12, replace=False))
    cols = np.r_[0:128, 4096:4224]  # two 128-column blocks of dX (two 128-row blocks of W^T)
    q_ref, s_ref = quantize_1x128_e5m2(dY[torch.from_numpy(rows).cuda()].float().cpu().numpy())
    assert np.array_equal(qdy[torch.from_numpy(rows).cuda()].cpu().numpy(), q_ref)
    assert np.array_equal(sa_from_device(sdy, dY.shape[0])[rows], s_ref)
    wt = WT[e].float().cpu().numpy()
    q0, s0 = quantize_128x128(wt[0:128])
    q1, s1 = quantize_128x128(wt[4096:4224])
    assert np.array_equal(qwt[e, 0:128].cpu().numpy(), q0) and np.array_equal(qwt[e, 4096:4224].cpu().numpy(), q1)
    # the two weight blocks as a 256-row B of their own: its 128-row blocks 0 and 1
    ref = gemm_nt_dgrad(q_ref, s_ref, np.concatenate([q0, q1]), np.concatenate([s0, s1]))
    assert_gemm_close(bf16_to_np(dX)[rows][:, cols], ref, "full-size grouped dgrad")


def test_full_size_wgrad(layer):
    A, B, dY, offs = layer
    E, N, K = B.shape
    dYT, XT = dY.t().contiguous(), A.t().contiguous()  # [N, T], [K, T]
    qa, sa = g.quantize_1x128_e5m2(dYT)
    qb, sb = g.quantize_1x128(XT)
    dW = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    g.fp8_grouped_gemm_wgrad(qa, sa, qb, sb, dW, offs)
    torch.cuda.synchronize()
    check_status()
    rng = np.random.default_rng(4)
    rows = np.sort(rng.choice(N, 10, replace=False))
    cols = np.sort(rng.choice(K, 24, replace=False))
    qa_ref, sa_ref = quantize_1x128_e5m2(dYT[torch.from_numpy(rows).cuda()].float().cpu().numpy())
    qb_ref, sb_ref = quantize_1x128(XT[torch.from_numpy(cols).cuda()].float().cpu().numpy())
    assert np.array_equal(qa[torch.from_numpy(rows).cuda()].cpu().numpy(), qa_ref)
    assert np.array_equal(qb[torch.from_numpy(cols).cuda()].cpu().numpy(), qb_ref)
    ref = wgrad_k_grouped(qa_ref, sa_ref, qb_ref, sb_ref, offs.cpu().numpy())
    got = bf16_to_np(dW)[:, rows][:, :, cols]
    for e in range(E):
        assert_gemm_close(got[e], ref[e], f"full-size wgrad expert {e}")
