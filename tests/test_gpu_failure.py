"""Failure detection on the GPU without a fault: the bounded waits every GEMM role uses run out of
budget against an mbarrier phase and a flag that nothing completes, record FP8G_ERR_TIMEOUT and
return; the context stays usable (a GEMM afterwards is correct and reports OK)."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from oracle import gemm_nt, quantize_128x128, quantize_1x128
from tests.gpu_util import assert_gemm_close, bf16_to_np, need_gpu, sa_to_device, u8

pytestmark = pytest.mark.gpu


def test_bounded_waits_run_out_and_the_context_stays_usable():
    need_gpu()
    assert g.fp8g_get_status() == 0
    out = torch.zeros(3, dtype=torch.int32, device="cuda")
    st = g.lib().fp8g_selftest_bounded_waits(2_000_000, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert g.fp8g_get_status() == 5  # FP8G_ERR_TIMEOUT, read and cleared
    assert out.tolist() == [1, 1, 1]  # both waits gave up and raised the abort flag
    assert g.fp8g_get_status() == 0
    # the context is intact: a GEMM runs and is correct
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((200, 512)) * 2).astype(np.float32)
    w = (rng.standard_normal((256, 512)) / 22).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    w = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    qa, sa = quantize_1x128(x)
    qb, sb = quantize_128x128(w)
    D = torch.empty((200, 256), dtype=torch.bfloat16, device="cuda")
    g.fp8_gemm_nt(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D)
    assert g.fp8g_get_status() == 0
    assert_gemm_close(bf16_to_np(D), gemm_nt(qa, sa, qb, sb), "GEMM after the timeouts")
