"""The library baselines bench.py times compute the GEMM they stand in for.

The unfused FP8 baseline (codes and block scales dequantised to bf16 by torch elementwise ops, then the
cuBLAS BF16 GEMM) is checked against the oracle: its dequantised operands must equal code x scale rounded
to fp32 (one IEEE multiplication) and then to bf16, and its result must be close to the oracle's, within
what rounding each operand to bf16 allows.
"""

import numpy as np
import pytest
import torch

import bench
from oracle import bf16_bits_to_f32, e4m3_decode, gemm_nt, quantize_128x128, quantize_1x128
from tests.gpu_util import bf16_to_np, need_gpu, sa_to_device, u8

pytestmark = pytest.mark.gpu


def _bf16_round(x64):
    return torch.from_numpy(np.asarray(x64, np.float32)).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (77, 200, 384)])
def test_unfused_fp8_baseline(M, N, K):
    need_gpu()
    gen = torch.Generator().manual_seed(M + N + K)
    x = (torch.randn((M, K), generator=gen) * 2).to(torch.bfloat16).float().numpy()
    wt = (torch.randn((N, K), generator=gen) / np.sqrt(K)).to(torch.bfloat16).float().numpy()
    qa, sa = quantize_1x128(x)
    qb, sb = quantize_128x128(wt)
    ad = bench.dequant_block_bf16(u8(qa), sa_to_device(sa), M)
    bd = bench.dequant_weight_bf16(u8(qb).unsqueeze(0), torch.from_numpy(sb).cuda().unsqueeze(0))[0]
    torch.cuda.synchronize()
    # code x scale is exact in fp64; rounded to fp32 as the GPU multiplication rounds it, then to bf16
    want_a = _bf16_round(e4m3_decode(qa) * np.repeat(sa.astype(np.float64), 128, axis=1))
    sbe = np.repeat(np.repeat(sb.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
    want_b = _bf16_round(e4m3_decode(qb) * sbe)
    assert np.array_equal(bf16_to_np(ad), want_a) and np.array_equal(bf16_to_np(bd), want_b)
    D = bf16_to_np(torch.matmul(ad, bd.t()))
    ref = bf16_bits_to_f32(gemm_nt(qa, sa, qb, sb)).astype(np.float64)
    fro = np.linalg.norm(D - ref) / np.linalg.norm(ref)
    assert fro < 1e-2, fro  # bf16 operands: ~2^-9 relative per element
