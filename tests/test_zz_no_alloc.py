"""fp8_gemm_nt_noalloc: the dense GEMM with the library's fixed scratch buffer in place of the
per-stream stream-K workspace.  It must give exactly what fp8_gemm_nt gives, call after call,
and must not take device memory.  (Collected last; it also passes alone in a fresh process.)"""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from oracle import gemm_nt, quantize_128x128, quantize_1x128
from tests.gpu_util import assert_gemm_close, bf16_to_np, block_n, check_status, need_gpu, sa_to_device, u8

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    gen = torch.Generator().manual_seed(seed)
    x = (torch.randn((M, K), generator=gen) * 2).to(torch.bfloat16).float().numpy()
    w = (torch.randn((N, K), generator=gen) / np.sqrt(K)).to(torch.bfloat16).float().numpy()
    qa, sa = quantize_1x128(x)
    qb, sb = quantize_128x128(w)
    return qa, sa, qb, sb


# 640x768x4096: 15 tiles, every one split across several SMs (the scratch is used);
# 2560x2048x4096: a whole round of tiles, then 8 split tiles;  64x1024x512: no split at all
@pytest.mark.parametrize("M,N,K,splits", [(640, 768, 4096, True), (2560, 2048, 4096, True), (64, 1024, 512, False)])
def test_noalloc_equals_the_allocating_call_on_two_calls_in_a_row(M, N, K, splits):
    need_gpu()
    qa, sa, qb, sb = _operands(M, N, K, seed=M + N + K)
    A, SA, B, SB = u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    outs = {}
    with block_n(256 if M > 64 else None):
        for name, fn in (("alloc", g.fp8_gemm_nt), ("noalloc", g.fp8_gemm_nt_noalloc)):
            for i in range(2):
                D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
                fn(A, SA, B, SB, D)
                cfg = g.fp8g_last_config()
                # the split tail (which works in the fixed scratch) ran exactly where expected: on
                # every SM, or on fewer SMs than tiles-or-SMs without a split
                assert cfg["split"] == splits, (name, cfg)
                if splits:
                    assert cfg["grid"] == sms, (name, cfg)
                else:
                    assert cfg["grid"] < sms, (name, cfg)
                outs[(name, i)] = D
    torch.cuda.synchronize()
    check_status()
    first = outs[("alloc", 0)]
    for key, D in outs.items():
        assert torch.equal(D, first), key
    assert_gemm_close(bf16_to_np(first), gemm_nt(qa, sa, qb, sb), f"{M}x{N}x{K}")


def test_noalloc_takes_no_device_memory():
    # Device memory is measured around calls on streams this library has not used yet.  Each
    # stream is touched by a torch op first (PyTorch's own first use of a stream takes memory);
    # then the allocating entry point takes its workspace there and this one takes nothing.
    need_gpu()
    qa, sa, qb, sb = _operands(640, 768, 4096, seed=3)
    A, SA, B, SB = u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda()
    D = torch.empty((640, 768), dtype=torch.bfloat16, device="cuda")
    x = torch.ones(1024, device="cuda")

    def taken(fn):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            x.mul_(1.0)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        with torch.cuda.stream(s):
            for _ in range(3):
                fn(A, SA, B, SB, D)
        torch.cuda.synchronize()
        return free_before - torch.cuda.mem_get_info()[0]

    with block_n(256):
        g.fp8_gemm_nt_noalloc(A, SA, B, SB, D)  # the library's kernels are loaded from here on
        torch.cuda.synchronize()
        assert taken(g.fp8_gemm_nt_noalloc) == 0
        assert taken(g.fp8_gemm_nt) >= 19 * 2**20  # the per-stream workspace this call avoids
    check_status()
