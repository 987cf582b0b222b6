"""fp8_quantize_gemm_nt: quantise the bf16 activations and multiply in one call.  Decode shapes
(M <= 64) run as one launch with a grid barrier between the quantisation and the GEMM; the codes,
scales and the product must equal those of the two separate calls bit for bit (the separate calls
are compared with the oracle in test_gpu_quantize.py and test_gpu_gemm.py), on repeated calls, on
another stream and replayed from a CUDA graph."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from gpu_util import block_n, check_status, need_gpu, sa_from_device
from oracle import quantize_1x128

pytestmark = pytest.mark.gpu


def _x(M, K, seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    x = torch.randn((M, K), generator=gen, device="cuda")
    x[:, 3::97] *= 50.0  # outlier channels: block scales spread over several binades
    return x.to(torch.bfloat16)


def _weights(N, K, seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed + 1)
    w = (torch.randn((N, K), generator=gen, device="cuda") / K ** 0.5).to(torch.bfloat16)
    return g.quantize_128x128(w)


def _buffers(M, K, N):
    q = torch.full((M, K), 0x5A, dtype=torch.uint8, device="cuda")
    sA = torch.full((K // 128, (M + 3) // 4 * 4), -1.0, dtype=torch.float32, device="cuda")
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    return q, sA, D


def _separate(x, qb, sb):
    M, K = x.shape
    q, sA, D = _buffers(M, K, qb.shape[0])
    g.fp8_quantize_1x128(x, q, sA)
    g.fp8_gemm_nt(q, sA, qb, sb, D)
    return q, sA, D


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("M,N,K", [
    (1, 256, 512), (16, 1024, 1024), (17, 384, 1152), (40, 1792, 7168), (64, 7168, 7168),
    (64, 2048, 256),     # fewer stages than the operand ring holds
    (64, 4096, 384),     # an odd number of K blocks (a half-full last stage)
    (33, 16384, 1024),   # 64-wide tiles forced: more tiles than SMs, CTAs take several tiles
])
def test_fused_equals_quantise_then_multiply(M, N, K):
    need_gpu()
    x = _x(M, K, seed=M * 7 + N + K)
    qb, sb = _weights(N, K, seed=N + K)
    with block_n(64 if N > 64 * 152 else None):
        q0, s0, D0 = _separate(x, qb, sb)
        q, sA, D = _buffers(M, K, N)
        g.fp8_quantize_gemm_nt(x, q, sA, qb, sb, D)
        cfg = g.fp8g_last_config()
    torch.cuda.synchronize()
    check_status()
    assert cfg["fused"], cfg
    assert _same(q, q0), "codes"
    assert _same(sA[:, :M], s0[:, :M]), "scales"
    assert _same(D, D0), "product"


def test_fused_codes_match_the_oracle():
    need_gpu()
    M, N, K = 17, 384, 1152
    x = _x(M, K, seed=11)
    qb, sb = _weights(N, K, seed=12)
    q, sA, D = _buffers(M, K, N)
    g.fp8_quantize_gemm_nt(x, q, sA, qb, sb, D)
    torch.cuda.synchronize()
    check_status()
    q_ref, s_ref = quantize_1x128(x.float().cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sa_from_device(sA, M).view(np.uint32), s_ref.astype(np.float32).view(np.uint32))


def test_fused_repeated_calls_reuse_the_barrier():
    # the grid barrier resets itself: back-to-back calls on one stream, each with new activations
    need_gpu()
    M, N, K = 64, 7168, 2048
    qb, sb = _weights(N, K, seed=3)
    outs = []
    for i in range(6):
        x = _x(M, K, seed=100 + i)
        q, sA, D = _buffers(M, K, N)
        g.fp8_quantize_gemm_nt(x, q, sA, qb, sb, D)
        assert g.fp8g_last_config()["fused"]
        outs.append((x, q, sA, D))
    torch.cuda.synchronize()
    check_status()
    for x, q, sA, D in outs:
        q0, s0, D0 = _separate(x, qb, sb)
        assert _same(q, q0) and _same(sA[:, :M], s0[:, :M]) and _same(D, D0)


def test_fused_on_another_stream():
    need_gpu()
    M, N, K = 40, 3072, 1024
    x = _x(M, K, seed=21)
    qb, sb = _weights(N, K, seed=22)
    q0, s0, D0 = _separate(x, qb, sb)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        q, sA, D = _buffers(M, K, N)
        g.fp8_quantize_gemm_nt(x, q, sA, qb, sb, D)
        assert g.fp8g_last_config()["fused"]
    torch.cuda.synchronize()
    assert g.fp8g_get_status(side) == 0
    assert _same(q, q0) and _same(D, D0)


def test_fused_replayed_from_a_graph():
    need_gpu()
    M, N, K = 64, 2048, 1024
    qb, sb = _weights(N, K, seed=31)
    x = _x(M, K, seed=32)
    q, sA, D = _buffers(M, K, N)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.fp8_quantize_gemm_nt(x, q, sA, qb, sb, D)  # eager first: makes the stream's workspace
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.fp8_quantize_gemm_nt(x, q, sA, qb, sb, D)
        fused = g.fp8g_last_config()["fused"]
    assert fused
    for i in range(3):
        x.copy_(_x(M, K, seed=40 + i))
        graph.replay()
        torch.cuda.synchronize()
        assert g.fp8g_get_status(s) == 0
        q0, s0, D0 = _separate(x, qb, sb)
        assert _same(q, q0) and _same(sA[:, :M], s0[:, :M]) and _same(D, D0), f"replay {i}"


@pytest.mark.parametrize("M,N,K", [(65, 512, 1024), (300, 1024, 2048)])
def test_larger_m_quantises_then_multiplies(M, N, K):
    need_gpu()
    x = _x(M, K, seed=M + N)
    qb, sb = _weights(N, K, seed=K)
    q0, s0, D0 = _separate(x, qb, sb)
    q, sA, D = _buffers(M, K, N)
    g.fp8_quantize_gemm_nt(x, q, sA, qb, sb, D)
    assert not g.fp8g_last_config()["fused"]
    torch.cuda.synchronize()
    check_status()
    assert _same(q, q0) and _same(sA[:, :M], s0[:, :M]) and _same(D, D0)
