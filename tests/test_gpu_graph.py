"""The hot path inside a CUDA graph: quantisation + GEMM captured on a stream (after one eager call on
that stream, which gives it its stream-K workspace) and replayed, with the same bits as eager calls.
Covers dense GEMMs with and without the stream-K tail (whose flags are cleared by a memset and whose
launch is cooperative), the contiguous and the masked grouped forms."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from tests.gpu_util import check_status, need_gpu

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, E=1, seed=0):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    x = (torch.randn((M, K), generator=gen, device="cuda") * 2).to(torch.bfloat16)
    w = (torch.randn((E, N, K), generator=gen, device="cuda") / np.sqrt(K)).to(torch.bfloat16)
    qw, sw = g.quantize_128x128(w if E > 1 else w[0])
    return x, qw, sw


def _run_eager_then_graph(step, replays=3):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eager = step().clone()
    torch.cuda.synchronize()
    check_status()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        out = step()
    outs = []
    for _ in range(replays):
        out.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        outs.append(out.clone())
    check_status()
    for o in outs:
        assert torch.equal(o.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(512, 1024, 1024), (640, 768, 4096)])  # whole tiles; a split tail
def test_dense_in_a_graph(M, N, K):
    need_gpu()
    x, qw, sw = _inputs(M, N, K)
    qa = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def step():
        g.fp8_quantize_1x128(x, qa, sa)
        g.fp8_gemm_nt(qa, sa, qw, sw, D)
        return D

    _run_eager_then_graph(step)


def test_contiguous_in_a_graph():
    need_gpu()
    E, N, K = 4, 512, 2048
    offs = torch.tensor([0, 256, 256, 640, 768], dtype=torch.int32, device="cuda")
    x, qw, sw = _inputs(768, N, K, E, seed=1)
    qa = torch.empty((768, K), dtype=torch.uint8, device="cuda")
    sa = torch.empty((K // 128, 768), dtype=torch.float32, device="cuda")
    D = torch.empty((768, N), dtype=torch.bfloat16, device="cuda")

    def step():
        g.fp8_quantize_1x128(x, qa, sa)
        g.fp8_grouped_gemm_contiguous(qa, sa, qw, sw, D, offs)
        return D

    _run_eager_then_graph(step)


def test_masked_in_a_graph():
    need_gpu()
    E, cap, N, K = 4, 256, 512, 2048
    counts = torch.tensor([256, 0, 130, 5], dtype=torch.int32, device="cuda")
    x, qw, sw = _inputs(E * cap, N, K, E, seed=2)
    qa = torch.zeros((E, cap, K), dtype=torch.uint8, device="cuda")
    sa = torch.zeros((K // 128, E * cap), dtype=torch.float32, device="cuda")
    D = torch.zeros((E, cap, N), dtype=torch.bfloat16, device="cuda")

    def step():
        g.fp8_quantize_1x128_masked(x.view(E, cap, K), qa, sa, counts)
        g.fp8_grouped_gemm_masked(qa, sa, qw, sw, D, counts)
        return D

    valid = (torch.arange(cap, device="cuda")[None, :] < counts[:, None])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eager = step().clone()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        out = step()
    for _ in range(3):
        out.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out[valid].view(torch.int16), eager[valid].view(torch.int16))  # rows past the
        assert not out[~valid].view(torch.int16).any()  # count are never written (they stay 0 here)
    check_status()
