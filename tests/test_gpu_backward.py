"""GPU parity of the backward path (e5m2 gradient quantisation bit for bit; the data-gradient GEMM
and the K-grouped weight-gradient GEMM within the GEMM tolerance) against the oracle, through the
C ABI.  The GPU GEMMs are fed the oracle's codes and scales."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from oracle import quantize_128x128, quantize_1x128
from oracle.backward import gemm_nt_dgrad, quantize_1x128_e5m2, wgrad_k_grouped
from tests.gpu_util import (assert_gemm_close, bf16_to_np, block_n, check_status, env_var, need_gpu,
                            sa_from_device, sa_to_device, u8)

pytestmark = pytest.mark.gpu
SENTINEL = 0x7FC1


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    need_gpu()


def _draw(shape, seed, std=1.0):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=gen) * std).to(torch.bfloat16)


@pytest.mark.parametrize("M,K", [(1, 128), (37, 384), (256, 7168), (130, 1024)])
def test_e5m2_quantiser_bit_exact(M, K):
    x = _draw((M, K), M + K, 1e-3)
    x[:, 7] *= 300
    if M > 2:
        x[1] = 0
        x[2] *= 1e-30
    q_ref, s_ref = quantize_1x128_e5m2(x.float().numpy())
    q, sA = g.quantize_1x128_e5m2(x.cuda())
    torch.cuda.synchronize()
    check_status()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sa_from_device(sA, M).view(np.uint32), s_ref.view(np.uint32))


def test_e5m2_every_amax_significand():
    sig = np.arange(128, dtype=np.uint32)
    amax = (((127 - 10) << 23) | (sig << 16)).astype(np.uint32).view(np.float32)
    x = _draw((128, 256), 5).float().numpy() * amax[:, None] / 3
    x = np.clip(x, -amax[:, None], amax[:, None])
    x[:, 0] = amax
    x[:, 130] = -amax
    xb = torch.from_numpy(x).to(torch.bfloat16)
    q_ref, s_ref = quantize_1x128_e5m2(xb.float().numpy())
    q, sA = g.quantize_1x128_e5m2(xb.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref) and np.array_equal(sa_from_device(sA, 128), s_ref)


def _dgrad_problem(M, N, K, seed):
    dy = _draw((M, K), seed, 1e-3)
    if K >= 256:
        dy[:, 5] *= 40
    qa, sa = quantize_1x128_e5m2(dy.float().numpy())
    qb, sb = quantize_128x128(_draw((N, K), seed + 1, 1 / np.sqrt(K)).float().numpy())
    return qa, sa, qb, sb


@pytest.mark.parametrize("M,N,K,bn", [
    (128, 256, 512, None), (200, 208, 384, 256), (200, 208, 384, 128), (129, 272, 256, 64),
    (64, 1792, 2048, None),  # the small-M variant (lone issuers)
    (17, 128, 1152, 64),
    (513, 384, 256, None),
])
def test_dgrad_gemm(M, N, K, bn):
    qa, sa, qb, sb = _dgrad_problem(M, N, K, M + 3 * N + K)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with block_n(bn):
        g.fp8_gemm_nt_dgrad(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D)
    torch.cuda.synchronize()
    check_status()
    assert_gemm_close(bf16_to_np(D), gemm_nt_dgrad(qa, sa, qb, sb), f"dgrad {M}x{N}x{K} bn={bn}")


@pytest.mark.parametrize("M,N,K", [(64, 1792, 2048), (40, 1792, 7168)])
def test_dgrad_swapped_decode_tiles(M, N, K):
    # FP8G_SWAP_AB=1: the e5m2 gradient is the MMA's B operand (its format field moves with it);
    # (40, 1792, 7168) splits its K blocks over the SMs
    qa, sa, qb, sb = _dgrad_problem(M, N, K, 2 * M + N + K)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with env_var("FP8G_SWAP_AB", "1"):
        g.fp8_gemm_nt_dgrad(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D)
        torch.cuda.synchronize()
        assert g.fp8g_last_config()["swap_ab"]
    check_status()
    assert_gemm_close(bf16_to_np(D), gemm_nt_dgrad(qa, sa, qb, sb), f"dgrad swapped {M}x{N}x{K}")


def test_dgrad_stream_k_tail():
    # 10 x 2 tiles of 128 x 256 with 40 K blocks: the tail is split over all SMs
    qa, sa, qb, sb = _dgrad_problem(1280, 512, 5120, 9)
    D = torch.empty((1280, 512), dtype=torch.bfloat16, device="cuda")
    with env_var("FP8G_STREAMK", "1"), block_n(256):
        g.fp8_gemm_nt_dgrad(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D)
    torch.cuda.synchronize()
    check_status()
    assert_gemm_close(bf16_to_np(D), gemm_nt_dgrad(qa, sa, qb, sb), "dgrad stream-K")


def _wgrad_problem(M, N, offs, T, seed):
    dyT = _draw((M, T), seed, 1e-3)
    xT = _draw((N, T), seed + 1, 1.0)
    xT[3] *= 30  # an outlier channel
    qa, sa = quantize_1x128_e5m2(dyT.float().numpy())
    qb, sb = quantize_1x128(xT.float().numpy())
    return qa, sa, qb, sb


def _wgrad_gpu(qa, sa, qb, sb, offs, E, bn=None):
    M, T = qa.shape
    N = qb.shape[0]
    D = torch.empty((E, M, N), dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    with block_n(bn):
        g.fp8_grouped_gemm_wgrad(u8(qa), sa_to_device(sa), u8(qb), sa_to_device(sb), D,
                                 torch.from_numpy(np.asarray(offs, np.int32)).cuda())
    torch.cuda.synchronize()
    return D


@pytest.mark.parametrize("M,N,offs,T,bn", [
    (256, 512, [0, 384, 384, 1024], 1024, None),   # an empty expert
    (208, 272, [0, 128, 512, 640], 768, 256),      # ragged M and N; tokens 640.. in no expert
    (208, 272, [0, 128, 512, 640], 768, 128),
    (128, 256, [0, 2048], 2048, None),             # one expert, 16 K blocks
    (48, 64, [0, 0, 256, 256, 256], 256, None),    # most experts empty, M < 128
])
def test_wgrad_k_grouped(M, N, offs, T, bn):
    qa, sa, qb, sb = _wgrad_problem(M, N, offs, T, M + N + T)
    E = len(offs) - 1
    D = _wgrad_gpu(qa, sa, qb, sb, offs, E, bn)
    check_status()
    ref = wgrad_k_grouped(qa, sa, qb, sb, offs)
    got = bf16_to_np(D)
    for e in range(E):
        if offs[e + 1] == offs[e]:
            assert not np.any(got[e]), f"expert {e} without tokens must be zero"
        else:
            assert_gemm_close(got[e], ref[e], f"wgrad e={e} {M}x{N} T={T} bn={bn}")


def test_wgrad_bad_offsets_write_nothing():
    qa, sa, qb, sb = _wgrad_problem(128, 128, [0, 256], 256, 3)
    D = _wgrad_gpu(qa, sa, qb, sb, [0, 200], 1)  # not a multiple of 128
    assert g.fp8g_get_status() == 6  # FP8G_ERR_DEVICE_ASSERT
    assert torch.all(D.view(torch.int16) == SENTINEL)
    D = _wgrad_gpu(qa, sa, qb, sb, [0, 384], 1)  # past T
    assert g.fp8g_get_status() == 6
    assert torch.all(D.view(torch.int16) == SENTINEL)


def test_grouped_contiguous_dgrad():
    # the data gradient of a grouped layer: expert e's rows of dY times expert e's W^T
    E, N, K = 3, 256, 384
    off = np.array([0, 256, 256, 512], np.int32)
    M_total = 640  # rows 512.. in no group
    dy = _draw((M_total, K), 31, 1e-3)
    qa, sa = quantize_1x128_e5m2(dy.float().numpy())
    w = _draw((E, N, K), 32, 1 / np.sqrt(K)).float().numpy()
    qbs, sbs = zip(*(quantize_128x128(w[e]) for e in range(E)))
    qb, sb = np.stack(qbs), np.stack(sbs)
    D = torch.empty((M_total, N), dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    g.fp8_grouped_gemm_contiguous_dgrad(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D,
                                        torch.from_numpy(off).cuda())
    torch.cuda.synchronize()
    check_status()
    got = bf16_to_np(D)
    for e in (0, 2):
        r0, r1 = off[e], off[e + 1]
        assert_gemm_close(got[r0:r1], gemm_nt_dgrad(qa[r0:r1], sa[r0:r1], qb[e], sb[e]), f"grouped dgrad e={e}")
    assert torch.all(D.view(torch.int16)[512:] == SENTINEL)
