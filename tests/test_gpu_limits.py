"""GPU parity at the limits of the grouped calls: the largest expert count (2048, the size of the
group table the kernels keep in shared memory), the smallest N (16) and K (one 128-wide block),
experts with no rows, one row, or a partial m-block.  Outputs against the oracle; rows a call must
not write are checked against a sentinel."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from oracle import grouped_contiguous, grouped_masked, quantize_128x128, quantize_1x128
from oracle.backward import quantize_1x128_e5m2, wgrad_k_grouped
from oracle.scaled import grouped_masked_scaled, quantize_per_row
from tests.gpu_util import assert_gemm_close, bf16_to_np, check_status, need_gpu, sa_to_device, u8

pytestmark = pytest.mark.gpu
SENTINEL = 0x7FC1
E_MAX = 2048


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    need_gpu()


def _draw(shape, seed, std=1.0):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=gen) * std).to(torch.bfloat16).float().numpy()


def _sentinel(shape):
    return torch.empty(shape, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)


def _weights(E, N, K, seed):
    w = _draw((E * N, K), seed, 1 / np.sqrt(K)).reshape(E, N, K)
    qs, ss = zip(*(quantize_128x128(w[e]) for e in range(E)))
    return np.stack(qs), np.stack(ss)


def test_contiguous_with_the_largest_expert_count():
    E, N, K = E_MAX, 16, 128
    rng = np.random.default_rng(1)
    sizes = np.zeros(E, np.int64)
    sizes[rng.choice(E, 12, replace=False)] = 128  # 12 experts with one m-block, the rest empty
    sizes[E - 1] = 256                              # and the last expert with two
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M_total = int(off[-1]) + 128                    # one m-block in no group
    qa, sa = quantize_1x128(_draw((M_total, K), 2))
    qb, sb = _weights(E, N, K, 3)
    D = _sentinel((M_total, N))
    g.fp8_grouped_gemm_contiguous(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D,
                                  torch.from_numpy(off).cuda())
    torch.cuda.synchronize()
    check_status()
    ref = grouped_contiguous(qa, sa, qb, sb, off, np.full((M_total, N), SENTINEL, np.uint16))
    got = D.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all(got[off[-1]:] == SENTINEL)
    assert_gemm_close(bf16_to_np(D)[:off[-1]], ref[:off[-1]], "contiguous E=2048")


def test_masked_with_the_largest_expert_count():
    E, cap, N, K = E_MAX, 16, 16, 128
    rng = np.random.default_rng(4)
    masked = rng.integers(0, cap + 1, E).astype(np.int32)
    masked[:3] = [0, 1, cap]
    qa, sa = quantize_1x128(_draw((E * cap, K), 5))
    qb, sb = _weights(E, N, K, 6)
    D = _sentinel((E, cap, N))
    g.fp8_grouped_gemm_masked(u8(qa.reshape(E, cap, K)), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D,
                              torch.from_numpy(masked).cuda())
    torch.cuda.synchronize()
    check_status()
    ref = grouped_masked(qa.reshape(E, cap, K), sa.reshape(E, cap, 1), qb, sb, masked,
                         np.full((E, cap, N), SENTINEL, np.uint16))
    got_bits = D.view(torch.int16).cpu().numpy().view(np.uint16)
    valid = np.arange(cap)[None, :] < masked[:, None]
    assert np.all(got_bits[~valid] == SENTINEL)
    assert_gemm_close(bf16_to_np(D)[valid], ref[valid], "masked E=2048")


def test_masked_scaled_with_the_largest_expert_count():
    E, cap, N, K = E_MAX, 16, 32, 256
    rng = np.random.default_rng(7)
    masked = rng.integers(0, cap + 1, E).astype(np.int32)
    qa, sa = quantize_per_row(_draw((E * cap, K), 8))
    qw, sw = quantize_per_row(_draw((E * N, K), 9, 1 / np.sqrt(K)))
    D = _sentinel((E, cap, N))
    g.fp8_grouped_gemm_masked_scaled(u8(qa.reshape(E, cap, K)), torch.from_numpy(sa).cuda(),
                                     u8(qw.reshape(E, N, K)), torch.from_numpy(sw.reshape(E, N)).cuda(), D,
                                     torch.from_numpy(masked).cuda())
    torch.cuda.synchronize()
    check_status()
    ref = grouped_masked_scaled(qa.reshape(E, cap, K), sa, qw.reshape(E, N, K), sw.reshape(E, N), masked,
                                np.full((E, cap, N), SENTINEL, np.uint16))
    valid = np.arange(cap)[None, :] < masked[:, None]
    assert np.all(D.view(torch.int16).cpu().numpy().view(np.uint16)[~valid] == SENTINEL)
    assert_gemm_close(bf16_to_np(D)[valid], ref[valid], "masked scaled E=2048")


def test_wgrad_with_the_largest_expert_count():
    E, M, N, T = E_MAX, 16, 32, 512
    off = np.zeros(E + 1, np.int32)
    off[5:] = 128       # expert 4 owns tokens 0..127
    off[1000:] = 256    # expert 999 owns 128..255
    off[E] = 512        # the last expert owns 256..511
    qa, sa = quantize_1x128_e5m2(_draw((M, T), 10, 1e-3))
    qb, sb = quantize_1x128(_draw((N, T), 11))
    D = _sentinel((E, M, N))
    g.fp8_grouped_gemm_wgrad(u8(qa), sa_to_device(sa), u8(qb), sa_to_device(sb), D, torch.from_numpy(off).cuda())
    torch.cuda.synchronize()
    check_status()
    ref = wgrad_k_grouped(qa, sa, qb, sb, off)
    got = bf16_to_np(D)
    for e in (4, 999, E - 1):
        assert_gemm_close(got[e], ref[e], f"wgrad expert {e}")
    others = np.ones(E, bool)
    others[[4, 999, E - 1]] = False
    assert not np.any(got[others])  # experts without tokens: zero


@pytest.mark.parametrize("M,N", [(1, 16), (128, 16), (300, 48)])
def test_dense_minimum_n_and_single_k_block(M, N):
    K = 128
    qa, sa = quantize_1x128(_draw((M, K), M + N))
    qb, sb = quantize_128x128(_draw((N, K), M + N + 1, 1 / np.sqrt(K)))
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    g.fp8_gemm_nt(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D)
    torch.cuda.synchronize()
    check_status()
    from oracle import gemm_nt
    assert_gemm_close(bf16_to_np(D), gemm_nt(qa, sa, qb, sb), f"{M}x{N}x{K}")
