"""GPU parity of the block-scaled GEMMs (dense, contiguous-grouped, masked-grouped)
against the oracle, through the C ABI.

Small shapes are compared in full (several tiles, ragged tails, every tile width); the
full-size workloads are compared element by element in test_gpu_full_size.py.  Rows a
grouped call must not write are checked bit for bit against a sentinel.
"""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from moe_grouped_gemm_block_gb300.workloads import WORKLOADS, make_inputs, round_up
from oracle import gemm_nt, grouped_contiguous, grouped_masked, quantize_128x128, quantize_1x128
from tests.gpu_util import (assert_gemm_close, bf16_bits, bf16_to_np, block_n, check_status, env_var, need_gpu, pair,
                            sa_to_device, u8)

pytestmark = pytest.mark.gpu
SENTINEL = 0x7FC1  # a bf16 NaN pattern the GEMM never produces


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    need_gpu()


def _draw(shape, seed, std=1.0):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=gen) * std).to(torch.bfloat16).float().numpy()


def _problem(M, N, K, seed):
    x = _draw((M, K), seed, 2.0)
    if K >= 256:
        x[:, 3] *= 50  # an outlier channel
    qa, sa = quantize_1x128(x)
    qb, sb = quantize_128x128(_draw((N, K), seed + 1, 1 / np.sqrt(K)))
    return qa, sa, qb, sb


def _dense_gpu(qa, sa, qb, sb, bn=None):
    M, K = qa.shape
    N = qb.shape[0]
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with block_n(bn):
        g.fp8_gemm_nt(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D)
    torch.cuda.synchronize()
    check_status()
    return D


@pytest.mark.parametrize("M,N,K,bn", [
    (128, 256, 512, None), (1, 16, 128, 64), (64, 64, 128, None), (200, 208, 384, 256),
    (200, 208, 384, 128), (200, 208, 384, 64), (300, 512, 1024, 256), (129, 272, 256, 128),
    (200, 208, 384, 192), (300, 592, 1024, 192), (513, 400, 640, 192),
    (200, 208, 384, 160), (300, 592, 1024, 160), (513, 400, 640, 160), (257, 1024, 640, 160),
    (64, 1792, 7168, 64), (257, 1024, 640, 256), (513, 384, 256, None),
    (40, 256, 384, 64), (17, 128, 1152, 64),  # small M, odd K-block counts (part-filled stages)
    # 48-wide small-M tiles: tiles straddling a 128-column weight-scale block, N tails, odd K blocks
    (1, 16, 128, 48), (40, 256, 384, 48), (17, 208, 1152, 48), (64, 1792, 7168, 48), (64, 7168, 2048, 48),
])
def test_dense_small_shapes(M, N, K, bn):
    qa, sa, qb, sb = _problem(M, N, K, seed=M * 7 + N + K)
    D = _dense_gpu(qa, sa, qb, sb, bn)
    assert_gemm_close(bf16_to_np(D), gemm_nt(qa, sa, qb, sb), f"{M}x{N}x{K} bn={bn}")


@pytest.mark.parametrize("use_pair", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (300, 272, 384), (640, 768, 1024), (129, 512, 256)])
def test_dense_256_wide_single_cta_and_pair(M, N, K, use_pair):
    qa, sa, qb, sb = _problem(M, N, K, seed=M + 3 * N + K)
    with pair(use_pair):
        D = _dense_gpu(qa, sa, qb, sb, 256)
        cfg = g.fp8g_last_config()
    paired = use_pair and M > 128  # a single m-block never runs as a pair
    want = {0: (256, 4), 1: (256, 5), 2: (128, 8)}[use_pair if paired else 0]
    assert (cfg["block_n"], cfg["stages"]) == want
    assert_gemm_close(bf16_to_np(D), gemm_nt(qa, sa, qb, sb), f"{M}x{N}x{K} pair={use_pair}")


def test_dense_strided_operands():
    M, N, K = 150, 160, 384
    qa, sa, qb, sb = _problem(M, N, K, seed=3)
    A = torch.zeros((M, K + 64), dtype=torch.uint8, device="cuda")
    A[:, :K] = u8(qa)
    B = torch.zeros((N, K + 128), dtype=torch.uint8, device="cuda")
    B[:, :K] = u8(qb)
    D = torch.full((M, N + 24), 7.0, dtype=torch.bfloat16, device="cuda")
    g.fp8_gemm_nt(A[:, :K], sa_to_device(sa, ld_sa=160), B[:, :K], torch.from_numpy(sb).cuda(), D[:, :N])
    torch.cuda.synchronize()
    check_status()
    assert_gemm_close(bf16_to_np(D[:, :N]), gemm_nt(qa, sa, qb, sb), "strided")
    assert torch.all(D[:, N:] == 7.0)


def test_dense_tiny_workload_in_full():
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, "cpu")
    qa, sa = quantize_1x128(inp["A"].float().numpy())
    qb, sb = quantize_128x128(inp["B"].float().numpy())
    D = _dense_gpu(qa, sa, qb, sb)
    assert_gemm_close(bf16_to_np(D), gemm_nt(qa, sa, qb, sb), "tiny")


def test_dense_all_scales_equal_power_of_two_case():
    # per-tensor special case: scaling A by 2^k and its scales by 2^-k must not change D
    qa, sa, qb, sb = _problem(256, 512, 512, seed=11)
    D1 = _dense_gpu(qa, sa, qb, sb)
    D2 = _dense_gpu(qa, sa * np.float32(2.0 ** 10), qb, sb * np.float32(2.0 ** -10))
    assert torch.equal(D1, D2)


# ---------------------------------------------------------------- swapped decode tiles
# FP8G_SWAP_AB=1, M <= 64: D^T = B A^T, the weight rows on the MMA's M = 128 and the
# tokens on its N = 64 (rows past M read as zero and are never stored), stored transposed.  The
# N / 128 weight slabs are fewer than the SMs, so their K blocks are split over all SMs (stream-K)
# when that saves enough; (24, 6016, 5120) splits into pieces of 13 K blocks, so pieces start on
# odd K blocks inside the two-K-block stages.

@pytest.mark.parametrize("M,N,K,split", [
    (1, 16, 128, False), (16, 208, 384, False), (17, 384, 1152, False), (33, 528, 2560, False),
    (40, 1792, 7168, True), (64, 2048, 7168, True), (24, 6016, 5120, True),
])
def test_dense_swapped_decode_tiles(M, N, K, split):
    qa, sa, qb, sb = _problem(M, N, K, seed=5 * M + N + K)
    with env_var("FP8G_SWAP_AB", "1"):
        D = _dense_gpu(qa, sa, qb, sb)
        cfg = g.fp8g_last_config()
    assert cfg["swap_ab"] and cfg["split"] == split, cfg
    assert_gemm_close(bf16_to_np(D), gemm_nt(qa, sa, qb, sb), f"swapped {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,ck,want", [
    (64, 1024, 1024, 2, 2),    # 4 tiles, 4 K blocks a rank
    (64, 1792, 2048, 4, 4),
    (40, 768, 1024, 4, 4),     # two K blocks a rank
    (128, 512, 2048, 8, 8),    # eight ranks
    (1, 256, 512, 2, 2),
    (200, 512, 1024, 2, 2),    # two m-blocks, ragged M
    (100, 2304, 4096, 4, 4),   # ragged N (9 tiles)
    (64, 1024, 1152, 4, 0),    # 9 K blocks: 4 does not divide them, no split
    (64, 768, 1536, 3, 3),     # clusters of 3, 5, 6 and 7 CTAs (12, 20, 12 and 14 K blocks)
    (130, 1280, 2560, 5, 5),
    (96, 512, 1536, 6, 6),
    (64, 256, 1792, 7, 7),
])
def test_dense_cluster_k_split(M, N, K, ck, want):
    # FP8G_CLUSTER_K: each 256-wide tile's K blocks split over a cluster of CTAs, rank 0 adding the
    # other ranks' FP32 partials before the one rounding
    qa, sa, qb, sb = _problem(M, N, K, seed=7 * M + N + K)
    with env_var("FP8G_CLUSTER_K", str(ck)):
        D = _dense_gpu(qa, sa, qb, sb)
        cfg = g.fp8g_last_config()
    check_status()
    assert cfg["cluster_k"] == want, cfg
    assert_gemm_close(bf16_to_np(D), gemm_nt(qa, sa, qb, sb), f"cluster K split {M}x{N}x{K} ck={ck}")


def test_dense_cluster_k_split_by_default_for_few_tiles_and_long_k():
    # 128 x 1024 x 16384: four 256-wide tiles and 128 K blocks -- clusters of 8 CTAs by default;
    # FP8G_CLUSTER_K=0 turns it off; both within the tolerance of the oracle
    M, N, K = 128, 1024, 16384
    qa, sa, qb, sb = _problem(M, N, K, seed=123)
    ref = gemm_nt(qa, sa, qb, sb)
    with env_var("FP8G_CLUSTER_K", None):
        D = _dense_gpu(qa, sa, qb, sb)
        assert g.fp8g_last_config()["cluster_k"] == 8
    check_status()
    assert_gemm_close(bf16_to_np(D), ref, "cluster K split by default")
    with env_var("FP8G_CLUSTER_K", "0"):
        D0 = _dense_gpu(qa, sa, qb, sb)
        assert g.fp8g_last_config()["cluster_k"] == 0
    check_status()
    assert_gemm_close(bf16_to_np(D0), ref, "cluster K split turned off")


def test_dense_swapped_tiles_switch_and_strides():
    # by default M <= 64 takes the 64-wide small-M tiles; strided operands and ld_sa > M in the
    # swapped form (FP8G_SWAP_AB=1)
    M, N, K = 20, 400, 1024
    qa, sa, qb, sb = _problem(M, N, K, seed=31)
    D0 = _dense_gpu(qa, sa, qb, sb)
    assert not g.fp8g_last_config()["swap_ab"]
    A = torch.zeros((M, K + 32), dtype=torch.uint8, device="cuda")
    A[:, :K] = u8(qa)
    B = torch.zeros((N, K + 64), dtype=torch.uint8, device="cuda")
    B[:, :K] = u8(qb)
    D = torch.full((M, N + 8), 7.0, dtype=torch.bfloat16, device="cuda")
    with env_var("FP8G_SWAP_AB", "1"):
        g.fp8_gemm_nt(A[:, :K], sa_to_device(sa, ld_sa=36), B[:, :K], torch.from_numpy(sb).cuda(), D[:, :N])
        torch.cuda.synchronize()
        assert g.fp8g_last_config()["swap_ab"]
    check_status()
    ref = gemm_nt(qa, sa, qb, sb)
    assert_gemm_close(bf16_to_np(D[:, :N]), ref, "swapped, strided")
    assert_gemm_close(bf16_to_np(D0), ref, "small-M tiles")
    assert torch.all(D[:, N:] == 7.0)


# ---------------------------------------------------------------- contiguous

def _contig_problem(sizes, N, K, seed, extra_rows=0):
    E = len(sizes)
    offs = [0]
    for s in sizes:
        offs.append(offs[-1] + round_up(s, 128))
    M_total = offs[-1] + extra_rows
    x = np.zeros((M_total, K), np.float32)
    for e, s in enumerate(sizes):
        x[offs[e]:offs[e] + s] = _draw((s, K), seed + e, 1.5)
    qa, sa = quantize_1x128(x)
    qbs, sbs = zip(*(quantize_128x128(_draw((N, K), seed + 100 + e, 1 / np.sqrt(K))) for e in range(E)))
    return qa, sa, np.stack(qbs), np.stack(sbs), np.array(offs, np.int32)


def _contig_gpu(qa, sa, qb, sb, offs, bn=None):
    M_total, K = qa.shape
    N = qb.shape[1]
    D = torch.full((M_total, N), 0, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    with block_n(bn):
        g.fp8_grouped_gemm_contiguous(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D,
                                      torch.from_numpy(offs).cuda())
    torch.cuda.synchronize()
    return D


@pytest.mark.parametrize("bn,use_pair", [(None, 1), (256, 1), (256, 0), (192, 0), (160, 0), (128, 1), (64, 1), (None, 2),
                                          (256, 2)])
def test_contiguous_small(bn, use_pair):
    qa, sa, qb, sb, offs = _contig_problem([100, 0, 300, 128, 1], N=272, K=384, seed=5, extra_rows=128)
    with pair(use_pair):
        D = _contig_gpu(qa, sa, qb, sb, offs, bn)
    check_status()
    init = np.full((qa.shape[0], qb.shape[1]), SENTINEL, np.uint16)
    ref = grouped_contiguous(qa, sa, qb, sb, offs, init)
    got = bf16_bits(D)
    last = offs[-1]
    assert np.array_equal(got[last:], ref[last:])  # rows outside every group: untouched
    assert_gemm_close(bf16_to_np(D[:last]), ref[:last], f"contiguous bn={bn}")


def test_contiguous_pages_two_experts_eight_tokens():
    qa, sa, qb, sb, offs = _contig_problem([8, 8], N=128, K=256, seed=9)
    D = _contig_gpu(qa, sa, qb, sb, offs)
    check_status()
    ref = grouped_contiguous(qa, sa, qb, sb, offs, np.zeros((256, 128), np.uint16))
    assert_gemm_close(bf16_to_np(D), ref, "2 experts x 8 tokens")
    assert not bf16_to_np(D[8:128]).any() and not bf16_to_np(D[136:]).any()  # zero padding rows


def test_contiguous_bad_offsets_sets_device_assert_and_writes_nothing():
    qa, sa, qb, sb, offs = _contig_problem([128, 128], N=128, K=128, seed=2)
    for bad in ([0, 100, 256], [0, 256, 128], [0, 128, 512]):
        D = _contig_gpu(qa, sa, qb, sb, np.array(bad, np.int32))
        assert g.fp8g_get_status() == 6
        assert np.all(bf16_bits(D) == SENTINEL)
    check_status()


# ---------------------------------------------------------------- masked

def _masked_gpu(qa, sa, qb, sb, masked, bn=None):
    E, cap, K = qa.shape
    N = qb.shape[1]
    D = torch.full((E, cap, N), 0, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    with block_n(bn):
        g.fp8_grouped_gemm_masked(u8(qa), sa_to_device(sa.reshape(E * cap, -1)), u8(qb),
                                  torch.from_numpy(sb).cuda(), D, torch.tensor(masked, dtype=torch.int32).cuda())
    torch.cuda.synchronize()
    return D


def _masked_problem(E, cap, N, K, seed):
    qa, sa = quantize_1x128(_draw((E * cap, K), seed, 1.5))
    qbs, sbs = zip(*(quantize_128x128(_draw((N, K), seed + 50 + e, 1 / np.sqrt(K))) for e in range(E)))
    return qa.reshape(E, cap, K), sa.reshape(E, cap, -1), np.stack(qbs), np.stack(sbs)


@pytest.mark.parametrize("bn,use_pair", [(None, 1), (256, 1), (256, 0), (192, 0), (160, 0), (128, 1), (64, 1), (None, 2),
                                          (256, 2)])
def test_masked_small(bn, use_pair):
    E, cap, N, K = 5, 160, 272, 384
    masked = [0, 1, 160, 37, 129]
    qa, sa, qb, sb = _masked_problem(E, cap, N, K, seed=21)
    with pair(use_pair):
        D = _masked_gpu(qa, sa, qb, sb, masked, bn)
    check_status()
    ref = grouped_masked(qa, sa, qb, sb, masked, np.full((E, cap, N), SENTINEL, np.uint16))
    got = bf16_bits(D)
    for e in range(E):
        m = masked[e]
        assert np.all(got[e, m:] == SENTINEL), f"expert {e}: rows past masked_m written"
        if m:
            assert_gemm_close(bf16_to_np(D[e, :m]), ref[e, :m], f"masked e={e} bn={bn}")


def test_masked_counts_out_of_range_are_clamped_and_flagged():
    E, cap, N, K = 2, 32, 128, 128
    qa, sa, qb, sb = _masked_problem(E, cap, N, K, seed=4)
    D = _masked_gpu(qa, sa, qb, sb, [40, -3])
    assert g.fp8g_get_status() == 6
    ref = grouped_masked(qa, sa, qb, sb, [32, 0], np.full((E, cap, N), SENTINEL, np.uint16))
    assert_gemm_close(bf16_to_np(D[0]), ref[0], "clamped")
    assert np.all(bf16_bits(D[1]) == SENTINEL)


def test_status_clear_after_many_calls_on_two_streams():
    qa, sa, qb, sb = _problem(256, 512, 512, seed=8)
    A, B, sBt = u8(qa), u8(qb), torch.from_numpy(sb).cuda()
    sAt = sa_to_device(sa)
    outs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for i in range(8):
        with torch.cuda.stream(streams[i % 2]):
            D = torch.empty((256, 512), dtype=torch.bfloat16, device="cuda")
            g.fp8_gemm_nt(A, sAt, B, sBt, D)
            outs.append(D)
    torch.cuda.synchronize()
    check_status()
    for D in outs[1:]:
        assert torch.equal(D, outs[0])


# ---------------------------------------------------------------- stream-K tail
# With FP8G_STREAMK on (the default), tiles that do not fill whole rounds of the grid have their
# K blocks split over all SMs when that saves at least 24 K blocks per CTA; CTAs holding part of a
# tile write FP32 partials that the CTA with its first K blocks adds.  These shapes split tiles
# (K = 4096: 32 K blocks, 8 per CTA), with and without a round of whole tiles before the tail.

def streamk(on):
    return env_var("FP8G_STREAMK", None if on else 0)


@pytest.mark.parametrize("on", [True, False])
@pytest.mark.parametrize("M,N,K,bn", [
    (640, 768, 4096, 256),    # 15 tiles: every tile split among 4 CTAs
    (300, 512, 4096, 128),    # 12 tiles of width 128, ragged M
    (2560, 2048, 4096, 256),  # 160 tiles: one whole round, then 8 tiles split in four
    (640, 768, 2048, 256),    # too few K blocks for a split to pay: whole tiles on every SM
])
def test_dense_stream_k_tail(M, N, K, bn, on):
    qa, sa, qb, sb = _problem(M, N, K, seed=M + N + 7 * K)
    with streamk(on):
        D = _dense_gpu(qa, sa, qb, sb, bn)
        cfg = g.fp8g_last_config()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = -(-M // 128) * -(-N // bn)
    kb = K // 128
    u = max(-(-((tiles % sms) * kb) // sms), min(8, kb))
    split = on and tiles % sms != 0 and kb - u >= 24  # the library's split rule
    assert (cfg["grid"] == sms) == (split or tiles >= sms)
    assert_gemm_close(bf16_to_np(D), gemm_nt(qa, sa, qb, sb), f"{M}x{N}x{K} bn={bn} streamk={on}")


@pytest.mark.parametrize("on", [True, False])
def test_contiguous_stream_k_tail(on):
    qa, sa, qb, sb, offs = _contig_problem([300, 0, 128, 77], N=512, K=4096, seed=31, extra_rows=128)
    with streamk(on):
        D = _contig_gpu(qa, sa, qb, sb, offs, 256)
    check_status()
    init = np.full((qa.shape[0], qb.shape[1]), SENTINEL, np.uint16)
    ref = grouped_contiguous(qa, sa, qb, sb, offs, init)
    got = bf16_bits(D)
    last = offs[-1]
    assert np.array_equal(got[last:], ref[last:])  # rows outside every group: untouched
    assert_gemm_close(bf16_to_np(D[:last]), ref[:last], f"contiguous streamk={on}")


@pytest.mark.parametrize("on", [True, False])
def test_masked_stream_k_tail(on):
    E, cap, N, K = 4, 256, 512, 4096
    masked = [256, 0, 130, 5]
    qa, sa, qb, sb = _masked_problem(E, cap, N, K, seed=41)
    with streamk(on):
        D = _masked_gpu(qa, sa, qb, sb, masked, 256)
    check_status()
    ref = grouped_masked(qa, sa, qb, sb, masked, np.full((E, cap, N), SENTINEL, np.uint16))
    got = bf16_bits(D)
    for e in range(E):
        m = masked[e]
        assert np.all(got[e, m:] == SENTINEL), f"expert {e}: rows past masked_m written"
        if m:
            assert_gemm_close(bf16_to_np(D[e, :m]), ref[e, :m], f"masked e={e} streamk={on}")


def test_stream_k_repeated_calls_and_two_streams():
    # the per-stream workspace's flags are cleared before every launch: repeated calls, and calls
    # alternating between two streams (each with its own workspace), give the same result
    qa, sa, qb, sb = _problem(640, 768, 4096, seed=5)
    ref = gemm_nt(qa, sa, qb, sb)
    A, SA, B, SB = u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    with block_n(256):
        for i in range(6):
            D = torch.empty((640, 768), dtype=torch.bfloat16, device="cuda")
            with torch.cuda.stream(s1 if i % 2 else s2):
                g.fp8_gemm_nt(A, SA, B, SB, D)
            outs.append(D)
    torch.cuda.synchronize()
    check_status()
    for D in outs:
        assert torch.equal(D, outs[0])
    assert_gemm_close(bf16_to_np(outs[0]), ref, "stream-K repeated")
