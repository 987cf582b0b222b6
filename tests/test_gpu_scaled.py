"""GPU parity of the per-tensor / per-token / per-channel path (quantisers bit for bit, the
epilogue-scaled GEMMs within the GEMM tolerance) against the oracle, through the C ABI.

Inputs come from seeded draws; the oracle quantises them itself, and the GPU GEMMs are fed the
oracle's codes and scales, so no oracle input comes from the CUDA path.  The full-size dense
shape is compared on sampled rows and column blocks after checking that the GPU's own codes
equal the oracle's there.
"""

import ctypes

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from moe_grouped_gemm_block_gb300.workloads import WORKLOADS, make_inputs
from oracle.scaled import (gemm_nt_scaled, grouped_contiguous_scaled, grouped_masked_scaled, quantize_per_row,
                           quantize_per_tensor)
from tests.gpu_util import assert_gemm_close, bf16_to_np, block_n, check_status, env_var, need_gpu, u8

pytestmark = pytest.mark.gpu
SENTINEL = 0x7FC1


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    need_gpu()


def _draw(shape, seed, std=1.0):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=gen) * std).to(torch.bfloat16)


def _f32(t):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(t, np.float32).reshape(-1))).cuda()


def _quant_ref(x_bf16, per_row):
    x = x_bf16.float().numpy()
    return quantize_per_row(x) if per_row else quantize_per_tensor(x)


# ------------------------------------------------------------------ quantisers

@pytest.mark.parametrize("M,K", [(1, 128), (37, 384), (256, 7168), (3, 17024), (130, 16384)])
def test_per_row_quantiser_bit_exact(M, K):
    x = _draw((M, K), seed=M + K, std=3.0)
    x[:, 5] *= 40
    if M > 2:
        x[1] = 0  # a zero row: s = 0, codes 0
        x[2] *= 1e-35  # subnormal scale
    q_ref, s_ref = quantize_per_row(x.float().numpy())
    q, s = g.quantize_per_row(x.cuda())
    torch.cuda.synchronize()
    check_status()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


def test_per_row_strided():
    M, K = 50, 640
    x = _draw((M, K + 64), seed=5)
    q = torch.full((M, K + 32), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.empty(M, dtype=torch.float32, device="cuda")
    g.fp8_quantize_per_row(x.cuda()[:, :K], q[:, :K], s)
    torch.cuda.synchronize()
    q_ref, s_ref = quantize_per_row(x[:, :K].float().numpy())
    assert np.array_equal(q[:, :K].cpu().numpy(), q_ref) and torch.all(q[:, K:] == 0xAB)
    assert np.array_equal(s.cpu().numpy(), s_ref)


@pytest.mark.parametrize("shape", [(1, 128), (300, 1024), (4, 96, 512), (2048, 7168)])
def test_per_tensor_quantiser_bit_exact(shape):
    x = _draw(shape, seed=sum(shape), std=0.7)
    q, s = g.quantize_per_tensor(x.cuda())
    torch.cuda.synchronize()
    check_status()
    xs = x.float().numpy().reshape(-1, *shape[-2:])
    for e in range(xs.shape[0]):
        q_ref, s_ref = quantize_per_tensor(xs[e])
        assert np.array_equal(q.cpu().numpy().reshape(xs.shape)[e], q_ref), e
        assert s.cpu().numpy()[e].view(np.uint32) == s_ref[0].view(np.uint32), e


@pytest.mark.parametrize("E,M,K", [(1, 37, 384), (3, 37, 384), (2, 130, 1024)])
def test_per_tensor_strided_c_abi(E, M, K):
    # row strides past K on both sides (through the C ABI; the binding takes contiguous tensors):
    # the codes land in the first K bytes of each row, the rest of each row is left alone
    ldx, ldq = K + 72, K + 48
    x_full = _draw((E * M, ldx), seed=E * M + K, std=1.3)
    x_full[:, K:] = 1e30  # outside the rows' K values: must not reach any amax
    q_full = torch.full((E * M, ldq), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.empty(E, dtype=torch.float32, device="cuda")
    xd = x_full.cuda()
    rc = g.lib().fp8_quantize_per_tensor(ctypes.c_void_p(xd.data_ptr()), E, M, K, ldx, ctypes.c_void_p(q_full.data_ptr()),
                                         ldq, ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    check_status()
    xs = x_full[:, :K].float().numpy().reshape(E, M, K)
    q = q_full.cpu().numpy()
    for e in range(E):
        q_ref, s_ref = quantize_per_tensor(xs[e])
        assert np.array_equal(q[e * M:(e + 1) * M, :K], q_ref), e
        assert s.cpu().numpy()[e].view(np.uint32) == s_ref[0].view(np.uint32), e
    assert np.all(q[:, K:] == 0xAB)


def test_per_tensor_zero_and_empty():
    x = torch.zeros((3, 64, 256), dtype=torch.bfloat16, device="cuda")
    x[1, 7, 9] = -2.5
    q, s = g.quantize_per_tensor(x)
    torch.cuda.synchronize()
    assert s[0].item() == 0 and s[2].item() == 0 and not q[0].any() and not q[2].any()
    assert s[1].item() == np.float32(2.5) / np.float32(448)
    s2 = torch.full((2,), 5.0, device="cuda")
    g.fp8_quantize_per_tensor(torch.empty((2, 0, 128), dtype=torch.bfloat16, device="cuda"),
                              torch.empty((2, 0, 128), dtype=torch.uint8, device="cuda"), s2)
    torch.cuda.synchronize()
    assert torch.all(s2 == 0)


def test_every_amax_significand_both_quantisers():
    # the direct product is taken or not by amax's bf16 significand: cover all 128, each with
    # a spread of values below it (per row), and the per-tensor recovery of amax from s
    K = 256
    sig = np.arange(128, dtype=np.uint32)
    amax_bits = ((127 + 3) << 23 | sig << 16).astype(np.uint32)  # 8 .. 16
    amax = amax_bits.view(np.float32)
    x = _draw((128, K), seed=77).float().numpy() * amax[:, None] / 4
    x = np.clip(x, -amax[:, None], amax[:, None])
    x[:, 0] = amax
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(xb.float().numpy()[:, 0], amax)
    q, s = g.quantize_per_row(xb.cuda())
    torch.cuda.synchronize()
    q_ref, s_ref = quantize_per_row(xb.float().numpy())
    assert np.array_equal(q.cpu().numpy(), q_ref) and np.array_equal(s.cpu().numpy(), s_ref)
    for r in range(0, 128, 9):  # one row per tensor: per-tensor amax = that row's
        qt, st = g.quantize_per_tensor(xb[r:r + 1].cuda())
        torch.cuda.synchronize()
        qt_ref, st_ref = quantize_per_tensor(xb[r:r + 1].float().numpy())
        assert np.array_equal(qt.cpu().numpy(), qt_ref) and st.item() == st_ref[0], r


# ------------------------------------------------------------------ GEMM

def _problem(M, N, K, seed, per_row, per_col):
    x = _draw((M, K), seed, 2.0)
    if K >= 256:
        x[:, 3] *= 50
    qa, sa = _quant_ref(x, per_row)
    qb, sb = _quant_ref(_draw((N, K), seed + 1, 1 / np.sqrt(K)), per_col)
    return qa, sa, qb, sb


def _dense(qa, sa, qb, sb, bn=None):
    D = torch.empty((qa.shape[0], qb.shape[0]), dtype=torch.bfloat16, device="cuda")
    with block_n(bn):
        g.fp8_gemm_nt_scaled(u8(qa), _f32(sa), u8(qb), _f32(sb), D)
    torch.cuda.synchronize()
    check_status()
    return D


MODES = [(True, True), (False, False), (True, False), (False, True)]


@pytest.mark.parametrize("per_row,per_col", MODES)
@pytest.mark.parametrize("M,N,K,bn", [
    (128, 256, 512, None), (1, 16, 128, None), (200, 208, 384, 256), (200, 208, 384, 128),
    (300, 512, 1024, 256), (129, 272, 256, 128), (64, 1792, 7168, None), (513, 384, 256, None),
    (17, 128, 1152, 64),  # a forced 64 becomes 128 (no 64-wide tiles in this variant)
])
def test_dense_scaled_small_shapes(M, N, K, bn, per_row, per_col):
    qa, sa, qb, sb = _problem(M, N, K, M * 5 + N + K, per_row, per_col)
    D = _dense(qa, sa, qb, sb, bn)
    assert g.fp8g_last_config()["block_n"] in (128, 256)
    assert_gemm_close(bf16_to_np(D), gemm_nt_scaled(qa, sa, qb, sb), f"{M}x{N}x{K} bn={bn} {per_row}{per_col}")


@pytest.mark.parametrize("streamk", ["0", "1"])
def test_dense_scaled_stream_k_tail(streamk):
    # 10 x 2 tiles of 128 x 256 with 40 K blocks on every SM count: the tail is split when on
    M, N, K = 1280, 512, 5120
    qa, sa, qb, sb = _problem(M, N, K, 21, True, True)
    with env_var("FP8G_STREAMK", streamk):
        D = _dense(qa, sa, qb, sb, 256)
    assert_gemm_close(bf16_to_np(D), gemm_nt_scaled(qa, sa, qb, sb), f"stream-K={streamk}")


def test_dense_scaled_strided_operands():
    M, N, K = 150, 160, 384
    qa, sa, qb, sb = _problem(M, N, K, 3, True, True)
    A = torch.zeros((M, K + 64), dtype=torch.uint8, device="cuda")
    A[:, :K] = u8(qa)
    B = torch.zeros((N, K + 128), dtype=torch.uint8, device="cuda")
    B[:, :K] = u8(qb)
    D = torch.full((M, N + 24), 7.0, dtype=torch.bfloat16, device="cuda")
    g.fp8_gemm_nt_scaled(A[:, :K], _f32(sa), B[:, :K], _f32(sb), D[:, :N])
    torch.cuda.synchronize()
    check_status()
    assert_gemm_close(bf16_to_np(D[:, :N]), gemm_nt_scaled(qa, sa, qb, sb), "strided")
    assert torch.all(D[:, N:] == 7.0)


def test_per_tensor_equals_power_of_two_rescaled_per_row():
    # per-row scales that are all the same power-of-two multiple of the per-tensor scale
    # give the per-tensor result times that power, bit for bit
    qa, sa, qb, sb = _problem(256, 512, 1024, 9, False, False)
    D1 = _dense(qa, sa, qb, sb)
    sa_rows = np.full(256, sa[0] * np.float32(2.0 ** -6), np.float32)
    D2 = _dense(qa, sa_rows, qb, sb)
    assert torch.equal(D1.float() * 2.0 ** -6, D2.float())


def _routed(T, E, K, seed):
    gen = torch.Generator().manual_seed(seed)
    counts = torch.randint(0, T, (E,), generator=gen).tolist()
    counts[1] = 0  # an empty expert
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + (c + 127) // 128 * 128)
    M_total = offs[-1] + 128  # one more block in no group
    x = _draw((M_total, K), seed + 1, 1.5)
    for e, c in enumerate(counts):  # zero padding rows, as a router would leave them
        x[offs[e] + c:offs[e + 1]] = 0
    return x, np.array(offs, np.int32), M_total


@pytest.mark.parametrize("per_row,per_col", MODES)
def test_grouped_contiguous_scaled(per_row, per_col):
    E, N, K = 4, 384, 512
    x, offs, M_total = _routed(300, E, K, 31)
    qa, sa = _quant_ref(x, per_row)
    w = _draw((E, N, K), 33, 1 / np.sqrt(K))
    if per_col:
        qw, sw = quantize_per_row(w.reshape(E * N, K).float().numpy())
        qb, sb = qw.reshape(E, N, K), sw.reshape(E, N)
    else:
        parts = [quantize_per_tensor(w[e].float().numpy()) for e in range(E)]
        qb, sb = np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts])
    D = torch.full((M_total, N), 0, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    g.fp8_grouped_gemm_contiguous_scaled(u8(qa), _f32(sa), u8(qb), _f32(sb), D,
                                         torch.from_numpy(offs).cuda())
    torch.cuda.synchronize()
    check_status()
    init = np.full((M_total, N), SENTINEL, np.uint16)
    ref = grouped_contiguous_scaled(qa, sa, qb, sb, offs, init)
    got = D.view(torch.int16).cpu().numpy().view(np.uint16)
    rows = np.concatenate([np.arange(offs[e], offs[e + 1]) for e in range(E)])
    assert np.all(got[offs[-1]:] == SENTINEL)
    assert_gemm_close(bf16_to_np(D)[rows], ref[rows], f"contiguous {per_row}{per_col}")


@pytest.mark.parametrize("per_row,per_col", MODES)
def test_grouped_masked_scaled(per_row, per_col):
    E, cap, N, K = 5, 256, 256, 384
    x = _draw((E * cap, K), 41, 1.0)
    qa, sa = _quant_ref(x, per_row)
    w = _draw((E * N, K), 43, 1 / np.sqrt(K))
    if per_col:
        qw, sw = quantize_per_row(w.float().numpy())
        sb = sw.reshape(E, N)
    else:
        parts = [quantize_per_tensor(w[e * N:(e + 1) * N].float().numpy()) for e in range(E)]
        qw, sb = np.concatenate([p[0] for p in parts]), np.stack([p[1] for p in parts])
    masked = np.array([0, 1, 130, 256, 77], np.int32)
    D = torch.empty((E, cap, N), dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    g.fp8_grouped_gemm_masked_scaled(u8(qa.reshape(E, cap, K)), _f32(sa), u8(qw.reshape(E, N, K)), _f32(sb), D,
                                     torch.from_numpy(masked).cuda())
    torch.cuda.synchronize()
    check_status()
    init = np.full((E, cap, N), SENTINEL, np.uint16)
    ref = grouped_masked_scaled(qa.reshape(E, cap, K), sa, qw.reshape(E, N, K), sb, masked, init)
    got_bits = D.view(torch.int16).cpu().numpy().view(np.uint16)
    got = bf16_to_np(D)
    for e in range(E):
        m = masked[e]
        assert np.all(got_bits[e, m:] == SENTINEL), e
        if m:
            assert_gemm_close(got[e, :m], ref[e, :m], f"masked e={e} {per_row}{per_col}")


def test_full_size_dense_sampled():
    # 4096 x 8192 x 8192 with per-token / per-channel scales quantised on the GPU; the GPU
    # codes of sampled rows and columns must equal the oracle's, then D is compared there
    w = WORKLOADS["large_4096x8192"]
    inp = make_inputs(w, "cuda")
    A, B = inp["A"], inp["B"]
    qa, sa = g.quantize_per_row(A)
    qb, sb = g.quantize_per_row(B)
    D = g.gemm_nt_scaled(qa, sa, qb, sb)
    torch.cuda.synchronize()
    check_status()
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(A.shape[0], 24, replace=False))
    cols = np.sort(rng.choice(B.shape[0], 96, replace=False))
    qa_ref, sa_ref = quantize_per_row(A[rows].float().cpu().numpy())
    qb_ref, sb_ref = quantize_per_row(B[cols].float().cpu().numpy())
    assert np.array_equal(qa[rows].cpu().numpy(), qa_ref) and np.array_equal(sa[rows].cpu().numpy(), sa_ref)
    assert np.array_equal(qb[cols].cpu().numpy(), qb_ref) and np.array_equal(sb[cols].cpu().numpy(), sb_ref)
    ref = gemm_nt_scaled(qa_ref, sa_ref, qb_ref, sb_ref)
    got = bf16_to_np(D)[rows][:, cols]
    assert_gemm_close(got, ref, "4096x8192x8192 per-channel")


def test_scaled_rejects_bad_mode_flags():
    A = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones(128, dtype=torch.float32, device="cuda")
    D = torch.empty((128, 128), dtype=torch.bfloat16, device="cuda")
    lib = g.lib()
    st = lib.fp8_gemm_nt_scaled(A.data_ptr(), 128, s.data_ptr(), 2, A.data_ptr(), 128, s.data_ptr(), 1,
                                D.data_ptr(), 128, 128, 128, 128, torch.cuda.current_stream().cuda_stream)
    assert st == 1
    st = lib.fp8_gemm_nt_scaled(A.data_ptr(), 128, s.data_ptr(), 1, A.data_ptr(), 128, s.data_ptr() + 4, 1,
                                D.data_ptr(), 128, 128, 128, 128, torch.cuda.current_stream().cuda_stream)
    assert st == 2  # per-column sB must be 16-byte aligned
