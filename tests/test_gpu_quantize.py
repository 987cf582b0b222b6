"""GPU parity of the quantisation kernels against the oracle: bytes and scales bit-exact."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from moe_grouped_gemm_block_gb300.workloads import WORKLOADS, make_inputs
from oracle import quantize_128x128, quantize_1x128
from tests.gpu_util import check_status, need_gpu, sa_from_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    need_gpu()


def _bf16(shape, seed, scale=1.0):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def _np(x):
    return x.float().numpy()


def _check_1x128(x_cpu: torch.Tensor, rows=None):
    q, sA = g.quantize_1x128(x_cpu.cuda())
    torch.cuda.synchronize()
    check_status()
    M = x_cpu.shape[0]
    rows = np.arange(M) if rows is None else rows
    q_ref, s_ref = quantize_1x128(_np(x_cpu[rows]))
    assert np.array_equal(q.cpu().numpy()[rows], q_ref)
    s_gpu = sa_from_device(sA, M)[rows]
    assert np.array_equal(s_gpu.view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("M,K", [(1, 128), (3, 384), (128, 512), (200, 1024), (64, 7168)])
def test_1x128_small_shapes(M, K):
    _check_1x128(_bf16((M, K), seed=M + K, scale=3.0))


def test_1x128_edge_values():
    x = torch.zeros((8, 256))
    x[1, 0] = 448.0                    # s = 1: values map to themselves
    # midpoints between neighbouring codes (ties to even), the subnormal step, signed zero
    x[1, 1:8] = torch.tensor([1.0625, 1.1875, 0.0009765625, -0.0009765625, 2.0 ** -10, 432.0, -0.0])
    x[1, 8] = -448.0
    x[2, :128] = 1e-30                 # tiny block: s is subnormal in fp32
    x[2, 5] = -3e-30
    x[3, :] = -0.0                     # all (negative) zeros: s = 0, codes 0
    x[4, :] = torch.linspace(-5, 5, 256)
    x[5, 130] = 3.0e38                 # bf16-representable huge value
    x[6, :128] = 2.0 ** -133           # smallest bf16 subnormal
    x[7, ::7] = 1.0
    x[7, 128] = 464.0                  # rounds past 448 before saturation when s = 1
    _check_1x128(x.to(torch.bfloat16))


def test_1x128_zero_rows_and_strided_layouts():
    x = _bf16((40, 512), seed=7)
    x[5] = 0
    big = torch.zeros((40, 640), dtype=torch.bfloat16)
    big[:, :512] = x
    xs = big.cuda()[:, :512]  # ldx = 640
    q = torch.full((40, 528), 0x55, dtype=torch.uint8, device="cuda")[:, :512]  # ldq = 528
    sA = torch.full((4, 48), -1.0, device="cuda")  # ld_sa = 48 > M
    g.fp8_quantize_1x128(xs, q, sA)
    torch.cuda.synchronize()
    check_status()
    q_ref, s_ref = quantize_1x128(_np(x))
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sA[:, :40].cpu().numpy().T, s_ref)
    assert torch.all(sA[:, 40:] == -1.0)  # entries past M untouched


def test_1x128_m_zero_is_noop():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((0, 256), dtype=torch.uint8, device="cuda")
    sA = torch.empty((2, 4), device="cuda")
    g.fp8_quantize_1x128(x, q, sA)
    check_status()


@pytest.mark.parametrize("name", ["decode", "large_4096", "moe_contiguous", "moe_masked"])
def test_1x128_full_size_workloads(name):
    w = WORKLOADS[name]
    x = make_inputs(w, device="cuda")["A"]
    x = x.reshape(-1, w.K)
    q, sA = g.quantize_1x128(x)
    torch.cuda.synchronize()
    check_status()
    M = x.shape[0]
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(M, min(M, 192), replace=False), [0, M - 1]]))
    q_ref, s_ref = quantize_1x128(x[rows].float().cpu().numpy())
    assert np.array_equal(q[rows].cpu().numpy(), q_ref)
    assert np.array_equal(sa_from_device(sA, M)[rows], s_ref)


@pytest.mark.parametrize("E,N,K", [(1, 128, 128), (2, 200, 384), (3, 16, 256), (1, 7168 // 8, 512)])
def test_128x128_small_shapes(E, N, K):
    w = _bf16((E, N, K), seed=E * N + K, scale=0.05)
    q, sB = g.quantize_128x128(w.cuda())
    torch.cuda.synchronize()
    check_status()
    for e in range(E):
        q_ref, s_ref = quantize_128x128(_np(w[e]))
        assert np.array_equal(q[e].cpu().numpy(), q_ref)
        assert np.array_equal(sB[e].cpu().numpy(), s_ref)


def test_128x128_full_size_masked_weights_sampled_experts():
    w = WORKLOADS["moe_masked"]
    B = make_inputs(w, device="cuda")["B"]
    q, sB = g.quantize_128x128(B)
    torch.cuda.synchronize()
    check_status()
    for e in (0, 17, w.E - 1):
        q_ref, s_ref = quantize_128x128(B[e].float().cpu().numpy())
        assert np.array_equal(q[e].cpu().numpy(), q_ref)
        assert np.array_equal(sB[e].cpu().numpy(), s_ref)


def test_1x128_quotients_on_every_rounding_midpoint():
    # amax = 448 * 2^k makes s = 2^k, so x / s is exact: blocks full of e4m3 midpoints (ties to
    # even) and of their bf16 neighbours exercise both the multiply path and the division path.
    tab = [(1 + m / 8) * 2.0 ** (e - 7) for e in range(1, 16) for m in range(8)]
    tab = [v for v in tab if v <= 448]
    mids = [(a + b) / 2 for a, b in zip(tab[:-1], tab[1:])]
    vals = torch.tensor(mids + [2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -7 + 2.0 ** -10])
    rows = []
    for k in (-20, -3, 0, 5, 30):
        for nudge in (0, 1, -1):  # the midpoint and its bf16 neighbours
            blk = torch.zeros(128)
            v = vals.to(torch.bfloat16)
            if nudge:
                v = (v.view(torch.int16) + nudge).view(torch.bfloat16)
            v = v.float()
            blk[:v.numel()] = v
            blk[127] = 448.0
            sign = torch.where(torch.arange(128) % 2 == 0, 1.0, -1.0)
            rows.append(blk * sign * 2.0 ** k)
    x = torch.stack(rows).to(torch.bfloat16)
    _check_1x128(x)


def test_1x128_every_amax_significand_against_every_x():
    # One block per (amax significand A, chunk of x): element 0 is amax, the rest are bf16 values
    # +-X * 2^-k with |x| <= amax, so every (A, x) pair the code decision depends on is covered,
    # for marked significands (direct product) and unmarked ones (bracket) alike, at three amax
    # exponents.
    X = np.arange(128, 256, dtype=np.float64) / 128.0
    rows = []
    for scale in (1.0, 2.0 ** -30, 2.0 ** 40):
        for A in range(128, 256):
            amax = A / 128.0
            x = np.concatenate([X * 2.0 ** -k for k in range(32)])
            x = x[x <= amax]
            x = np.concatenate([x, -x])
            for i in range(0, x.size, 127):
                row = np.zeros(128)
                row[0] = amax
                chunk = x[i:i + 127]
                row[1:1 + chunk.size] = chunk
                rows.append(row * scale)
    xt = torch.from_numpy(np.stack(rows)).to(torch.bfloat16)
    assert torch.equal(xt.double(), torch.from_numpy(np.stack(rows)))  # every value is a bf16
    _check_1x128(xt)


@pytest.mark.parametrize("E,cap,K", [
    (5, 256, 512), (3, 16, 128), (32, 256, 7168),
    (40, 48, 384),     # three K blocks a row: groups of a warp leave the item loop at different passes
    (1024, 16, 256),   # many experts, one grid row each
    (1100, 16, 256),
])
def test_masked_rows_quantiser(E, cap, K):
    # only rows m < masked_m[e] are quantised (counts clamped to [0, cap]); the rest keep their bytes
    import moe_grouped_gemm_block_gb300 as g
    from oracle import quantize_1x128
    gen = torch.Generator().manual_seed(E * cap + K)
    x = (torch.randn((E, cap, K), generator=gen) * 2).to(torch.bfloat16)
    counts = torch.randint(0, cap + 1, (E,), generator=gen, dtype=torch.int32)
    counts[0] = 0
    if E > 2:
        counts[1] = cap
        counts[2] = -3  # out of contract: clamped to 0
    if E > 3:
        counts[3] = cap + 7  # clamped to cap
    q = torch.full((E, cap, K), 0xAB, dtype=torch.uint8, device="cuda")
    ld = E * cap
    sA = torch.full((K // 128, ld), -1.0, dtype=torch.float32, device="cuda")
    g.fp8_quantize_1x128_masked(x.cuda(), q, sA, counts.cuda())
    torch.cuda.synchronize()
    qh, sh = q.cpu().numpy(), sA.cpu().numpy()
    for e in range(E):
        m = min(max(int(counts[e]), 0), cap)
        if m:
            q_ref, s_ref = quantize_1x128(x[e, :m].float().numpy())
            assert np.array_equal(qh[e, :m], q_ref), e
            assert np.array_equal(sh[:, e * cap:e * cap + m].T, s_ref), e
        assert np.all(qh[e, m:] == 0xAB) and np.all(sh[:, e * cap + m:(e + 1) * cap] == -1.0), e
