"""The C-ABI library without a GPU: it loads, exports every function the header declares,
and its host-side validation rejects bad arguments before anything is launched."""

import ctypes

import pytest

import moe_grouped_gemm_block_gb300 as g

INVALID, ALIGN = 1, 2
P = 1 << 20  # a 16-byte-aligned fake device address (never dereferenced: validation fails first)


@pytest.fixture(scope="module")
def lib():
    return g.lib()


def test_header_declares_the_four_calls_and_status():
    names = g.header_functions()
    for want in ("fp8_quantize_1x128", "fp8_quantize_128x128", "fp8_gemm_nt",
                 "fp8_grouped_gemm_contiguous", "fp8_grouped_gemm_masked", "fp8g_get_status",
                 "fp8g_status_string", "fp8g_last_config"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in g.header_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in g.STATUS.items():
        assert g.status_string(code) == name
    assert g.status_string(99) == "FP8G_UNKNOWN_STATUS"


@pytest.mark.parametrize("args,want", [
    ((P, 4, 100, 128, P, 128, P, 4, None), INVALID),     # K % 128
    ((P, -1, 128, 128, P, 128, P, 4, None), INVALID),    # M < 0
    ((P, 4, 128, 64, P, 128, P, 4, None), INVALID),      # ldx < K
    ((P, 8, 128, 128, P, 128, P, 4, None), INVALID),     # ld_sa < M
    ((None, 4, 128, 128, P, 128, P, 4, None), INVALID),  # null
    ((P + 8, 4, 128, 128, P, 128, P, 4, None), ALIGN),   # misaligned x
    ((P, 4, 128, 132, P, 128, P, 4, None), ALIGN),       # ldx % 8
    ((P, 4, 128, 128, P, 136, P, 4, None), ALIGN),       # ldq % 16
    ((P, 3, 128, 128, P, 128, P, 3, None), ALIGN),       # ld_sa % 4
])
def test_quantize_1x128_validation(lib, args, want):
    assert lib.fp8_quantize_1x128(*args) == want


def test_quantize_128x128_validation(lib):
    assert lib.fp8_quantize_128x128(P, 0, 128, 128, P, P, None) == INVALID
    assert lib.fp8_quantize_128x128(P, 1, 128, 130, P, P, None) == INVALID
    assert lib.fp8_quantize_128x128(P, 1, 128, 128, P + 4, P, None) == ALIGN


def _nt(**kw):
    a = dict(A=P, lda=256, sA=P, ld_sa=64, B=P, ldb=256, sB=P, D=P, ldd=256, M=64, N=256, K=256, s=None)
    a.update(kw)
    return tuple(a.values())


@pytest.mark.parametrize("kw,want", [
    (dict(K=200), INVALID), (dict(N=250), INVALID), (dict(M=-1), INVALID), (dict(N=0), INVALID),
    (dict(lda=128), INVALID), (dict(ldd=128), INVALID), (dict(ld_sa=32), INVALID),
    (dict(A=None), INVALID), (dict(sB=None), INVALID),
    (dict(A=P + 1), ALIGN), (dict(D=P + 2), ALIGN), (dict(lda=264), ALIGN), (dict(ldd=260), ALIGN),
    (dict(ld_sa=66), ALIGN),
])
def test_gemm_nt_validation(lib, kw, want):
    assert lib.fp8_gemm_nt(*_nt(**kw)) == want


def test_grouped_validation(lib):
    off = P
    # contiguous: E range, M_total % 128, N % 16, K % 128, ld_sa, null offsets
    assert lib.fp8_grouped_gemm_contiguous(P, P, 256, P, P, P, off, 0, 256, 256, 256, None) == INVALID
    assert lib.fp8_grouped_gemm_contiguous(P, P, 256, P, P, P, off, 5000, 256, 256, 256, None) == INVALID
    assert lib.fp8_grouped_gemm_contiguous(P, P, 256, P, P, P, off, 2, 200, 256, 256, None) == INVALID
    assert lib.fp8_grouped_gemm_contiguous(P, P, 256, P, P, P, off, 2, 256, 250, 256, None) == INVALID
    assert lib.fp8_grouped_gemm_contiguous(P, P, 128, P, P, P, off, 2, 256, 256, 256, None) == INVALID
    assert lib.fp8_grouped_gemm_contiguous(P, P, 256, P, P, P, None, 2, 256, 256, 256, None) == INVALID
    assert lib.fp8_grouped_gemm_contiguous(P, P, 256, P, P, P, off + 2, 2, 256, 256, 256, None) == ALIGN
    # masked: cap % 16, ld_sa >= E*cap, negative cap
    assert lib.fp8_grouped_gemm_masked(P, P, 512, P, P, P, P, 2, 100, 256, 256, None) == INVALID
    assert lib.fp8_grouped_gemm_masked(P, P, 128, P, P, P, P, 2, 128, 256, 256, None) == INVALID
    assert lib.fp8_grouped_gemm_masked(P, P, 512, P, P, P, P, 2, -16, 256, 256, None) == INVALID
    assert lib.fp8_grouped_gemm_masked(P, P, 512, P, P + 4, P, P, 2, 128, 256, 256, None) == ALIGN


def test_valid_arguments_without_a_gpu_report_an_error_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present: covered by the GPU tests")
    assert lib.fp8_gemm_nt(*_nt()) in (3, 4)  # no device: CUDA error, nothing launched
    assert lib.fp8g_get_status(None) in (3, 4)


def test_last_config_null_pointer(lib):
    null = ctypes.POINTER(ctypes.c_int)()
    assert lib.fp8g_last_config(null, null, null) == INVALID
    assert lib.fp8g_last_split(null) == INVALID
    assert lib.fp8g_last_swap_ab(null) == INVALID
    assert lib.fp8g_last_cluster_k(null) == INVALID


def test_binding_fails_loudly_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(g, "_lib", None)
    monkeypatch.setattr(g, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        g.lib()


@pytest.mark.parametrize("kw,want", [
    (dict(K=200), INVALID), (dict(N=250), INVALID), (dict(M=-1), INVALID), (dict(ldd=128), INVALID),
    (dict(A=None), INVALID), (dict(A=P + 1), ALIGN), (dict(lda=264), ALIGN),
])
def test_gemm_nt_noalloc_validation(lib, kw, want):
    # the fixed-scratch variant takes fp8_gemm_nt's arguments and rules
    assert lib.fp8_gemm_nt_noalloc(*_nt(**kw)) == want


def test_gemm_nt_noalloc_m_zero_is_a_noop(lib):
    assert lib.fp8_gemm_nt_noalloc(*_nt(M=0, A=None, sA=None, B=None, sB=None, D=None)) == 0


def _nts(**kw):
    a = dict(A=P, lda=256, sA=P, pa=1, B=P, ldb=256, sB=P, pb=1, D=P, ldd=256, M=64, N=256, K=256, s=None)
    a.update(kw)
    return tuple(a.values())


@pytest.mark.parametrize("kw,want", [
    (dict(K=200), INVALID), (dict(N=250), INVALID), (dict(M=-1), INVALID), (dict(ldd=128), INVALID),
    (dict(pa=2), INVALID), (dict(pb=-1), INVALID), (dict(A=None), INVALID), (dict(sA=None), INVALID),
    (dict(A=P + 1), ALIGN), (dict(lda=264), ALIGN), (dict(sA=P + 2), ALIGN),
    (dict(sB=P + 4), ALIGN),            # one scale per column: float4 reads need 16-byte alignment
])
def test_gemm_nt_scaled_validation(lib, kw, want):
    assert lib.fp8_gemm_nt_scaled(*_nts(**kw)) == want


def test_gemm_nt_scaled_per_tensor_b_needs_only_4_byte_alignment(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present: covered by the GPU tests")
    # passes validation (then fails for want of a device)
    assert lib.fp8_gemm_nt_scaled(*_nts(sB=P + 4, pb=0)) in (3, 4)
    assert lib.fp8_gemm_nt_scaled(*_nts(M=0, A=None, sA=None, B=None, sB=None, D=None)) == 0


def test_grouped_scaled_validation(lib):
    c, m = lib.fp8_grouped_gemm_contiguous_scaled, lib.fp8_grouped_gemm_masked_scaled
    assert c(P, P, 1, P, P, 1, P, P, 0, 256, 256, 256, None) == INVALID      # E
    assert c(P, P, 1, P, P, 1, P, P, 2, 200, 256, 256, None) == INVALID      # M_total % 128
    assert c(P, P, 3, P, P, 1, P, P, 2, 256, 256, 256, None) == INVALID      # mode flag
    assert c(P, P, 1, P, P, 1, P, None, 2, 256, 256, 256, None) == INVALID   # offsets
    assert c(P, P, 1, P, P + 8, 1, P, P, 2, 256, 256, 256, None) == ALIGN
    assert m(P, P, 1, P, P, 1, P, P, 2, 100, 256, 256, None) == INVALID      # cap % 16
    assert m(P, P, 1, P, P, 0, P, P, 2, 128, 250, 256, None) == INVALID      # N % 16
    assert m(P, P + 1, 1, P, P, 0, P, P, 2, 128, 256, 256, None) == ALIGN


def test_quantise_per_row_and_per_tensor_validation(lib):
    r, t = lib.fp8_quantize_per_row, lib.fp8_quantize_per_tensor
    assert r(P, 4, 100, 128, P, 128, P, None) == INVALID      # K % 128
    assert r(P, 4, 128, 64, P, 128, P, None) == INVALID       # ldx < K
    assert r(P, 0, 128, 128, None, 128, None, None) == 0      # M == 0: no-op
    assert r(P + 8, 4, 128, 128, P, 128, P, None) == ALIGN
    assert r(P, 4, 128, 128, P, 136, P, None) == ALIGN        # ldq % 16
    assert t(P, 0, 4, 128, 128, P, 128, P, None) == INVALID   # E
    assert t(P, 1, 4, 128, 128, P, 128, None, None) == INVALID
    assert t(P, 1, 4, 128, 128, P, 128, P + 2, None) == ALIGN
    assert t(P, 1, 1 << 28, 128, 128, P, 128, P, None) == INVALID  # M * K / 8 >= 2^31


def test_backward_entry_points_validation(lib):
    q = lib.fp8_quantize_1x128_e5m2
    assert q(P, 4, 100, 128, P, 128, P, 4, None) == INVALID          # K % 128
    assert q(P, 8, 128, 128, P, 128, P, 4, None) == INVALID          # ld_sa < M
    assert q(P + 8, 4, 128, 128, P, 128, P, 4, None) == ALIGN
    assert q(P, 0, 128, 128, None, 128, None, 4, None) == 0           # M == 0: no-op
    assert lib.fp8_gemm_nt_dgrad(*_nt(K=200)) == INVALID
    assert lib.fp8_gemm_nt_dgrad(*_nt(A=P + 1)) == ALIGN
    assert lib.fp8_gemm_nt_dgrad(*_nt(M=0, A=None, sA=None, B=None, sB=None, D=None)) == 0
    c = lib.fp8_grouped_gemm_contiguous_dgrad
    assert c(P, P, 256, P, P, P, P, 2, 200, 256, 256, None) == INVALID  # M_total % 128
    assert c(P, P, 256, P, P, P, P + 2, 2, 256, 256, 256, None) == ALIGN
    w = lib.fp8_grouped_gemm_wgrad
    # (A, lda, sA, ld_sa, B, ldb, sB, ld_sb, D, offsets, E, M, N, T, stream)
    assert w(P, 256, P, 64, P, 256, P, 256, P, P, 2, 64, 256, 200, None) == INVALID   # T % 128
    assert w(P, 256, P, 64, P, 256, P, 256, P, P, 2, 72, 256, 256, None) == INVALID   # M % 16
    assert w(P, 256, P, 32, P, 256, P, 256, P, P, 2, 64, 256, 256, None) == INVALID   # ld_sa < M
    assert w(P, 256, P, 64, P, 256, P, 128, P, P, 2, 64, 256, 256, None) == INVALID   # ld_sb < N
    assert w(P, 128, P, 64, P, 256, P, 256, P, P, 2, 64, 256, 256, None) == INVALID   # lda < T
    assert w(P, 256, P, 64, P, 256, P, 256, P, P, 0, 64, 256, 256, None) == INVALID   # E
    assert w(P, 256, P, 64, P, 256, P, 256, P, P + 2, 2, 64, 256, 256, None) == ALIGN
    assert w(P, 256, P, 66, P, 256, P, 256, P, P, 2, 64, 256, 256, None) == ALIGN     # ld_sa % 4
    assert w(P, 256, P, 64, P, 256, P, 256, P, P, 2, 0, 256, 256, None) == 0          # M == 0: no-op


def test_masked_quantiser_validation(lib):
    f = lib.fp8_quantize_1x128_masked
    # (x, E, cap, K, masked_m, q, sA, ld_sa, stream)
    assert f(P, 0, 256, 128, P, P, P, 256, None) == INVALID      # E
    assert f(P, 2, 256, 100, P, P, P, 512, None) == INVALID      # K % 128
    assert f(P, 2, 256, 128, P, P, P, 256, None) == INVALID      # ld_sa < E*cap
    assert f(P, 2, 0, 128, None, None, None, 0, None) == 0        # cap == 0: no-op
    assert f(P, 2, 256, 128, None, P, P, 512, None) == INVALID   # counts
    assert f(P + 8, 2, 256, 128, P, P, P, 512, None) == ALIGN
    assert f(P, 2, 256, 128, P + 2, P, P, 512, None) == ALIGN
    assert f(P, 2, 256, 128, P, P, P, 514, None) == ALIGN        # ld_sa % 4


def test_selftest_validation(lib):
    f = lib.fp8g_selftest_bounded_waits
    assert f(0, P, None) == INVALID
    assert f(-5, P, None) == INVALID
    assert f(1 << 41, P, None) == INVALID
    assert f(1000, None, None) == INVALID
    assert f(1000, P + 2, None) == ALIGN
