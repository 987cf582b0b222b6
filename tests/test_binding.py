"""The Python binding's argument checks (no GPU): wrong dtypes, shapes or layouts raise ValueError before
anything reaches the library, and the helpers size their outputs as the C ABI expects."""

import pytest
import torch

import moe_grouped_gemm_block_gb300 as g


def _u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


def _f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def _bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def test_gemm_checks_operand_types():
    with pytest.raises(ValueError, match="A: e4m3"):
        g.fp8_gemm_nt(_f32(4, 128), _f32(1, 4), _u8(16, 128), _f32(1, 1), _bf16(4, 16))
    with pytest.raises(ValueError, match="D: bf16"):
        g.fp8_gemm_nt(_u8(4, 128), _f32(1, 4), _u8(16, 128), _f32(1, 1), _f32(4, 16))


def test_scaled_gemm_checks_scale_counts():
    with pytest.raises(ValueError, match="sA"):
        g.fp8_gemm_nt_scaled(_u8(4, 128), _f32(3), _u8(16, 128), _f32(16), _bf16(4, 16))
    with pytest.raises(ValueError, match="sB"):
        g.fp8_gemm_nt_scaled(_u8(4, 128), _f32(4), _u8(16, 128), _f32(5), _bf16(4, 16))
    with pytest.raises(ValueError, match="sB"):
        g.fp8_grouped_gemm_contiguous_scaled(_u8(128, 128), _f32(128), _u8(2, 16, 128), _f32(3), _bf16(128, 16),
                                             torch.zeros(3, dtype=torch.int32))
    # group offsets must be device memory: the kernel reads them, the host never does
    with pytest.raises(ValueError, match="CUDA tensors"):
        g.fp8_grouped_gemm_contiguous_scaled(_u8(128, 128), _f32(128), _u8(2, 16, 128), _f32(2), _bf16(128, 16),
                                             torch.zeros(3, dtype=torch.int32))


def test_grouped_calls_check_group_tensors():
    with pytest.raises(ValueError, match="group_offsets"):
        g.fp8_grouped_gemm_contiguous(_u8(128, 128), _f32(1, 128), _u8(2, 16, 128), _f32(2, 1, 1),
                                      _bf16(128, 16), torch.zeros(3, dtype=torch.int64))
    with pytest.raises(ValueError, match="CUDA tensors"):
        g.fp8_grouped_gemm_masked(_u8(2, 16, 128), _f32(1, 32), _u8(2, 16, 128), _f32(2, 1, 1),
                                  _bf16(2, 16, 16), torch.zeros(2, dtype=torch.int32))  # not on the device


def test_quantiser_checks():
    with pytest.raises(ValueError, match="x: bf16"):
        g.fp8_quantize_1x128(_f32(4, 128), _u8(4, 128), _f32(1, 4))
    with pytest.raises(ValueError, match="sA"):
        g.fp8_quantize_1x128(_bf16(4, 256), _u8(4, 256), _f32(1, 4))  # K/128 = 2 rows of scales
    with pytest.raises(ValueError, match="s: f32"):
        g.fp8_quantize_per_row(_bf16(4, 128), _u8(4, 128), _f32(5))
    with pytest.raises(ValueError, match="s: f32"):
        g.fp8_quantize_per_tensor(_bf16(3, 4, 128), _u8(3, 4, 128), _f32(1))
    with pytest.raises(ValueError, match="q: e5m2"):
        g.fp8_quantize_1x128_e5m2(_bf16(4, 128), _f32(4, 128), _f32(1, 4))


def test_wgrad_checks_operands_and_offsets():
    with pytest.raises(ValueError, match="D: bf16"):
        g.fp8_grouped_gemm_wgrad(_u8(16, 256), _f32(2, 16), _u8(32, 256), _f32(2, 32), _bf16(2, 16 * 32),
                                 torch.zeros(3, dtype=torch.int32))
    with pytest.raises(ValueError, match="offsets: int32 device tensor"):
        g.fp8_grouped_gemm_wgrad(_u8(16, 256), _f32(2, 16), _u8(32, 256), _f32(2, 32), _bf16(2, 16, 32),
                                 torch.zeros(3, dtype=torch.int64))
    with pytest.raises(ValueError, match="CUDA tensors"):
        g.fp8_grouped_gemm_wgrad(_u8(16, 256), _f32(2, 16), _u8(32, 256), _f32(2, 32), _bf16(2, 16, 32),
                                 torch.zeros(3, dtype=torch.int32))


def test_route_capacity_covers_the_worst_padding():
    for T, k, E in [(0, 1, 1), (1, 2, 8), (4096, 2, 8), (5, 1, 2048)]:
        cap = g.route_capacity(T, k, E)
        assert cap % 128 == 0 and cap >= T * k + 127 * E


@pytest.mark.parametrize("fn", [g.fp8_gemm_nt, g.fp8_gemm_nt_noalloc])
def test_dense_gemm_checks_every_shape_before_a_launch(fn):
    # M=4, N=16, K=256: A [4,256], sA [2, >=4], B [16,256], sB [1,2], D [4,16]
    A, sA, B, sB, D = _u8(4, 256), _f32(2, 4), _u8(16, 256), _f32(1, 2), _bf16(4, 16)
    with pytest.raises(ValueError, match="D \\[M,N\\]"):
        fn(A, sA, B, sB, _bf16(3, 16))  # too few rows: TMA stores would run past D
    with pytest.raises(ValueError, match="B \\[N,K\\]"):
        fn(A, sA, _u8(16, 128), sB, D)  # B's K differs from A's
    with pytest.raises(ValueError, match="sA"):
        fn(A, _f32(2, 3), B, sB, D)  # fewer A-row scales than rows
    with pytest.raises(ValueError, match="sA"):
        fn(A, _f32(1, 4), B, sB, D)  # one K block of scales for two
    with pytest.raises(ValueError, match="sB"):
        fn(A, sA, B, _f32(1, 1), D)  # one weight scale where two are read
    with pytest.raises(ValueError, match="CUDA tensors"):
        fn(A, sA, B, sB, D)  # consistent shapes, but host memory


def test_grouped_gemms_check_shapes():
    offs = torch.zeros(3, dtype=torch.int32)
    with pytest.raises(ValueError, match="shapes"):  # D rows != M_total
        g.fp8_grouped_gemm_contiguous(_u8(256, 128), _f32(1, 256), _u8(2, 16, 128), _f32(2, 1, 1),
                                      _bf16(128, 16), offs)
    with pytest.raises(ValueError, match="sB"):  # one expert's weight scales for two experts
        g.fp8_grouped_gemm_contiguous(_u8(256, 128), _f32(1, 256), _u8(2, 16, 128), _f32(1, 1, 1),
                                      _bf16(256, 16), offs)
    counts = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="shapes"):  # D's capacity differs from A's
        g.fp8_grouped_gemm_masked(_u8(2, 16, 128), _f32(1, 32), _u8(2, 16, 128), _f32(2, 1, 1),
                                  _bf16(2, 8, 16), counts)
    with pytest.raises(ValueError, match="sA"):  # scales for fewer rows than E * cap
        g.fp8_grouped_gemm_masked(_u8(2, 16, 128), _f32(1, 16), _u8(2, 16, 128), _f32(2, 1, 1),
                                  _bf16(2, 16, 16), counts)
