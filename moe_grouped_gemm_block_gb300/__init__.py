"""FP8 e4m3 block-scaled GEMM for GB300 (sm_103a): Python binding of ``libfp8gemm.so``.

Argument marshalling only: every step runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams.  The C ABI is declared in ``include/fp8gemm.h``;
functions here carry the same names and take torch tensors:

    fp8_quantize_1x128(x, q, sA)                      x bf16 [M,K] -> q e4m3 [M,K], sA f32 [K/128, ld_sa]
    fp8_quantize_128x128(w, q, sB)                    w bf16 [E,N,K] (or [N,K]) -> q, sB f32 [E,ceil(N/128),K/128]
    fp8_gemm_nt(A, sA, B, sB, D)                      D bf16 [M,N] = A [M,K] x B [N,K]^T with block scales
    fp8_grouped_gemm_contiguous(A, sA, B, sB, D, group_offsets)
    fp8_grouped_gemm_masked(A, sA, B, sB, D, masked_m)
    fp8_route_gather_quantize_1x128 (see route_gather_quantize_1x128)
    fp8_quantize_per_row(x, q, s) / fp8_quantize_per_tensor(x, q, s)   one scale per row / per tensor
    fp8_gemm_nt_scaled(A, sA, B, sB, D)                  epilogue scales: sA [M] or [1], sB [N] or [1]
    fp8_grouped_gemm_contiguous_scaled(A, sA, B, sB, D, group_offsets)   sB [E,N] or [E]
    fp8_grouped_gemm_masked_scaled(A, sA, B, sB, D, masked_m)
    fp8_quantize_1x128_masked(x, q, sA, masked_m)      masked layout: only each expert's valid rows
    fp8_quantize_1x128_e5m2(x, q, sA)                  gradients: e5m2 codes, s = amax / 57344
    fp8_gemm_nt_dgrad(A, sA, B, sB, D)                 data gradient: A e5m2 [M,K], B e4m3 [N,K] (= W^T)
    fp8_grouped_gemm_contiguous_dgrad(A, sA, B, sB, D, group_offsets)   grouped data gradient
    fp8_grouped_gemm_wgrad(A, sA, B, sB, D, offsets)   weight gradient per expert over its tokens

e4m3 tensors may be torch.uint8 or torch.float8_e4m3fn.  Work is enqueued on the
current CUDA stream of the tensors' device.  A non-zero status raises Fp8GemmError.
Convenience wrappers (``quantize_1x128``, ``quantize_128x128``, ``gemm_nt``) allocate
their outputs with torch and call the above.
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libfp8gemm.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "fp8gemm.h")

STATUS = {
    0: "FP8G_OK", 1: "FP8G_ERR_INVALID_ARG", 2: "FP8G_ERR_ALIGNMENT",
    3: "FP8G_ERR_UNSUPPORTED_DEVICE", 4: "FP8G_ERR_CUDA", 5: "FP8G_ERR_TIMEOUT",
    6: "FP8G_ERR_DEVICE_ASSERT",
}


class Fp8GemmError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what} failed: {STATUS.get(code, code)}")


_lib = None

_I64, _I32, _P, _FP = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p
_SIGNATURES = {
    "fp8_quantize_1x128": [_P, _I64, _I64, _I64, _P, _I64, _FP, _I64, _P],
    "fp8_quantize_128x128": [_P, _I64, _I64, _I64, _P, _FP, _P],
    "fp8_gemm_nt": [_P, _I64, _FP, _I64, _P, _I64, _FP, _P, _I64, _I64, _I64, _I64, _P],
    "fp8_gemm_nt_noalloc": [_P, _I64, _FP, _I64, _P, _I64, _FP, _P, _I64, _I64, _I64, _I64, _P],
    "fp8_route_gather_quantize_1x128": [_P, _I64, _I64, _I64, _P, _I32, _I32, _P, _I64, _FP, _I64, _P, _P,
                                        _P, _I64, _P],
    "fp8_grouped_gemm_contiguous": [_P, _FP, _I64, _P, _FP, _P, _P, _I32, _I64, _I64, _I64, _P],
    "fp8_grouped_gemm_masked": [_P, _FP, _I64, _P, _FP, _P, _P, _I32, _I64, _I64, _I64, _P],
    "fp8_quantize_per_row": [_P, _I64, _I64, _I64, _P, _I64, _FP, _P],
    "fp8_quantize_per_tensor": [_P, _I64, _I64, _I64, _I64, _P, _I64, _FP, _P],
    "fp8_gemm_nt_scaled": [_P, _I64, _FP, _I32, _P, _I64, _FP, _I32, _P, _I64, _I64, _I64, _I64, _P],
    "fp8_grouped_gemm_contiguous_scaled": [_P, _FP, _I32, _P, _FP, _I32, _P, _P, _I32, _I64, _I64, _I64, _P],
    "fp8_grouped_gemm_masked_scaled": [_P, _FP, _I32, _P, _FP, _I32, _P, _P, _I32, _I64, _I64, _I64, _P],
    "fp8_quantize_1x128_masked": [_P, _I32, _I64, _I64, _P, _P, _FP, _I64, _P],
    "fp8_quantize_1x128_e5m2": [_P, _I64, _I64, _I64, _P, _I64, _FP, _I64, _P],
    "fp8_gemm_nt_dgrad": [_P, _I64, _FP, _I64, _P, _I64, _FP, _P, _I64, _I64, _I64, _I64, _P],
    "fp8_grouped_gemm_contiguous_dgrad": [_P, _FP, _I64, _P, _FP, _P, _P, _I32, _I64, _I64, _I64, _P],
    "fp8_grouped_gemm_wgrad": [_P, _I64, _FP, _I64, _P, _I64, _FP, _I64, _P, _P, _I32, _I64, _I64, _I64, _P],
    "fp8g_selftest_bounded_waits": [_I64, _P, _P],
    "fp8g_get_status": [_P],
    "fp8g_last_config": [ctypes.POINTER(ctypes.c_int)] * 3,
    "fp8g_last_split": [ctypes.POINTER(ctypes.c_int)],
    "fp8g_last_swap_ab": [ctypes.POINTER(ctypes.c_int)],
    "fp8g_last_cluster_k": [ctypes.POINTER(ctypes.c_int)],
}


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m moe_grouped_gemm_block_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        handle.fp8g_status_string.argtypes = [ctypes.c_int]
        handle.fp8g_status_string.restype = ctypes.c_char_p
        _lib = handle
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/fp8gemm.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return re.findall(r"^(?:int|const char\*)\s+(\w+)\(", text, flags=re.M)


def status_string(code: int) -> str:
    return lib().fp8g_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != 0:
        raise Fp8GemmError(code, what)


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def _is_fp8(t: torch.Tensor) -> bool:
    return t.dtype in (torch.uint8, torch.float8_e4m3fn)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _block_scales(sA: torch.Tensor, sB: torch.Tensor, rows: int, N: int, K: int, E: int) -> int:
    """Checks the 1x128 activation scales sA [K/128, ld_sa >= rows] (row stride ld_sa, unit column
    stride) and the 128x128 weight scales sB [E, ceil(N/128), K/128] (contiguous) against the
    problem size, so that no kernel reads past either; returns ld_sa."""
    _need(sA.dtype == torch.float32 and sA.dim() == 2 and sA.shape[0] == K // 128 and sA.stride(1) == 1
          and sA.shape[1] >= rows and (sA.shape[0] == 1 or sA.stride(0) >= sA.shape[1]),
          f"sA: f32 [K/128, ld_sa >= {rows}]")
    _need(sB.dtype == torch.float32 and sB.is_contiguous() and sB.numel() == E * ((N + 127) // 128) * (K // 128),
          f"sB: f32 [{E}, ceil(N/128), K/128] contiguous")
    return sA.stride(0) if sA.shape[0] > 1 else sA.shape[1]


def _on_one_device(*ts: torch.Tensor):
    """Every operand, group offsets and counts included, in device memory of one GPU: the library
    dereferences them all on the device (the host never reads the offsets or counts)."""
    dev = ts[0].device
    _need(all(t.is_cuda and t.device == dev for t in ts), "operands: CUDA tensors on one device")


# ------------------------------------------------------------------ C-ABI calls

def fp8_quantize_1x128(x: torch.Tensor, q: torch.Tensor, sA: torch.Tensor) -> None:
    _need(x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1, "x: bf16 [M,K], K contiguous")
    _need(_is_fp8(q) and q.shape == x.shape and q.stride(1) == 1, "q: e4m3 [M,K]")
    M, K = x.shape
    _need(sA.dtype == torch.float32 and sA.dim() == 2 and sA.shape[0] == K // 128 and sA.stride(1) == 1,
          "sA: f32 [K/128, ld_sa]")
    ld_sa = sA.stride(0) if sA.shape[0] > 1 else sA.shape[1]
    _need(sA.shape[1] >= M, "sA: f32 [K/128, ld_sa >= M]")
    _on_one_device(x, q, sA)
    _check(lib().fp8_quantize_1x128(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(sA), ld_sa,
                                    _stream(x)), "fp8_quantize_1x128")


def fp8_quantize_128x128(w: torch.Tensor, q: torch.Tensor, sB: torch.Tensor) -> None:
    _need(w.dtype == torch.bfloat16 and w.is_contiguous() and w.dim() in (2, 3), "w: bf16 [E,N,K] contiguous")
    _need(_is_fp8(q) and q.shape == w.shape and q.is_contiguous(), "q: e4m3, same shape as w")
    E, N, K = (1, *w.shape) if w.dim() == 2 else w.shape
    _need(sB.dtype == torch.float32 and sB.is_contiguous() and sB.numel() == E * ((N + 127) // 128) * (K // 128),
          "sB: f32 [E, ceil(N/128), K/128] contiguous")
    _on_one_device(w, q, sB)
    _check(lib().fp8_quantize_128x128(_ptr(w), E, N, K, _ptr(q), _ptr(sB), _stream(w)),
           "fp8_quantize_128x128")


def fp8_gemm_nt(A, sA, B, sB, D) -> None:
    _need(_is_fp8(A) and A.dim() == 2 and A.stride(1) == 1, "A: e4m3 [M,K]")
    _need(_is_fp8(B) and B.dim() == 2 and B.stride(1) == 1, "B: e4m3 [N,K]")
    _need(D.dtype == torch.bfloat16 and D.dim() == 2 and D.stride(1) == 1, "D: bf16 [M,N]")
    M, K = A.shape
    N = B.shape[0]
    _need(B.shape[1] == K and D.shape == (M, N), "shapes: A [M,K], B [N,K], D [M,N]")
    ld_sa = _block_scales(sA, sB, M, N, K, 1)
    _on_one_device(A, sA, B, sB, D)
    _check(lib().fp8_gemm_nt(_ptr(A), A.stride(0), _ptr(sA), ld_sa, _ptr(B), B.stride(0), _ptr(sB),
                             _ptr(D), D.stride(0), M, N, K, _stream(A)), "fp8_gemm_nt")


def fp8_gemm_nt_noalloc(A, sA, B, sB, D) -> None:
    """fp8_gemm_nt without any device allocation: the library's fixed scratch buffer replaces the
    per-stream stream-K workspace.  Calls that overlap in time share that buffer and race, so
    order them; make the first call on each device before capturing any stream."""
    _need(_is_fp8(A) and A.dim() == 2 and A.stride(1) == 1, "A: e4m3 [M,K]")
    _need(_is_fp8(B) and B.dim() == 2 and B.stride(1) == 1, "B: e4m3 [N,K]")
    _need(D.dtype == torch.bfloat16 and D.dim() == 2 and D.stride(1) == 1, "D: bf16 [M,N]")
    M, K = A.shape
    N = B.shape[0]
    _need(B.shape[1] == K and D.shape == (M, N), "shapes: A [M,K], B [N,K], D [M,N]")
    ld_sa = _block_scales(sA, sB, M, N, K, 1)
    _on_one_device(A, sA, B, sB, D)
    _check(lib().fp8_gemm_nt_noalloc(_ptr(A), A.stride(0), _ptr(sA), ld_sa, _ptr(B), B.stride(0), _ptr(sB),
                                     _ptr(D), D.stride(0), M, N, K, _stream(A)), "fp8_gemm_nt_noalloc")


def fp8_grouped_gemm_contiguous(A, sA, B, sB, D, group_offsets) -> None:
    _need(_is_fp8(A) and A.dim() == 2 and A.is_contiguous(), "A: e4m3 [M_total,K] contiguous")
    _need(_is_fp8(B) and B.dim() == 3 and B.is_contiguous(), "B: e4m3 [E,N,K] contiguous")
    _need(D.dtype == torch.bfloat16 and D.is_contiguous(), "D: bf16 [M_total,N] contiguous")
    _need(group_offsets.dtype == torch.int32, "group_offsets: int32 device tensor")
    M_total, K = A.shape
    E, N, _ = B.shape
    _need(B.shape[2] == K and D.shape == (M_total, N) and group_offsets.numel() == E + 1,
          "shapes: A [M_total,K], B [E,N,K], D [M_total,N], group_offsets [E+1]")
    ld_sa = _block_scales(sA, sB, M_total, N, K, E)
    _on_one_device(A, sA, B, sB, D, group_offsets)
    _check(lib().fp8_grouped_gemm_contiguous(_ptr(A), _ptr(sA), ld_sa, _ptr(B), _ptr(sB), _ptr(D),
                                             _ptr(group_offsets), E, M_total, N, K, _stream(A)),
           "fp8_grouped_gemm_contiguous")


def fp8_grouped_gemm_masked(A, sA, B, sB, D, masked_m) -> None:
    _need(_is_fp8(A) and A.dim() == 3 and A.is_contiguous(), "A: e4m3 [E,cap,K] contiguous")
    _need(_is_fp8(B) and B.dim() == 3 and B.is_contiguous(), "B: e4m3 [E,N,K] contiguous")
    _need(D.dtype == torch.bfloat16 and D.is_contiguous(), "D: bf16 [E,cap,N] contiguous")
    _need(masked_m.dtype == torch.int32, "masked_m: int32 device tensor")
    E, cap, K = A.shape
    N = B.shape[1]
    _need(B.shape[0] == E and B.shape[2] == K and D.shape == (E, cap, N) and masked_m.numel() == E,
          "shapes: A [E,cap,K], B [E,N,K], D [E,cap,N], masked_m [E]")
    ld_sa = _block_scales(sA, sB, E * cap, N, K, E)
    _on_one_device(A, sA, B, sB, D, masked_m)
    _check(lib().fp8_grouped_gemm_masked(_ptr(A), _ptr(sA), ld_sa, _ptr(B), _ptr(sB), _ptr(D),
                                         _ptr(masked_m), E, cap, N, K, _stream(A)),
           "fp8_grouped_gemm_masked")


def fp8_quantize_per_row(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor) -> None:
    _need(x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1, "x: bf16 [M,K], K contiguous")
    _need(_is_fp8(q) and q.shape == x.shape and q.stride(1) == 1, "q: e4m3 [M,K]")
    M, K = x.shape
    _need(s.dtype == torch.float32 and s.is_contiguous() and s.numel() == M, "s: f32 [M]")
    _on_one_device(x, q, s)
    _check(lib().fp8_quantize_per_row(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(s), _stream(x)),
           "fp8_quantize_per_row")


def fp8_quantize_per_tensor(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor) -> None:
    """x bf16 [M,K] (one tensor) or [E,M,K] (E tensors, each its own scale) -> q, s f32 [E]."""
    _need(x.dtype == torch.bfloat16 and x.dim() in (2, 3) and x.is_contiguous(), "x: bf16 [(E,) M, K] contiguous")
    _need(_is_fp8(q) and q.shape == x.shape and q.is_contiguous(), "q: e4m3, same shape as x")
    E, M, K = (1, *x.shape) if x.dim() == 2 else x.shape
    _need(s.dtype == torch.float32 and s.is_contiguous() and s.numel() == E, "s: f32 [E]")
    _on_one_device(x, q, s)
    _check(lib().fp8_quantize_per_tensor(_ptr(x), E, M, K, K, _ptr(q), K, _ptr(s), _stream(x)),
           "fp8_quantize_per_tensor")


def _epi_scale(t: torch.Tensor, n: int, what: str) -> int:
    """1 when t holds one scale per row / column (n of them), 0 when it holds one."""
    _need(t.dtype == torch.float32 and t.is_contiguous() and t.numel() in (1, n), f"{what}: f32 [{n}] or [1]")
    return 1 if t.numel() == n and n != 1 else 0


def fp8_gemm_nt_scaled(A, sA, B, sB, D) -> None:
    _need(_is_fp8(A) and A.dim() == 2 and A.stride(1) == 1, "A: e4m3 [M,K]")
    _need(_is_fp8(B) and B.dim() == 2 and B.stride(1) == 1, "B: e4m3 [N,K]")
    _need(D.dtype == torch.bfloat16 and D.dim() == 2 and D.stride(1) == 1, "D: bf16 [M,N]")
    M, K = A.shape
    N = B.shape[0]
    _need(B.shape[1] == K and D.shape == (M, N), "shapes: A [M,K], B [N,K], D [M,N]")
    pa, pb = _epi_scale(sA, M, "sA"), _epi_scale(sB, N, "sB")
    _on_one_device(A, sA, B, sB, D)
    _check(lib().fp8_gemm_nt_scaled(_ptr(A), A.stride(0), _ptr(sA), pa, _ptr(B), B.stride(0), _ptr(sB), pb,
                                    _ptr(D), D.stride(0), M, N, K, _stream(A)), "fp8_gemm_nt_scaled")


def fp8_grouped_gemm_contiguous_scaled(A, sA, B, sB, D, group_offsets) -> None:
    _need(_is_fp8(A) and A.dim() == 2 and A.is_contiguous(), "A: e4m3 [M_total,K] contiguous")
    _need(_is_fp8(B) and B.dim() == 3 and B.is_contiguous(), "B: e4m3 [E,N,K] contiguous")
    _need(D.dtype == torch.bfloat16 and D.is_contiguous(), "D: bf16 [M_total,N] contiguous")
    _need(group_offsets.dtype == torch.int32, "group_offsets: int32 device tensor")
    M_total, K = A.shape
    E, N, _ = B.shape
    pa = _epi_scale(sA, M_total, "sA")
    _need(sB.dtype == torch.float32 and sB.is_contiguous() and sB.numel() in (E, E * N), "sB: f32 [E,N] or [E]")
    pb = 1 if sB.numel() == E * N and N != 1 else 0
    _need(B.shape[2] == K and D.shape == (M_total, N) and group_offsets.numel() == E + 1,
          "shapes: A [M_total,K], B [E,N,K], D [M_total,N], group_offsets [E+1]")
    _on_one_device(A, sA, B, sB, D, group_offsets)
    _check(lib().fp8_grouped_gemm_contiguous_scaled(_ptr(A), _ptr(sA), pa, _ptr(B), _ptr(sB), pb, _ptr(D),
                                                    _ptr(group_offsets), E, M_total, N, K, _stream(A)),
           "fp8_grouped_gemm_contiguous_scaled")


def fp8_grouped_gemm_masked_scaled(A, sA, B, sB, D, masked_m) -> None:
    _need(_is_fp8(A) and A.dim() == 3 and A.is_contiguous(), "A: e4m3 [E,cap,K] contiguous")
    _need(_is_fp8(B) and B.dim() == 3 and B.is_contiguous(), "B: e4m3 [E,N,K] contiguous")
    _need(D.dtype == torch.bfloat16 and D.is_contiguous(), "D: bf16 [E,cap,N] contiguous")
    _need(masked_m.dtype == torch.int32, "masked_m: int32 device tensor")
    E, cap, K = A.shape
    N = B.shape[1]
    pa = _epi_scale(sA, E * cap, "sA")
    _need(sB.dtype == torch.float32 and sB.is_contiguous() and sB.numel() in (E, E * N), "sB: f32 [E,N] or [E]")
    pb = 1 if sB.numel() == E * N and N != 1 else 0
    _need(B.shape[0] == E and B.shape[2] == K and D.shape == (E, cap, N) and masked_m.numel() == E,
          "shapes: A [E,cap,K], B [E,N,K], D [E,cap,N], masked_m [E]")
    _on_one_device(A, sA, B, sB, D, masked_m)
    _check(lib().fp8_grouped_gemm_masked_scaled(_ptr(A), _ptr(sA), pa, _ptr(B), _ptr(sB), pb, _ptr(D),
                                                _ptr(masked_m), E, cap, N, K, _stream(A)),
           "fp8_grouped_gemm_masked_scaled")


def fp8_quantize_1x128_masked(x: torch.Tensor, q: torch.Tensor, sA: torch.Tensor, masked_m: torch.Tensor) -> None:
    """x bf16 [E,cap,K] -> q e4m3 [E,cap,K], sA f32 [K/128, ld_sa >= E*cap]: only rows m < masked_m[e]."""
    _need(x.dtype == torch.bfloat16 and x.dim() == 3 and x.is_contiguous(), "x: bf16 [E,cap,K] contiguous")
    _need(_is_fp8(q) and q.shape == x.shape and q.is_contiguous(), "q: e4m3 [E,cap,K] contiguous")
    _need(masked_m.dtype == torch.int32, "masked_m: int32 device tensor")
    E, cap, K = x.shape
    _need(sA.dtype == torch.float32 and sA.dim() == 2 and sA.shape[0] == K // 128 and sA.stride(1) == 1,
          "sA: f32 [K/128, ld_sa]")
    ld_sa = sA.stride(0) if sA.shape[0] > 1 else sA.shape[1]
    _need(sA.shape[1] >= E * cap and masked_m.numel() == E, "sA: f32 [K/128, ld_sa >= E*cap]; masked_m [E]")
    _on_one_device(x, q, sA, masked_m)
    _check(lib().fp8_quantize_1x128_masked(_ptr(x), E, cap, K, _ptr(masked_m), _ptr(q), _ptr(sA), ld_sa,
                                           _stream(x)), "fp8_quantize_1x128_masked")


def fp8_quantize_1x128_e5m2(x: torch.Tensor, q: torch.Tensor, sA: torch.Tensor) -> None:
    _need(x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1, "x: bf16 [M,K], K contiguous")
    _need(q.dtype in (torch.uint8, torch.float8_e5m2) and q.shape == x.shape and q.stride(1) == 1, "q: e5m2 [M,K]")
    M, K = x.shape
    _need(sA.dtype == torch.float32 and sA.dim() == 2 and sA.shape[0] == K // 128 and sA.stride(1) == 1,
          "sA: f32 [K/128, ld_sa]")
    ld_sa = sA.stride(0) if sA.shape[0] > 1 else sA.shape[1]
    _need(sA.shape[1] >= M, "sA: f32 [K/128, ld_sa >= M]")
    _on_one_device(x, q, sA)
    _check(lib().fp8_quantize_1x128_e5m2(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(sA), ld_sa,
                                         _stream(x)), "fp8_quantize_1x128_e5m2")


def fp8_gemm_nt_dgrad(A, sA, B, sB, D) -> None:
    """fp8_gemm_nt with A in e5m2 (the output gradient dY) and B = W^T in e4m3."""
    _need(A.dtype in (torch.uint8, torch.float8_e5m2) and A.dim() == 2 and A.stride(1) == 1, "A: e5m2 [M,K]")
    _need(_is_fp8(B) and B.dim() == 2 and B.stride(1) == 1, "B: e4m3 [N,K]")
    _need(D.dtype == torch.bfloat16 and D.dim() == 2 and D.stride(1) == 1, "D: bf16 [M,N]")
    M, K = A.shape
    N = B.shape[0]
    _need(B.shape[1] == K and D.shape == (M, N), "shapes: A [M,K], B [N,K], D [M,N]")
    ld_sa = _block_scales(sA, sB, M, N, K, 1)
    _on_one_device(A, sA, B, sB, D)
    _check(lib().fp8_gemm_nt_dgrad(_ptr(A), A.stride(0), _ptr(sA), ld_sa, _ptr(B), B.stride(0), _ptr(sB),
                                   _ptr(D), D.stride(0), M, N, K, _stream(A)), "fp8_gemm_nt_dgrad")


def fp8_grouped_gemm_contiguous_dgrad(A, sA, B, sB, D, group_offsets) -> None:
    """fp8_grouped_gemm_contiguous with A in e5m2 (dY) and B [E, K_in, N] = each expert's W^T."""
    _need(A.dtype in (torch.uint8, torch.float8_e5m2) and A.dim() == 2 and A.is_contiguous(),
          "A: e5m2 [M_total,K] contiguous")
    _need(_is_fp8(B) and B.dim() == 3 and B.is_contiguous(), "B: e4m3 [E,N,K] contiguous")
    _need(D.dtype == torch.bfloat16 and D.is_contiguous(), "D: bf16 [M_total,N] contiguous")
    _need(group_offsets.dtype == torch.int32, "group_offsets: int32 device tensor")
    M_total, K = A.shape
    E, N, _ = B.shape
    _need(B.shape[2] == K and D.shape == (M_total, N) and group_offsets.numel() == E + 1,
          "shapes: A [M_total,K], B [E,N,K], D [M_total,N], group_offsets [E+1]")
    ld_sa = _block_scales(sA, sB, M_total, N, K, E)
    _on_one_device(A, sA, B, sB, D, group_offsets)
    _check(lib().fp8_grouped_gemm_contiguous_dgrad(_ptr(A), _ptr(sA), ld_sa, _ptr(B), _ptr(sB), _ptr(D),
                                                   _ptr(group_offsets), E, M_total, N, K, _stream(A)),
           "fp8_grouped_gemm_contiguous_dgrad")


def fp8_grouped_gemm_wgrad(A, sA, B, sB, D, offsets) -> None:
    """A e5m2 [M,T] (dY^T), sA f32 [T/128, ld_sa]; B e4m3 [N,T] (X^T), sB f32 [T/128, ld_sb];
    D bf16 [E,M,N]; offsets int32 [E+1] device (token ranges per expert, multiples of 128)."""
    _need(A.dtype in (torch.uint8, torch.float8_e5m2) and A.dim() == 2 and A.stride(1) == 1, "A: e5m2 [M,T]")
    _need(_is_fp8(B) and B.dim() == 2 and B.stride(1) == 1, "B: e4m3 [N,T]")
    _need(D.dtype == torch.bfloat16 and D.dim() == 3 and D.is_contiguous(), "D: bf16 [E,M,N] contiguous")
    _need(offsets.dtype == torch.int32, "offsets: int32 device tensor")
    M, T = A.shape
    N = B.shape[0]
    E = D.shape[0]
    _need(B.shape[1] == T and offsets.numel() == E + 1 and D.shape[1:] == (M, N), "shapes")
    for t, rows, name in ((sA, M, "sA"), (sB, N, "sB")):
        _need(t.dtype == torch.float32 and t.dim() == 2 and t.shape[0] == T // 128 and t.stride(1) == 1
              and t.shape[1] >= rows and (t.shape[0] == 1 or t.stride(0) >= t.shape[1]),
              f"{name}: f32 [T/128, ld >= {rows}]")
    ld_sa = sA.stride(0) if sA.shape[0] > 1 else sA.shape[1]
    ld_sb = sB.stride(0) if sB.shape[0] > 1 else sB.shape[1]
    _on_one_device(A, sA, B, sB, D, offsets)
    _check(lib().fp8_grouped_gemm_wgrad(_ptr(A), A.stride(0), _ptr(sA), ld_sa, _ptr(B), B.stride(0), _ptr(sB),
                                        ld_sb, _ptr(D), _ptr(offsets), E, M, N, T, _stream(A)),
           "fp8_grouped_gemm_wgrad")


def fp8g_get_status(stream: torch.cuda.Stream | None = None) -> int:
    s = (stream or torch.cuda.current_stream()).cuda_stream
    return lib().fp8g_get_status(s)


def fp8g_last_config() -> dict:
    """Tile width, stages, grid, whether the tail was split (stream-K), whether the tiles were swapped
    (decode shapes: weight rows on the MMA's M) and the cluster size of a cluster K split (0: none) in
    this thread's last GEMM."""
    bn, st, gr, sp, sw = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    ck = ctypes.c_int()
    _check(lib().fp8g_last_config(ctypes.byref(bn), ctypes.byref(st), ctypes.byref(gr)), "fp8g_last_config")
    _check(lib().fp8g_last_split(ctypes.byref(sp)), "fp8g_last_split")
    _check(lib().fp8g_last_swap_ab(ctypes.byref(sw)), "fp8g_last_swap_ab")
    _check(lib().fp8g_last_cluster_k(ctypes.byref(ck)), "fp8g_last_cluster_k")
    return {"block_n": bn.value, "stages": st.value, "grid": gr.value, "split": bool(sp.value),
            "swap_ab": bool(sw.value), "cluster_k": ck.value}


# ------------------------------------------------------------------ allocating wrappers

def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def quantize_1x128(x: torch.Tensor, ld_sa: int | None = None):
    """bf16 [M,K] -> (q uint8 [M,K], sA f32 [K/128, ld_sa]); ld_sa defaults to round_up(M, 4)."""
    M, K = x.shape
    ld = ld_sa or max(round_up(M, 4), 4)
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sA = torch.zeros((K // 128, ld), dtype=torch.float32, device=x.device)
    fp8_quantize_1x128(x, q, sA)
    return q, sA


def route_capacity(T: int, topk: int, E: int) -> int:
    """Rows the routed layout may need: every group padded to 128 (T*topk + 127*E, rounded)."""
    return round_up(T * topk + 127 * E, 128)


def fp8_route_gather_quantize_1x128(x, topk_ids, E, q, sA, group_offsets, row_token, entry_row) -> None:
    """The routed layout into caller buffers: tokens x bf16 [T,K], topk_ids int32 [T,topk] ->
    q uint8 [M_cap,K], sA f32 [K/128, ld_sa >= M_cap], group_offsets int32 [E+1], row_token int32
    [M_cap], entry_row int32 [T,topk] (all on the device)."""
    _need(x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1, "x: bf16 [T,K], K contiguous")
    T, K = x.shape
    _need(topk_ids.dtype == torch.int32 and topk_ids.dim() == 2 and topk_ids.shape[0] == T
          and topk_ids.is_contiguous(), "topk_ids: int32 [T,topk] contiguous")
    topk = topk_ids.shape[1]
    m = q.shape[0]
    _need(_is_fp8(q) and q.dim() == 2 and q.shape[1] == K and q.stride(1) == 1, "q: e4m3 [M_cap,K]")
    _need(sA.dtype == torch.float32 and sA.dim() == 2 and sA.shape[0] == K // 128 and sA.stride(1) == 1
          and sA.shape[1] >= m, "sA: f32 [K/128, ld_sa >= M_cap]")
    _need(group_offsets.dtype == torch.int32 and group_offsets.numel() == E + 1, "group_offsets: int32 [E+1]")
    _need(row_token.dtype == torch.int32 and row_token.numel() == m, "row_token: int32 [M_cap]")
    _need(entry_row.dtype == torch.int32 and entry_row.shape == topk_ids.shape and entry_row.is_contiguous(),
          "entry_row: int32 [T,topk]")
    _on_one_device(x, topk_ids, q, sA, group_offsets, row_token, entry_row)
    _check(lib().fp8_route_gather_quantize_1x128(_ptr(x), T, K, x.stride(0), _ptr(topk_ids), topk, E, _ptr(q),
                                                 q.stride(0), _ptr(sA), sA.stride(0), _ptr(group_offsets),
                                                 _ptr(row_token), _ptr(entry_row), m, _stream(x)),
           "fp8_route_gather_quantize_1x128")


def route_gather_quantize_1x128(x: torch.Tensor, topk_ids: torch.Tensor, E: int, m_cap: int | None = None):
    """bf16 tokens [T,K] + int32 expert choices [T,topk] (device) -> (q uint8 [m_cap,K],
    sA f32 [K/128, m_cap], group_offsets int32 [E+1], row_token int32 [m_cap],
    entry_row int32 [T,topk]), all on the device: the contiguous grouped layout, quantised, and the
    row of each (token, slot) entry (-1: dropped).  m_cap defaults to route_capacity(T, topk, E)."""
    T, K = x.shape
    _need(topk_ids.dtype == torch.int32 and topk_ids.dim() == 2 and topk_ids.shape[0] == T
          and topk_ids.is_contiguous(), "topk_ids: int32 [T,topk] contiguous")
    topk = topk_ids.shape[1]
    m = m_cap or route_capacity(T, topk, E)
    q = torch.empty((m, K), dtype=torch.uint8, device=x.device)
    sA = torch.empty((K // 128, m), dtype=torch.float32, device=x.device)
    offs = torch.empty(E + 1, dtype=torch.int32, device=x.device)
    rows = torch.empty(m, dtype=torch.int32, device=x.device)
    entry = torch.empty((T, topk), dtype=torch.int32, device=x.device)
    _check(lib().fp8_route_gather_quantize_1x128(_ptr(x), T, K, x.stride(0), _ptr(topk_ids), topk, E, _ptr(q),
                                                 q.stride(0), _ptr(sA), m, _ptr(offs), _ptr(rows), _ptr(entry),
                                                 m, _stream(x)), "fp8_route_gather_quantize_1x128")
    return q, sA, offs, rows, entry


def quantize_128x128(w: torch.Tensor):
    """bf16 [N,K] or [E,N,K] -> (q uint8, sB f32 [(E,) ceil(N/128), K/128])."""
    N, K = w.shape[-2:]
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    sB = torch.empty((*w.shape[:-2], (N + 127) // 128, K // 128), dtype=torch.float32, device=w.device)
    fp8_quantize_128x128(w, q, sB)
    return q, sB


def gemm_nt(A, sA, B, sB) -> torch.Tensor:
    D = torch.empty((A.shape[0], B.shape[0]), dtype=torch.bfloat16, device=A.device)
    fp8_gemm_nt(A, sA, B, sB, D)
    return D


def quantize_per_row(x: torch.Tensor):
    """bf16 [M,K] -> (q uint8 [M,K], s f32 [M]): per-token (activations) or per-channel (weights)."""
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    s = torch.empty(x.shape[0], dtype=torch.float32, device=x.device)
    fp8_quantize_per_row(x, q, s)
    return q, s


def quantize_per_tensor(x: torch.Tensor):
    """bf16 [M,K] -> (q, s f32 [1]); bf16 [E,M,K] -> (q, s f32 [E]), one scale per tensor."""
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    s = torch.empty(1 if x.dim() == 2 else x.shape[0], dtype=torch.float32, device=x.device)
    fp8_quantize_per_tensor(x, q, s)
    return q, s


def quantize_1x128_e5m2(x: torch.Tensor, ld_sa: int | None = None):
    """bf16 [M,K] gradients -> (q uint8 e5m2 [M,K], sA f32 [K/128, ld_sa])."""
    M, K = x.shape
    ld = ld_sa or max(round_up(M, 4), 4)
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    sA = torch.zeros((K // 128, ld), dtype=torch.float32, device=x.device)
    fp8_quantize_1x128_e5m2(x, q, sA)
    return q, sA


def gemm_nt_scaled(A, sA, B, sB) -> torch.Tensor:
    D = torch.empty((A.shape[0], B.shape[0]), dtype=torch.bfloat16, device=A.device)
    fp8_gemm_nt_scaled(A, sA, B, sB, D)
    return D
