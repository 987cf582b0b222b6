"""Helpers shared by the GPU parity tests: layout conversion between the oracle's
arrays and the library's device tensors, and the GEMM tolerance check.

GEMM tolerance (per element and overall), on the same seeded inputs:
    |gpu - ref| <= 8e-3 * |ref| + 1e-2 * rms(ref)      and      ||gpu - ref||_F / ||ref||_F <= 2e-3
Quantisation is compared bit for bit.
"""

import os

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from oracle import bf16_bits_to_f32

REL_ELEM, ABS_RMS, REL_FRO = 8e-3, 1e-2, 2e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    major, minor = torch.cuda.get_device_capability()
    if (major, minor) != (10, 3):
        pytest.skip(f"needs sm_103 (found sm_{major}{minor})")


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> float32 numpy (exact)."""
    return t.detach().float().cpu().numpy()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def sa_to_device(sa: np.ndarray, ld_sa: int | None = None) -> torch.Tensor:
    """oracle layout [M, KB] -> library layout [KB, ld_sa] on the GPU."""
    M, KB = sa.shape
    ld = ld_sa or max((M + 3) // 4 * 4, 4)
    out = np.zeros((KB, ld), dtype=np.float32)
    out[:, :M] = sa.T
    return torch.from_numpy(out).cuda()


def sa_from_device(sA: torch.Tensor, M: int) -> np.ndarray:
    """library layout [KB, ld_sa] -> oracle layout [M, KB]."""
    return sA[:, :M].cpu().numpy().T.copy()


def u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_gemm_close(gpu: np.ndarray, ref_bits: np.ndarray, what: str = ""):
    ref = bf16_bits_to_f32(ref_bits).astype(np.float64)
    got = np.asarray(gpu, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = REL_ELEM * np.abs(ref) + ABS_RMS * rms
    bad = err > bound
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"worst at {np.unravel_index(np.argmax(err - bound), err.shape)}: "
                           f"got {got.flat[np.argmax(err - bound)]} ref {ref.flat[np.argmax(err - bound)]}")
    assert fro <= REL_FRO, f"{what}: relative Frobenius error {fro:.3e}"
    return {"max_abs": float(err.max(initial=0)), "fro": float(fro), "exact": float(np.mean(err == 0))}


class env_var:
    """Set (or, with None, clear) one environment variable inside the block."""

    def __init__(self, name, value):
        self.name, self.value = name, value

    def __enter__(self):
        self.old = os.environ.get(self.name)
        if self.value is None:
            os.environ.pop(self.name, None)
        else:
            os.environ[self.name] = str(self.value)

    def __exit__(self, *exc):
        if self.old is None:
            os.environ.pop(self.name, None)
        else:
            os.environ[self.name] = self.old


def block_n(bn):
    """Force the tile width of the GEMM calls inside the block (FP8G_BLOCK_N)."""
    return env_var("FP8G_BLOCK_N", bn or None)


def pair(mode):
    """CTA pairs inside the block (FP8G_PAIR): 0 / False off, 1 / True 256 x 256 pair tiles,
    2 for 256 x 128 pair tiles."""
    return env_var("FP8G_PAIR", int(mode) if mode else None)


def check_status():
    st = g.fp8g_get_status()
    assert st == 0, g.STATUS.get(st, st)
