"""Generator of the quantiser's direct-path table (build helper; its output is pasted into
csrc/quantize.cu as kDirectMode0..7 and a CPU test checks the two agree).

The quantisers compute e4m3(RN(x / s)) with s = RN(amax / 448).  For most blocks a single product
y = RN(x * r) with a fixed multiplier r already has the same e4m3 code for every bf16 x with
|x| <= amax, so the kernel can skip its bracketing test.  Whether a given r works depends only on
amax's 8-bit bf16 significand A: s, 1/s, the products and the codes all scale exactly with a
power-of-two change of amax and x (while s is a normal float; subnormal s takes the division path
anyway), and so does r moved by whole ulps.  This script enumerates, for each A in 128..255, every
x = +-X * 2^-k (X in 128..255, k >= 0, |x| <= amax, down to where the codes are 0) and records the
first multiplier that gives no different code: mode 1 for RN(1/s), 2 for RN(1/s) one ulp up, 3 for
one ulp down; mode 0 when none does (the block keeps the bracketing test).

Arithmetic: IEEE binary32 in numpy (division, reciprocal and products rounded to nearest even)
and PyTorch's float8_e4m3fn cast for the e4m3 code (round to nearest even; every quotient here is
at most 448 * (1 + 2^-23), which rounds to 448).
"""

import numpy as np
import torch

ULP_STEP = {1: 0, 2: 1, 3: -1}  # mode -> ulps added to RN(1/s)


def e4m3_codes(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def all_x(amax: np.float32) -> np.ndarray:
    X = np.arange(128, 256, dtype=np.float64) / 128.0
    x = np.concatenate([X * 2.0 ** -k for k in range(32)])
    x = x[x <= float(amax)].astype(np.float32)
    return np.concatenate([x, -x])


def step_ulps(r: np.float32, d: int) -> np.float32:
    return (np.array([r], dtype=np.float32).view(np.uint32).astype(np.int64) + d).astype(np.uint32).view(
        np.float32)[0]


def direct_modes() -> list[int]:
    """Mode of each significand A = 128..255 (index A - 128)."""
    f32 = np.float32
    modes = []
    for A in range(128, 256):
        amax = f32(A / 128.0)
        s = f32(amax / f32(448.0))
        r = f32(f32(1.0) / s)
        x = all_x(amax)
        want = e4m3_codes((x / s).astype(np.float32))  # RN(x / s)
        mode = 0
        for m in (1, 2, 3):
            if np.array_equal(want, e4m3_codes((x * step_ulps(r, ULP_STEP[m])).astype(np.float32))):
                mode = m
                break
        modes.append(mode)
    return modes


def mode_words(modes: list[int]) -> list[int]:
    """2 bits per significand, 16 per 32-bit word: bits 2(i % 16) .. of word i // 16, i = A - 128."""
    w = [0] * 8
    for i, m in enumerate(modes):
        w[i >> 4] |= m << (2 * (i & 15))
    return w


if __name__ == "__main__":
    words = mode_words(direct_modes())
    print(", ".join(f"kDirectMode{i} = 0x{v:08X}u" for i, v in enumerate(words)))
