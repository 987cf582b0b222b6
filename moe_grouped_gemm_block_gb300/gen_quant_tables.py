"""Generator of the quantiser's direct-path table (build helper; its output is pasted into
csrc/quantize.cu as kDirectSafe0..3 and a CPU test checks the two agree).

The quantisers compute e4m3(RN(x / s)) with s = RN(amax / 448).  For most blocks the product
y = RN(x * RN(1/s)) already has the same e4m3 code for every bf16 x with |x| <= amax, so the
kernel can skip its bracketing test.  Whether that holds depends only on amax's 8-bit bf16
significand A: s, 1/s, the products and the codes all scale exactly with a power-of-two change of
amax and x (while s is a normal float; subnormal s takes the division path anyway).  This script
enumerates, for each A in 128..255, every x = +-X * 2^-k (X in 128..255, k >= 0, |x| <= amax, down
to where both codes are 0) and marks A "safe" when no x gives different codes.

Arithmetic: IEEE binary32 in numpy (division, reciprocal and products rounded to nearest even)
and PyTorch's float8_e4m3fn cast for the e4m3 code (round to nearest even; every quotient here is
at most 448 * (1 + 2^-23), which rounds to 448).
"""

import numpy as np
import torch


def e4m3_codes(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def safe_significands() -> list[int]:
    f32 = np.float32
    X = np.arange(128, 256, dtype=np.float64) / 128.0
    safe = []
    for A in range(128, 256):
        amax = f32(A / 128.0)
        s = f32(amax / f32(448.0))
        r = f32(f32(1.0) / s)
        x = np.concatenate([X * 2.0 ** -k for k in range(32)])
        x = x[x <= float(amax)].astype(np.float32)
        x = np.concatenate([x, -x])
        exact = (x / s).astype(np.float32)     # RN(x / s)
        direct = (x * r).astype(np.float32)    # RN(x * RN(1 / s))
        if np.array_equal(e4m3_codes(exact), e4m3_codes(direct)):
            safe.append(A)
    return safe


def mask_words(safe: list[int]) -> list[int]:
    """Bit (A - 128) of the 128-bit mask, as four 32-bit words (word 0 holds A = 128..159)."""
    w = [0, 0, 0, 0]
    for A in safe:
        i = A - 128
        w[i >> 5] |= 1 << (i & 31)
    return w


if __name__ == "__main__":
    words = mask_words(safe_significands())
    print(", ".join(f"kDirectSafe{i} = 0x{v:08X}u" for i, v in enumerate(words)))
