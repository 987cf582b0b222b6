"""The 1x128 quantisers compute the block scale s = RN(amax / c) (c = 448 for e4m3, 57344 for e5m2)
without a division: q = RN(amax * RN(1/c)), then the nearest of q and its two fp32 neighbours by
the residual amax - c * q' (exact in one FMA).  This checks that method, written out here in numpy,
against the IEEE fp32 quotient for every bf16 significand at every exponent whose scale is a
normal number (subnormal scales take the division in the kernel).  The GPU tests then check the
kernel's scales bit for bit against the oracle."""

import numpy as np
import pytest

TINY = np.float32(1.17549435e-38)  # smallest normal fp32


def scale_by_multiply(a: np.float32, c: float) -> np.float32:
    r = np.float32(1.0) / np.float32(c)
    q = np.float32(a * r)
    bits = np.array(q).view(np.uint32)
    best, best_res = q, None
    for d in (0, -1, 1):  # q, then its lower and upper neighbour
        cand = np.array(np.uint32(int(bits) + d)).view(np.float32)
        # the residual in float64 is exact here (27 significant bits at most)
        res = abs(float(a) - float(c) * float(cand))
        if best_res is None or res < best_res:
            best, best_res = cand, res
    return np.float32(best)


@pytest.mark.parametrize("c", [448.0, 57344.0])
def test_multiply_with_residual_choice_equals_the_division(c):
    checked = 0
    for A in range(128, 256):  # bf16 significand (8 bits with the hidden one)
        for e in range(-140, 120):
            a = np.float32(np.ldexp(float(A), e))
            if not np.isfinite(a):
                continue
            ref = np.float32(a / np.float32(c))
            if not ref >= TINY:
                continue
            assert scale_by_multiply(a, c) == ref, (A, e)
            checked += 1
    assert checked > 25000


def test_a_plain_multiply_is_not_enough():
    # the residual step is needed: one multiply by RN(1/448) misses RN(a / 448) for many amax
    r = np.float32(1.0) / np.float32(448.0)
    misses = sum(np.float32(np.float32(A) * r) != np.float32(np.float32(A) / np.float32(448.0)) for A in range(128, 256))
    assert misses > 0
