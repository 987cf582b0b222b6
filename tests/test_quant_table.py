"""The quantiser's direct-path table (kDirectMode0..7 in csrc/quantize.cu), checked without a GPU.

For an amax whose 8-bit bf16 significand A has a non-zero mode, the kernel takes the e4m3 code of the
single product RN(x * r) instead of its bracketing test, with r = RN(1/s) (mode 1), one ulp above
(mode 2) or one ulp below (mode 3).  Here the committed words must (1) equal what the independent
generator next to the package computes, and (2) be exact against the oracle's definition of the
code, e4m3(RN(x / s)) (pages: "DeepGEMM explainer" sec. 3.1, quantisation by division with
s = amax / 448): for every A with a mode, its multiplier agrees for every bf16 x with |x| <= amax;
for every A with mode 1, 2 or 3, no earlier mode works; and every A with mode 0 has, for each of
the three multipliers, at least one x where the product alone would be wrong."""

import os
import re

import numpy as np
import pytest

from oracle.e4m3 import e4m3_encode

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
QUANT_CU = os.path.join(ROOT, "moe_grouped_gemm_block_gb300", "csrc", "quantize.cu")
STEP = {1: 0, 2: 1, 3: -1}


def committed_words():
    src = open(QUANT_CU).read()
    words = {int(i): int(v, 16) for i, v in re.findall(r"kDirectMode(\d) = 0x([0-9A-Fa-f]+)u", src)}
    assert sorted(words) == list(range(8))
    return [words[i] for i in range(8)]


def mode_of(words, A):
    i = A - 128
    return (words[i >> 4] >> (2 * (i & 15))) & 3


def all_x(amax: np.float32) -> np.ndarray:
    X = np.arange(128, 256, dtype=np.float64) / 128.0
    x = np.concatenate([X * 2.0 ** -k for k in range(32)])
    x = x[x <= float(amax)].astype(np.float32)
    return np.concatenate([x, -x])


def moved(r, d):
    return (np.array([r], np.float32).view(np.uint32).astype(np.int64) + d).astype(np.uint32).view(np.float32)[0]


def test_committed_table_matches_the_generator():
    pytest.importorskip("torch")
    from moe_grouped_gemm_block_gb300.gen_quant_tables import direct_modes, mode_words
    assert committed_words() == mode_words(direct_modes())


def test_table_is_exact_against_the_oracle_for_every_significand():
    words = committed_words()
    counts = [0, 0, 0, 0]
    for A in range(128, 256):
        amax = np.float32(A / 128.0)
        s = np.float32(amax / np.float32(448.0))
        r = np.float32(np.float32(1.0) / s)
        x = all_x(amax)
        want = e4m3_encode((x / s).astype(np.float32))
        works = {m: np.array_equal(want, e4m3_encode((x * moved(r, STEP[m])).astype(np.float32))) for m in STEP}
        m = mode_of(words, A)
        counts[m] += 1
        if m:
            assert works[m], f"A={A}: mode {m} is not exact"
            assert not any(works[k] for k in STEP if k < m), f"A={A}: an earlier mode works"
        else:
            assert not any(works.values()), f"A={A}: marked for the bracket, yet a multiplier works"
    assert counts == [7, 102, 15, 4]
