"""The quantiser's direct-path table (kDirectSafe0..3 in csrc/quantize.cu), checked without a GPU.

For an amax whose 8-bit bf16 significand A is marked, the kernel takes the e4m3 code of the single
product RN(x * RN(1/s)) instead of its bracketing test.  Here the committed words must (1) equal
what the independent generator next to the package computes, and (2) be exact against the oracle's
definition of the code, e4m3(RN(x / s)) (pages: "DeepGEMM explainer" sec. 3.1, quantisation by
division with s = amax / 448): every marked A agrees for every bf16 x with |x| <= amax, and every
unmarked A has at least one x where the product alone would be wrong."""

import os
import re

import numpy as np
import pytest

from oracle.e4m3 import e4m3_encode

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
QUANT_CU = os.path.join(ROOT, "moe_grouped_gemm_block_gb300", "csrc", "quantize.cu")


def committed_words():
    src = open(QUANT_CU).read()
    words = {int(i): int(v, 16) for i, v in re.findall(r"kDirectSafe(\d) = 0x([0-9A-Fa-f]+)u", src)}
    assert sorted(words) == [0, 1, 2, 3]
    return [words[i] for i in range(4)]


def marked(words, A):
    i = A - 128
    return (words[i >> 5] >> (i & 31)) & 1 == 1


def all_x(amax: np.float32) -> np.ndarray:
    X = np.arange(128, 256, dtype=np.float64) / 128.0
    x = np.concatenate([X * 2.0 ** -k for k in range(32)])
    x = x[x <= float(amax)].astype(np.float32)
    return np.concatenate([x, -x])


def test_committed_table_matches_the_generator():
    pytest.importorskip("torch")
    from moe_grouped_gemm_block_gb300.gen_quant_tables import mask_words, safe_significands
    assert committed_words() == mask_words(safe_significands())


def test_table_is_exact_against_the_oracle_for_every_significand():
    words = committed_words()
    n_marked = 0
    for A in range(128, 256):
        amax = np.float32(A / 128.0)
        s = np.float32(amax / np.float32(448.0))
        r = np.float32(np.float32(1.0) / s)
        x = all_x(amax)
        want = e4m3_encode((x / s).astype(np.float32))
        direct = e4m3_encode((x * r).astype(np.float32))
        agree = np.array_equal(want, direct)
        assert agree == marked(words, A), f"A={A}: table says {marked(words, A)}, oracle says {agree}"
        n_marked += agree
    assert n_marked == 102
