"""The README's usage example runs as written, and its grouped GEMM matches the oracle on sampled rows."""

import os
import re

import numpy as np
import pytest
import torch

from oracle import gemm_nt, quantize_128x128, quantize_1x128
from tests.gpu_util import assert_gemm_close, bf16_to_np, need_gpu

pytestmark = pytest.mark.gpu
README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def test_readme_example():
    need_gpu()
    code = re.search(r"```python\n(.*?)```", open(README).read(), re.S).group(1)
    ns = {}
    exec(compile(code, "README.md", "exec"), ns)  # noqa: S102 -- the repository's own example
    x, w, D, offsets, row_token = ns["x"], ns["w"], ns["D"], ns["offsets"], ns["row_token"]
    offs = offsets.cpu().numpy()
    rows = row_token.cpu().numpy()
    e = 3
    r0, r1 = int(offs[e]), int(offs[e + 1])
    pick = np.arange(r0, r1)[:: max(1, (r1 - r0) // 16)][:16]  # sampled rows of expert 3
    pick = pick[rows[pick] >= 0]
    cols = np.r_[0:128, 2048:2176]
    qa, sa = quantize_1x128(x[torch.from_numpy(rows[pick]).long().cuda()].float().cpu().numpy())
    # the two 128-row weight blocks those columns lie in (blocks 0 and 16), quantised on their own
    wb = w[e].float().cpu().numpy()
    q0, s0 = quantize_128x128(wb[0:128])
    q1, s1 = quantize_128x128(wb[2048:2176])
    sb = np.zeros((w.shape[1] // 128, s0.shape[1]), np.float32)
    sb[0], sb[16] = s0[0], s1[0]
    ref = gemm_nt(qa, sa, np.concatenate([q0, q1]), sb, n_index=cols)
    assert_gemm_close(bf16_to_np(D)[pick][:, cols], ref, "README example, expert 3")
