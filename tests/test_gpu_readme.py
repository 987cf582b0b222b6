"""The README's Python example runs as printed, and its grouped GEMM result matches the oracle
(sampled rows of every expert) at the GEMM tolerance."""

import pathlib
import re

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from gpu_util import assert_gemm_close, bf16_to_np, check_status, need_gpu, sa_from_device
from oracle import gemm_nt

README = pathlib.Path(__file__).resolve().parent.parent / "README.md"


def _u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).cpu().numpy()


@pytest.mark.gpu
def test_readme_example_runs_and_matches_the_oracle():
    need_gpu()
    blocks = re.findall(r"```python\n(.*?)```", README.read_text(encoding="utf-8"), re.S)
    assert len(blocks) == 1, "the README holds one Python example"
    torch.manual_seed(0)
    ns = {}
    exec(compile(blocks[0], str(README), "exec"), ns)  # noqa: S102 - the repository's own README
    torch.cuda.synchronize()
    check_status()
    qa, sa, qw, sw, D, offsets = (ns[k] for k in ("qa", "sa", "qw", "sw", "D", "offsets"))
    off = offsets.cpu().numpy().astype(np.int64)
    E = qw.shape[0]
    assert off.shape == (E + 1,) and off[0] == 0 and off[-1] <= qa.shape[0]
    qa_np, qw_np = _u8(qa), _u8(qw)
    sa_np = sa_from_device(sa, qa.shape[0])
    sw_np = sw.cpu().numpy()
    d_np = bf16_to_np(D)
    checked = 0
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 <= r0:
            continue
        rows = np.unique(np.array([r0, r0 + 1, (r0 + r1) // 2, r1 - 1]).clip(r0, r1 - 1))
        ref = gemm_nt(qa_np[rows], sa_np[rows], qw_np[e], sw_np[e])
        assert_gemm_close(d_np[rows], ref, f"README example, expert {e}")
        checked += 1
    assert checked == E
