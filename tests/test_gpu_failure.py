"""Failure detection on the GPU without a fault: the bounded waits every GEMM role uses run out of
budget against an mbarrier phase and a flag that nothing completes, record FP8G_ERR_TIMEOUT and
return; the context stays usable (a GEMM afterwards is correct and reports OK)."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from oracle import gemm_nt, quantize_128x128, quantize_1x128
from tests.gpu_util import assert_gemm_close, bf16_to_np, need_gpu, sa_to_device, u8

pytestmark = pytest.mark.gpu


def test_bounded_waits_run_out_and_the_context_stays_usable():
    need_gpu()
    assert g.fp8g_get_status() == 0
    out = torch.zeros(3, dtype=torch.int32, device="cuda")
    st = g.lib().fp8g_selftest_bounded_waits(2_000_000, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert g.fp8g_get_status() == 5  # FP8G_ERR_TIMEOUT, read and cleared
    assert out.tolist() == [1, 1, 1]  # both waits gave up and raised the abort flag
    assert g.fp8g_get_status() == 0
    # the context is intact: a GEMM runs and is correct
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((200, 512)) * 2).astype(np.float32)
    w = (rng.standard_normal((256, 512)) / 22).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    w = torch.from_numpy(w).to(torch.bfloat16).float().numpy()
    qa, sa = quantize_1x128(x)
    qb, sb = quantize_128x128(w)
    D = torch.empty((200, 256), dtype=torch.bfloat16, device="cuda")
    g.fp8_gemm_nt(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D)
    assert g.fp8g_get_status() == 0
    assert_gemm_close(bf16_to_np(D), gemm_nt(qa, sa, qb, sb), "GEMM after the timeouts")


_INJECTED = r"""
import os, sys, time
import numpy as np
import torch
sys.path.insert(0, os.environ["FP8G_REPO"])
import moe_grouped_gemm_block_gb300 as g
from oracle import gemm_nt, quantize_128x128, quantize_1x128
from tests.gpu_util import assert_gemm_close, bf16_to_np, sa_to_device, u8

rng = np.random.default_rng(5)
x = torch.from_numpy((rng.standard_normal((256, 1024)) * 2).astype(np.float32)).to(torch.bfloat16).float().numpy()
w = torch.from_numpy((rng.standard_normal((512, 1024)) / 32).astype(np.float32)).to(torch.bfloat16).float().numpy()
qa, sa = quantize_1x128(x)
qb, sb = quantize_128x128(w)
A, SA, B, SB = u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda()
ref = gemm_nt(qa, sa, qb, sb)
assert g.fp8g_get_status() == 0
# every CTA leaves its second operand stage unfilled: the issuer's wait for it runs out
os.environ["FP8G_TEST_SKIP_STAGE"] = "1"
D = torch.empty((256, 512), dtype=torch.bfloat16, device="cuda")
t0 = time.time()
g.fp8_gemm_nt(A, SA, B, SB, D)
torch.cuda.synchronize()  # the kernel returned: no role was left waiting
took = time.time() - t0
del os.environ["FP8G_TEST_SKIP_STAGE"]
st = g.fp8g_get_status()
assert st == 5, f"status {st}, expected FP8G_ERR_TIMEOUT"
assert g.fp8g_get_status() == 0
# the context stays usable: the same GEMM again, complete and correct
D2 = torch.empty((256, 512), dtype=torch.bfloat16, device="cuda")
g.fp8_gemm_nt(A, SA, B, SB, D2)
torch.cuda.synchronize()
assert g.fp8g_get_status() == 0
assert_gemm_close(bf16_to_np(D2), ref, "GEMM after the injected timeout")
print(f"INJECTED_TIMEOUT_OK {took:.3f}s")
"""


def test_gemm_wait_runs_out_inside_a_real_launch_and_the_context_stays_usable():
    # A real GEMM launch whose producer leaves one operand stage unfilled (a test hook, off unless
    # FP8G_TEST_SKIP_STAGE is set): the MMA issuer's bounded wait runs out, FP8G_ERR_TIMEOUT is
    # recorded, every role leaves its loop, the copies and MMAs already issued are awaited and TMEM
    # is freed.  Run in a child process so that the short wait budget (~10 ms; the budget is read
    # once per process) applies to it alone.
    need_gpu()
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, FP8G_REPO=root, FP8G_WAIT_BUDGET_CYCLES="20000000", FP8G_BLOCK_N="256")
    env.pop("FP8G_TEST_SKIP_STAGE", None)
    r = subprocess.run([sys.executable, "-c", _INJECTED], env=env, cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "INJECTED_TIMEOUT_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
