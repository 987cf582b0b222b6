"""Host-side logic without a GPU: the seeded workloads, the bench's FLOP accounting (pinned to the
H100 table the pages print), its clock-sample parsing, and the multi-rank timing reduction
(world size 2 over gloo)."""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
from moe_grouped_gemm_block_gb300.workloads import (WORKLOADS, Workload, gemm_flops, make_inputs,
                                                    small_variant)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "h100_gemm_table.txt")


def test_flop_accounting_reproduces_the_pages_h100_table():
    # "Production FP8 GEMM alignment and Tensor Core peak tuning", measurement table: TFLOPS = 2MNK / t
    rows = [line.split() for line in open(GOLDEN) if line.strip() and not line.startswith("#")]
    assert len(rows) == 4
    for name, M, N, K, t_ms, tflops in rows:
        w = Workload(name, "dense", M=int(M), N=int(N), K=int(K), seed=0)
        got = gemm_flops(w, {}) / (float(t_ms) * 1e-3) / 1e12
        assert abs(got - float(tflops)) / float(tflops) < 0.015, (name, got, tflops)


def test_dense_inputs_shapes_outliers_and_determinism():
    w = small_variant(WORKLOADS["decode"], M=16, N=256, K=1024)
    a = make_inputs(w, "cpu")
    b = make_inputs(w, "cpu")
    assert a["A"].dtype == torch.bfloat16 and a["A"].shape == (16, 1024) and a["B"].shape == (256, 1024)
    assert torch.equal(a["A"], b["A"]) and torch.equal(a["B"], b["B"])
    col_amax = a["A"].float().abs().amax(0)
    n_out = round(0.01 * 1024)
    assert (col_amax > 20).sum() >= n_out - 1  # the x50 outlier channels stand out
    assert abs(a["B"].float().std().item() - 1 / 32) < 0.005  # std = 1/sqrt(K)


def test_contiguous_layout_routing_and_padding():
    w = small_variant(WORKLOADS["moe_contiguous"], tokens=300, N=128, K=256)
    inp = make_inputs(w, "cpu")
    off = inp["group_offsets"].tolist()
    assert off[0] == 0 and all(o % 128 == 0 for o in off) and off == sorted(off)
    rt = inp["row_token"]
    assert inp["A"].shape[0] == off[-1] == rt.numel()
    valid = rt >= 0
    assert int(valid.sum()) == 300 * 2  # top-2: every token routed twice
    counts = torch.bincount(rt[valid], minlength=300)
    assert torch.all(counts == 2)
    for e in range(w.E):  # per expert: ascending tokens, then padding; padding rows are zero
        seg = rt[off[e]:off[e + 1]]
        toks = seg[seg >= 0]
        assert torch.all(toks[1:] > toks[:-1])
        assert torch.all(seg[toks.numel():] == -1)
    assert not inp["A"][~valid].float().any()


def test_masked_counts_in_range():
    w = WORKLOADS["moe_masked"]
    inp = make_inputs(small_variant(w, N=128, K=128, E=32, cap=256), "cpu")
    m = inp["masked_m"]
    assert m.dtype == torch.int32 and m.shape == (32,) and int(m.min()) >= 0 and int(m.max()) <= 256


def test_clock_sampler_parses_and_filters_to_the_window(tmp_path):
    p = tmp_path / "clk.csv"
    p.write_text("2026/12/02 10:00:00.000, 0, 1500, 2070, 500.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                 "2026/12/02 10:00:01.000, 0, 2070, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                 "2026/12/02 10:00:01.200, 0, 2050, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active\n")
    c = bench.ClockSampler(0)
    c.path = str(p)
    import datetime
    t0 = datetime.datetime(2026, 12, 2, 10, 0, 1).timestamp()
    c.mark(t0, t0 + 0.5)
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2060 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_env()
    dist = bench.maybe_init_pg(w)
    try:
        bench.barrier(dist)
        q.put((r, bench.max_over_ranks(1.5 + r, dist)))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_multi_rank_timing_takes_the_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_source_digest_ignores_comments_and_layout_only():
    import bench
    a = 'int x = 1; // note\n/* block\n  comment */ const char* s = "a // b";\n'
    b = 'int  x = 1;\n\n// another note\nconst char* s = "a // b"; /* more */\n'
    c = 'int x = 2; const char* s = "a // b";'
    d = 'int x = 1; const char* s = "a /* b";'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only(a) != bench._code_only(d)  # string contents are code


def test_reference_arm_prints_the_contract_line():
    # `bench.py --impl reference` times the oracle on the host cores; its line carries the contract's
    # keys, the reference marker, and describes the sample it timed
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1", "--workloads", "tiny,decode"], capture_output=True, text=True, cwd=root,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    for key in ("metric", "unit", "n_gpus", "ms_per_step", "higher_is_better", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["cpu_baseline"]["kind"] == "oracle" and "rows" in line["cpu_baseline"]["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0
