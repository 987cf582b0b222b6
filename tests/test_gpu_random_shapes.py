"""Seeded random shapes for the GEMM forms against the oracle: ragged M and N, K from one to a dozen
blocks, forced or chosen tile widths, the stream-K tail on or off, and for the grouped forms random
group sizes (empty groups included).  Each case is drawn from its own seed, so a failure names a
reproducible shape."""

import numpy as np
import pytest
import torch

import moe_grouped_gemm_block_gb300 as g
from oracle import gemm_nt, grouped_contiguous, grouped_masked, quantize_128x128, quantize_1x128
from oracle.backward import gemm_nt_dgrad, quantize_1x128_e5m2
from oracle.scaled import gemm_nt_scaled, quantize_per_row, quantize_per_tensor
from tests.gpu_util import assert_gemm_close, bf16_to_np, block_n, check_status, env_var, need_gpu, sa_to_device, u8

pytestmark = pytest.mark.gpu
SENTINEL = 0x7FC1
FORMS = ["dense", "contiguous", "masked", "scaled", "dgrad"]


def _draw(rng, shape, std=1.0):
    x = torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32))
    return x.to(torch.bfloat16).float().numpy()


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    form = FORMS[seed % len(FORMS)]
    return dict(rng=rng, form=form, M=int(rng.integers(1, 400)), N=int(rng.integers(1, 33)) * 16,
                K=int(rng.integers(1, 13)) * 128, bn=[None, 64, 128, 256][int(rng.integers(0, 4))],
                streamk=bool(rng.integers(0, 2)))


@pytest.mark.parametrize("seed", range(24))
def test_random_shape(seed):
    need_gpu()
    c = _case(seed)
    rng, form, M, N, K, bn = c["rng"], c["form"], c["M"], c["N"], c["K"], c["bn"]
    tag = f"seed={seed} {form} M={M} N={N} K={K} bn={bn} streamk={c['streamk']}"
    with env_var("FP8G_STREAMK", None if c["streamk"] else 0), block_n(bn):
        if form in ("dense", "dgrad"):
            x = _draw(rng, (M, K), 1e-3 if form == "dgrad" else 2.0)
            qa, sa = quantize_1x128_e5m2(x) if form == "dgrad" else quantize_1x128(x)
            qb, sb = quantize_128x128(_draw(rng, (N, K), 1 / np.sqrt(K)))
            D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            call = g.fp8_gemm_nt_dgrad if form == "dgrad" else g.fp8_gemm_nt
            call(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D)
            torch.cuda.synchronize()
            check_status()
            ref = gemm_nt_dgrad(qa, sa, qb, sb) if form == "dgrad" else gemm_nt(qa, sa, qb, sb)
            assert_gemm_close(bf16_to_np(D), ref, tag)
        elif form == "scaled":
            per_row, per_col = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
            xa, xb = _draw(rng, (M, K), 2.0), _draw(rng, (N, K), 1 / np.sqrt(K))
            qa, sa = quantize_per_row(xa) if per_row else quantize_per_tensor(xa)
            qb, sb = quantize_per_row(xb) if per_col else quantize_per_tensor(xb)
            D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            g.fp8_gemm_nt_scaled(u8(qa), torch.from_numpy(sa).cuda(), u8(qb), torch.from_numpy(sb).cuda(), D)
            torch.cuda.synchronize()
            check_status()
            assert_gemm_close(bf16_to_np(D), gemm_nt_scaled(qa, sa, qb, sb), tag)
        elif form == "contiguous":
            E = int(rng.integers(1, 7))
            sizes = rng.integers(0, 3, E) * 128  # 0, 128 or 256 rows per group
            off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
            M_total = int(off[-1]) + 128 * int(rng.integers(0, 2))  # maybe a block in no group
            M_total = max(M_total, 128)  # every group empty: one block in no group
            qa, sa = quantize_1x128(_draw(rng, (M_total, K)))
            w = _draw(rng, (E * N, K), 1 / np.sqrt(K)).reshape(E, N, K)
            qs, ss = zip(*(quantize_128x128(w[e]) for e in range(E)))
            qb, sb = np.stack(qs), np.stack(ss)
            D = torch.empty((M_total, N), dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
            g.fp8_grouped_gemm_contiguous(u8(qa), sa_to_device(sa), u8(qb), torch.from_numpy(sb).cuda(), D,
                                          torch.from_numpy(off).cuda())
            torch.cuda.synchronize()
            check_status()
            ref = grouped_contiguous(qa, sa, qb, sb, off, np.full((M_total, N), SENTINEL, np.uint16))
            last = int(off[-1])
            assert np.all(D.view(torch.int16).cpu().numpy().view(np.uint16)[last:] == SENTINEL), tag
            if last:
                assert_gemm_close(bf16_to_np(D)[:last], ref[:last], tag)
        else:  # masked
            E, cap = int(rng.integers(1, 6)), int(rng.integers(1, 17)) * 16
            masked = rng.integers(0, cap + 1, E).astype(np.int32)
            qa, sa = quantize_1x128(_draw(rng, (E * cap, K)))
            w = _draw(rng, (E * N, K), 1 / np.sqrt(K)).reshape(E, N, K)
            qs, ss = zip(*(quantize_128x128(w[e]) for e in range(E)))
            qb, sb = np.stack(qs), np.stack(ss)
            D = torch.empty((E, cap, N), dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
            g.fp8_grouped_gemm_masked(u8(qa.reshape(E, cap, K)), sa_to_device(sa), u8(qb),
                                      torch.from_numpy(sb).cuda(), D, torch.from_numpy(masked).cuda())
            torch.cuda.synchronize()
            check_status()
            ref = grouped_masked(qa.reshape(E, cap, K), sa.reshape(E, cap, -1), qb, sb, masked,
                                 np.full((E, cap, N), SENTINEL, np.uint16))
            valid = np.arange(cap)[None, :] < masked[:, None]
            assert np.all(D.view(torch.int16).cpu().numpy().view(np.uint16)[~valid] == SENTINEL), tag
            if valid.any():
                assert_gemm_close(bf16_to_np(D)[valid], ref[valid], tag)
