"""Seeded synthetic workloads for the FP8 block-scaled GEMM path.

This module only draws random inputs and lays them out; it holds none of the
method's arithmetic (no quantisation, no GEMM).  Both the CPU oracle (tests,
CPU baseline) and the CUDA path (tests, bench) take their inputs from here.

Shapes and distributions follow the workloads the pages discuss:
  * dense shapes, including the M=4096, N=8192, K=8192 case of the H100 table on
    "Production FP8 GEMM alignment and Tensor Core peak tuning" (timing table);
  * a decode shape with a small M ("DeepGEMM FP8 walk-through", sec. 1.2);
  * MoE grouped GEMMs where each expert gets a different number of tokens
    ("DeepGEMM explainer", sec. 3.2; walk-through sec. 5.3), in a contiguous
    layout (each expert's rows padded to 128) and a masked layout (fixed
    capacity per expert, a per-expert count of valid rows).

Recipe (all draws from one ``torch.Generator`` seeded per workload, in the
order A, B, outlier columns, routing/counts):
  * A ~ N(0, 1) in fp32; for the large shapes round(0.01*K) K-columns chosen by
    a seeded permutation are multiplied by 50 (outlier channels); cast to bf16
    with round-to-nearest-even.
  * B ~ N(0, std) with std = 1/sqrt(K) (std = 1 for the tiny case); bf16.
  * contiguous MoE: router logits [T, E] ~ N(0, 1), softmax, top-2 experts per
    token (the lower index wins ties); each expert's routed rows are gathered in
    ascending token order and zero-padded to a multiple of 128 rows.
  * masked MoE: valid rows per expert ~ Uniform{0..cap}; every row of A filled.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BLOCK = 128  # the scaling block edge (1x128 activations, 128x128 weights)


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "dense" | "contiguous" | "masked"
    N: int
    K: int
    seed: int
    M: int = 0  # dense rows
    E: int = 1  # experts
    tokens: int = 0  # contiguous: tokens routed
    topk: int = 0  # contiguous: experts per token
    cap: int = 0  # masked: rows per expert
    outliers: bool = False
    b_std_one: bool = False  # B ~ N(0,1) instead of N(0, 1/sqrt(K))
    extra: dict = field(default_factory=dict, compare=False)


# The workloads: a tiny dense case, a decode shape, two large dense shapes (4096^3 and the
# 4096 x 8192 x 8192 shape of the H100 table), and the two MoE layouts.
WORKLOADS = {
    "tiny": Workload("tiny", "dense", M=128, N=256, K=512, seed=0, b_std_one=True),
    "decode": Workload("decode", "dense", M=64, N=7168, K=7168, seed=1, outliers=True),
    "large_4096": Workload("large_4096", "dense", M=4096, N=4096, K=4096, seed=2, outliers=True),
    "large_4096x8192": Workload("large_4096x8192", "dense", M=4096, N=8192, K=8192, seed=2,
                                outliers=True),
    "moe_contiguous": Workload("moe_contiguous", "contiguous", N=4096, K=7168, E=8, tokens=4096,
                               topk=2, seed=3),
    "moe_masked": Workload("moe_masked", "masked", N=4096, K=7168, E=32, cap=256, seed=4),
}


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _apply_outliers(a32: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    K = a32.shape[-1]
    n_out = int(round(0.01 * K))
    cols = torch.randperm(K, generator=g, device=g.device)[:n_out]
    a32[..., cols] *= 50.0
    return a32


def _weights(w: Workload, g, device) -> torch.Tensor:
    std = 1.0 if w.b_std_one else 1.0 / math.sqrt(w.K)
    if w.E == 1 and w.kind == "dense":
        return _normal((w.N, w.K), std, g, device).to(torch.bfloat16)
    # one expert at a time keeps the fp32 temporary small
    out = torch.empty((w.E, w.N, w.K), dtype=torch.bfloat16, device=device)
    for e in range(w.E):
        out[e] = _normal((w.N, w.K), std, g, device).to(torch.bfloat16)
    return out


def route_top2(logits: torch.Tensor, topk: int):
    """Top-k expert choice per token from softmax(logits); ties -> lower index.

    Returns (expert_of_pair [T*topk], token_of_pair [T*topk]) in token-major order.
    """
    probs = torch.softmax(logits.double(), dim=-1)
    T, E = probs.shape
    # stable descending sort: equal probabilities keep ascending expert order
    order = torch.sort(-probs, dim=-1, stable=True).indices[:, :topk]
    tok = torch.arange(T).unsqueeze(1).expand(T, topk)
    return order.reshape(-1), tok.reshape(-1)


def contiguous_layout(expert_of_pair: torch.Tensor, token_of_pair: torch.Tensor, E: int):
    """Row order of the contiguous grouped layout.

    Each expert's rows hold its routed tokens in ascending token order; each
    group is padded with empty rows to a multiple of 128.  Returns
    (row_token [M_total] with -1 for padding rows, group_offsets [E+1] int32).
    """
    rows = []
    offsets = [0]
    for e in range(E):
        toks = torch.sort(token_of_pair[expert_of_pair == e]).values
        padded = round_up(int(toks.numel()), BLOCK)
        pad = torch.full((padded - toks.numel(),), -1, dtype=torch.int64)
        rows.append(torch.cat([toks.to(torch.int64), pad]))
        offsets.append(offsets[-1] + padded)
    return torch.cat(rows), torch.tensor(offsets, dtype=torch.int32)


def make_inputs(w: Workload, device="cpu") -> dict:
    """Draw the bf16 inputs of workload ``w`` on ``device``.

    Keys: "A" (bf16, [M,K] / [M_total,K] / [E,cap,K]), "B" (bf16 [N,K] or
    [E,N,K]); contiguous adds "group_offsets" (int32 [E+1], CPU), "row_token",
    and the unrouted "tokens" (bf16 [T,K]) with their "topk_ids" (int32 [T,topk],
    CPU); masked adds "masked_m" (int32 [E], CPU).
    """
    device = torch.device(device)
    g = _gen(w.seed, device)
    out = {}
    if w.kind == "dense":
        a32 = _normal((w.M, w.K), 1.0, g, device)
        B = _weights(w, g, device)
        if w.outliers:
            a32 = _apply_outliers(a32, g)
        out["A"] = a32.to(torch.bfloat16)
        out["B"] = B
    elif w.kind == "contiguous":
        x32 = _normal((w.tokens, w.K), 1.0, g, device)
        B = _weights(w, g, device)
        if w.outliers:
            x32 = _apply_outliers(x32, g)
        x = x32.to(torch.bfloat16)
        gr = _gen(w.seed + 1000, "cpu")  # routing is small: always on the host
        logits = torch.randn((w.tokens, w.E), generator=gr, dtype=torch.float32)
        exp_of, tok_of = route_top2(logits, w.topk)
        row_token, offsets = contiguous_layout(exp_of, tok_of, w.E)
        A = torch.zeros((row_token.numel(), w.K), dtype=torch.bfloat16, device=device)
        valid = (row_token >= 0).nonzero().squeeze(1)
        A[valid.to(device)] = x[row_token[valid].to(device)]
        out.update(A=A, B=B, group_offsets=offsets, row_token=row_token, tokens=x,
                   topk_ids=exp_of.reshape(w.tokens, w.topk).to(torch.int32))
    elif w.kind == "masked":
        a32 = _normal((w.E, w.cap, w.K), 1.0, g, device)
        B = _weights(w, g, device)
        if w.outliers:
            a32 = _apply_outliers(a32, g)
        gm = _gen(w.seed + 2000, "cpu")
        masked_m = torch.randint(0, w.cap + 1, (w.E,), generator=gm, dtype=torch.int32)
        out.update(A=a32.to(torch.bfloat16), B=B, masked_m=masked_m)
    else:
        raise ValueError(w.kind)
    return out


def small_variant(w: Workload, **over) -> Workload:
    """A copy of ``w`` with some fields replaced (for reduced-size test cases)."""
    d = {k: getattr(w, k) for k in w.__dataclass_fields__ if k != "extra"}
    d.update(over)
    return Workload(**d)


def gemm_flops(w: Workload, inputs: dict) -> float:
    """Algorithmic FLOPs (2*M*N*K over valid rows only)."""
    if w.kind == "dense":
        return 2.0 * w.M * w.N * w.K
    if w.kind == "contiguous":
        return 2.0 * w.tokens * w.topk * w.N * w.K
    m = int(inputs["masked_m"].sum())
    return 2.0 * m * w.N * w.K
