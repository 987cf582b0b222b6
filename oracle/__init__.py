"""CPU oracle for the FP8 block-scaled GEMM path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy code that says what the path computes.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import it.  The library (``moe_grouped_gemm_block_gb300``)
never imports it and shares no code, table or constant generator with it.

Pages followed (cited by title and section):
  [WT] "DeepGEMM FP8 walk-through" (m.czchanglian.com/news/60438)
  [PT] "Production FP8 GEMM alignment and Tensor Core peak tuning" (gtnt.cn/news/117510)
  [EX] "DeepGEMM explainer" (nxmr.cn/news/131680)

Modules:
  e4m3      -- the e4m3 (OCP "fn") codec written from the format's closed form
  quantize  -- 1x128 activation and 128x128 weight block quantisation
  gemm      -- the blockwise-dequantised GEMM with per-K-block promotion, and its
               contiguous / masked grouped MoE forms
  route     -- the contiguous grouped layout built from routed tokens, gathered and quantised
  scaled    -- per-tensor / per-token / per-channel quantisation and the GEMM that applies
               those scales once, in the epilogue, with its grouped forms
  e5m2      -- the e5m2 (OCP "E5M2") codec for gradients
  backward  -- 1x128 e5m2 gradient quantisation, the data-gradient GEMM (e5m2 x e4m3) and the
               K-grouped weight-gradient GEMM of a grouped MoE layer
Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
invariants, brute force on tiny inputs and library routines; none is "parity
unpinned".
"""

from .e4m3 import E4M3_MAX, e4m3_decode, e4m3_decode_table, e4m3_encode, bf16_round_bits, bf16_bits_to_f32
from .quantize import quantize_1x128, quantize_128x128
from .gemm import gemm_nt, grouped_contiguous, grouped_masked
from .route import route_gather_quantize, route_layout
from .backward import block_products, gemm_nt_dgrad, quantize_1x128_e5m2, wgrad_k_grouped
from .e5m2 import E5M2_MAX, e5m2_decode, e5m2_encode
from .scaled import (gemm_nt_scaled, grouped_contiguous_scaled, grouped_masked_scaled, quantize_per_row,
                     quantize_per_tensor)

__all__ = [
    "E4M3_MAX", "e4m3_decode", "e4m3_decode_table", "e4m3_encode", "bf16_round_bits",
    "bf16_bits_to_f32", "quantize_1x128", "quantize_128x128", "gemm_nt", "grouped_contiguous",
    "grouped_masked", "route_gather_quantize", "route_layout", "gemm_nt_scaled",
    "grouped_contiguous_scaled", "grouped_masked_scaled", "quantize_per_row", "quantize_per_tensor",
    "E5M2_MAX", "e5m2_decode", "e5m2_encode", "block_products", "gemm_nt_dgrad", "quantize_1x128_e5m2",
    "wgrad_k_grouped",
]
