"""CPU oracle for the FP8 SwiGLU FFN block.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import or run anything in this package.  The CUDA library
(``transformer_ffn_block_gb300``) never imports it and shares no code with
it; the only code both sides use is the seeded input generator
``ffn_inputs``, which holds none of the block's arithmetic.

It is a plain, slow, float64 restatement of what the pages compute:

* ``codecs``  -- bf16 and OCP FP8 E4M3 codecs written from the format
  definitions (round to nearest even; E4M3 saturating at 448).
* ``ffn``     -- the prefill chain (fused residual + RMSNorm + abs-max,
  per-tensor quantisation, scaled FP8 GEMMs, SwiGLU with abs-max and
  requantisation), its recompute form with the activation abs-maxes given
  (``swiglu_forward_quant``, ``ffn_forward_recompute``), the generic
  quantise-then-matmul of the attention projections (``qmm``), the FP8 backward of
  the FFN (``swiglu_backward``, ``backward_qmm``, ``ffn_backward``), and the single-token
  decode FFN (dual row-scaled GEMV, silu_mul, down GEMV).

Every function is pinned by ``tests/test_oracle_*.py`` against hand-worked
values (``tests/golden/``), closed forms, invariants, library cross-checks
and brute-force exact arithmetic on tiny inputs (``tests/brute.py``).
"""
from .codecs import (E4M3_MAX, bf16_to_f32, bf16_to_f64, e4m3_decode, e4m3_encode,
                     e4m3_to_scaled_int, f32_to_bf16, f64_to_bf16)
from .ffn import (absmax, backward_qmm, decode_forward, ffn_backward, ffn_forward,
                  ffn_forward_recompute, fp8_gemm_scaled, fp8_gemm_scaled_acc, gemv_dual, gemv_row_scaled, quantize_rows, quantize_tensor,
                  quantize_with_abs_max, qmm, residual_rmsnorm_absmax, rmsnorm_f64, silu_f64,
                  silu_mul, swiglu, swiglu_backward, swiglu_forward_quant, swiglu_quant)

__all__ = [
    "E4M3_MAX", "bf16_to_f32", "bf16_to_f64", "e4m3_decode", "e4m3_encode",
    "e4m3_to_scaled_int", "f32_to_bf16", "f64_to_bf16", "absmax", "backward_qmm", "decode_forward",
    "ffn_backward", "ffn_forward", "ffn_forward_recompute", "fp8_gemm_scaled", "fp8_gemm_scaled_acc", "gemv_dual", "gemv_row_scaled", "quantize_rows",
    "quantize_tensor", "quantize_with_abs_max", "qmm", "residual_rmsnorm_absmax", "rmsnorm_f64",
    "silu_f64", "silu_mul", "swiglu", "swiglu_backward", "swiglu_forward_quant", "swiglu_quant",
]
