"""CPU oracle for the FP8 SwiGLU FFN block.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import or run anything in this package.  The CUDA library
(``transformer_ffn_block_gb300``) never imports it and shares no code with
it; the only code both sides use is the seeded input generator
``ffn_inputs``, which holds none of the block's arithmetic.

The oracle is a plain, slow C++17 library (``ffn_oracle.cpp``, built in-tree
into ``liboracle.so`` by ``_lib.build``) that restates what the pages
compute: bf16 and OCP FP8 E4M3 codecs from the format definitions, the
prefill chain (fused residual + RMSNorm + abs-max in fp64, per-tensor
quantisation, scaled FP8 GEMMs with exact int64 sums, SwiGLU with abs-max and
requantisation), its recompute form, the attention projections'
quantise-then-matmul, the FP8 backward of the FFN, and the single-token
decode FFN (row-scaled GEMVs with compensated fp64 sums, silu_mul).  The
Python modules ``codecs`` and ``ffn`` only marshal numpy arrays into it.

Every function is pinned by ``tests/test_oracle_*.py`` against hand-worked
values (``tests/golden/``), closed forms, invariants, library cross-checks
and brute-force exact arithmetic on tiny inputs (``tests/brute.py``); the
``plant`` context manager puts one deliberate mistake into the library so
the tests can show that each pin fails on it.
"""
from .codecs import (E4M3_MAX, bf16_to_f32, bf16_to_f64, e4m3_decode, e4m3_encode,
                     e4m3_to_scaled_int, f32_to_bf16, f64_to_bf16)
from .ffn import (PLANTS, absmax, backward_qmm, decode_forward, ffn_backward, ffn_forward,
                  ffn_forward_recompute, fp8_gemm_exact, fp8_gemm_scaled, fp8_gemm_scaled_acc, gemv_dual,
                  gemv_exact, gemv_row_scaled, max_threads, plant, quantize_rows, quantize_tensor,
                  quantize_with_abs_max, qmm, residual_rmsnorm_absmax, rmsnorm_f64, set_threads, silu_f64,
                  silu_mul, swiglu, swiglu_backward, swiglu_forward_quant, swiglu_quant)

__all__ = [
    "E4M3_MAX", "bf16_to_f32", "bf16_to_f64", "e4m3_decode", "e4m3_encode",
    "e4m3_to_scaled_int", "f32_to_bf16", "f64_to_bf16", "PLANTS", "absmax", "backward_qmm",
    "decode_forward", "ffn_backward", "ffn_forward", "ffn_forward_recompute", "fp8_gemm_exact",
    "fp8_gemm_scaled", "fp8_gemm_scaled_acc", "gemv_dual", "gemv_exact", "gemv_row_scaled",
    "max_threads", "plant", "quantize_rows", "quantize_tensor", "quantize_with_abs_max", "qmm",
    "residual_rmsnorm_absmax", "rmsnorm_f64", "set_threads", "silu_f64", "silu_mul", "swiglu",
    "swiglu_backward", "swiglu_forward_quant", "swiglu_quant",
]
