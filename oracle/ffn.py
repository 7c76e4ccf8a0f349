"""CPU oracle for the FP8 SwiGLU FFN block: prefill chain and single-token decode.

TEST INFRASTRUCTURE: part of the CPU oracle; see ``oracle/__init__.py``.

Sources (page title, function):

* [llmq-model]  IST-DASLab/llmq "src/models/llama_model.cpp":
  ``LLamaModel::_forward_block`` (FFN half: ``fused_residual_rmsnorm_forward``
  -> ``forward_qmm`` on the up projection -> ``swiglu_forward`` ->
  ``forward_qmm`` on the down projection), ``forward_qmm`` (quantise with the
  recorded abs-max, then a matmul scaled by weight and activation scales),
  ``_recompute_block`` (``swiglu_forward_quant``), ``fill_block_shapes``
  (``UP_W [2H, C]``, ``DOWN_W [C, H]``), ``LLamaModel::forward``
  (``fill_zero(AbsMaxes)`` before the layers).
* [llmq-state]  IST-DASLab/llmq "src/models/llama_run_state.cpp":
  buffer shapes and dtypes (``allocate_basic_fwd_tensors``,
  ``allocate_fwd_quant_tensors``) and the stats block (two floats per
  quantised tensor, abs-max then scale).
* [metrale-decode]  metrale "layers/dense_ffn_decode.rs",
  ``DenseFfnLayer::forward``, FP8 arm: ``w8a16_gemv_dual`` (gate and up
  GEMVs over one input, each weight with a per-output-row fp32 scale),
  ``silu_mul`` writing back into the gate buffer, ``w8a16_gemv`` for down.

The pages call these kernels but do not define their arithmetic.  Where
they leave a step open this oracle takes the plain readings listed below
(each is repeated in the function that applies it):

R1  gate = columns/rows ``[0, H)`` of the fused up projection, up = ``[H, 2H)``.
R2  ``scale = abs_max / 448`` is the dequantisation multiplier.
R3  the norm reads the stored, bf16-rounded residual sum.
R4  RMSNorm: ``y = bf16(r * rstd * g)`` with one rounding; rstd kept as fp32.
R5  the abs-max is taken over the bf16 values that are quantised.
R6  element scaling: ``float(v) * (448f / abs_max)`` in fp32, then E4M3 RNE
    with saturation.
R7  ``abs_max == 0``: scale 1, every code 0.
R9  GEMM output: fp32-exact accumulate times both scales, one bf16 rounding;
    SwiGLU reads those bf16 values.
R10 ``silu(z) = z / (1 + exp(-z))``.
R11 the SwiGLU-with-quantisation result equals swiglu (recording the abs-max
    of bf16 h) followed by quantisation of that same bf16 h.
R14 decode g, u, h are bf16; the row scale multiplies the finished sum.
R15 the decode input is already normalised; no norm in the decode FFN.
R19 a matmul bias (the QKV projection's) is added to the scaled accumulator
    before its single rounding to bf16.
R20 backward: gradients are bf16 (the model dtype of the activation
    buffers); their FP8 copies use E4M3 like the activations (the pages leave
    the gradient FP8 type open).
R21 swiglu_backward: with g, u the bf16 gate/up values and dh the bf16
    gradient of h, ``dg = dh * u * sigmoid(g) * (1 + g * (1 - sigmoid(g)))``
    and ``du = dh * silu(g)``, each rounded once to bf16; gate gradient in
    columns ``[0, H)``, up in ``[H, 2H)``; the abs-max of both is recorded.
R22 weight-gradient accumulation (``accumulate_gradient``): the new value is
    ``bf16(old + scaled product)``, one rounding.

Precision: RMSNorm, SwiGLU and GEMV sums are float64 with one final rounding
to bf16; scales are IEEE fp32 divisions; the FP8 GEMM is exact (see
``fp8_gemm_scaled``).
"""
from __future__ import annotations

import numpy as np

from .codecs import (E4M3_MAX, bf16_to_f32, bf16_to_f64, e4m3_decode, e4m3_encode,
                     e4m3_to_scaled_int, f64_to_bf16)

_F448 = np.float32(E4M3_MAX)


# ------------------------------------------------------------------ A1 (K1/K2)
def rmsnorm_f64(r_bits, gain_bits, eps: float):
    """Unrounded RMSNorm of bf16 rows: returns (r * rstd * g in float64, rstd float64).

    ``ms = mean_C(r**2)``, ``rstd = 1 / sqrt(ms + eps)`` [llmq-model,
    ``fused_residual_rmsnorm_forward`` / ``rmsnorm_forward`` with
    ``Config.RmsNormEps``].
    """
    r = bf16_to_f64(r_bits)
    ms = np.mean(r * r, axis=-1)
    rstd = 1.0 / np.sqrt(ms + float(np.float32(eps)))
    return r * rstd[..., None] * bf16_to_f64(gain_bits), rstd


def residual_rmsnorm_absmax(res_bits, x_bits, gain_bits, eps: float):
    """Step A1: fused residual add + RMSNorm + abs-max of the normalised output.

    [llmq-model] ``_forward_block`` calls ``fused_residual_rmsnorm_forward(
    ResidualAtt, LN2.Value, LN2_Rstd, residual, AttO, LN2_w,
    LN2.Quant.abs_max(), eps, B*T, C)``: the residual sum is stored (bf16),
    the normalised row goes to ``ln2`` (bf16), rstd to ``ln2_rstd`` (fp32
    ``[B, T]``) and the tensor abs-max into the stats slot.  With
    ``res_bits=None`` it is ``rmsnorm_forward`` (no residual): r is x.

    Returns ``(r, y, rstd, amax)``: r, y bf16 bits ``[N, C]``, rstd fp32
    ``[N]``, amax fp32 scalar.
    """
    if res_bits is None:
        r = np.array(x_bits, dtype=np.uint16, copy=True)
    else:
        # the sum of two bf16 values, rounded once to bf16 (stored ResidualAtt)
        r = f64_to_bf16(bf16_to_f64(res_bits) + bf16_to_f64(x_bits))
    y64, rstd = rmsnorm_f64(r, gain_bits, eps)          # R3: norm of stored bf16 r
    y = f64_to_bf16(y64)                                # R4: one rounding
    amax = absmax(y)                                    # R5
    return r, y, rstd.astype(np.float32), amax


def absmax(bits) -> np.float32:
    """Tensor abs-max of bf16 values (brute force), as fp32 [llmq-model ``abs_max``]."""
    v = bf16_to_f64(bits)
    if v.size == 0:
        return np.float32(0.0)
    return np.float32(np.max(np.abs(v)))


# ------------------------------------------------------------------ A2 (K3)
def quantize_with_abs_max(v_bits, amax):
    """Step A2: per-tensor E4M3 quantisation from a recorded abs-max.

    [llmq-model] ``forward_qmm``: ``quantize_with_abs_max(inp.Quant,
    inp.Quant.scale(), inp.Value, inp.Quant.abs_max(), B*T*C)`` writes the
    FP8 copy and its scale; the matmul then multiplies by that scale.

    R2 ``scale = amax / 448`` (fp32 division); R6 each element is
    ``e4m3(float(v) * (448 / amax))`` with the product rounded to fp32;
    R7 ``amax == 0`` gives scale 1 and all-zero codes.
    Returns ``(codes uint8, scale fp32)``.
    """
    amax = np.float32(amax)
    v = bf16_to_f32(v_bits)
    if amax == 0:
        return np.zeros(v.shape, dtype=np.uint8), np.float32(1.0)
    scale = np.float32(amax / _F448)
    inv = np.float32(_F448 / amax)
    return e4m3_encode(v * inv), scale


def quantize_rows(w_bits):
    """Per-output-row E4M3 weight record for the decode GEMVs.

    [metrale-decode] the FP8 weights carry ``row_scale``: one fp32 scale per
    output row.  Each row is quantised like ``quantize_with_abs_max`` with its
    own abs-max (scale = row abs-max / 448).  Returns ``(codes [R, K] uint8,
    row_scale [R] fp32)``.
    """
    w = bf16_to_f32(w_bits)
    amax = np.max(np.abs(w), axis=1).astype(np.float32)          # per row
    zero = amax == 0
    safe = np.where(zero, np.float32(1.0), amax)
    scales = np.where(zero, np.float32(1.0), safe / _F448).astype(np.float32)
    inv = (_F448 / safe).astype(np.float32)
    codes = e4m3_encode(w * inv[:, None])                          # fp32 products
    codes[zero] = 0
    return codes, scales


def quantize_tensor(w_bits):
    """Per-tensor E4M3 record of a bf16 tensor: abs-max, then A2."""
    return quantize_with_abs_max(w_bits, absmax(w_bits))


# ------------------------------------------------------------------ A3 / A5 (K4)
def fp8_gemm_scaled(a_codes, a_scale, w_codes, w_scale):
    """Steps A3/A5: ``out[m, n] = bf16(a_scale * w_scale * sum_k A[m, k] * W[n, k])``.

    [llmq-model] ``forward_qmm`` -> ``matmul(out, weight, inp.Quant, bias,
    weight.scale(), inp.Quant.scale(), ..., OC, B*T, C, TN)``: both operands
    are FP8 with the reduction dimension contiguous ("TN"), the result is a
    model-dtype (bf16) buffer (R9).

    Exactness: every E4M3 value times ``2**9`` is an integer of magnitude at
    most 229376 < 2**18, so each product is an integer below 2**36 and any
    partial sum of at most 2**15 products stays below 2**51 < 2**53.  Float64
    represents all of these integers, so the float64 matrix product of the
    scaled integers is the exact integer sum regardless of summation order.
    The only roundings are the float64 products with the two scales
    (relative 2**-53) and the final bf16 rounding.
    """
    a = e4m3_to_scaled_int(a_codes)
    w = e4m3_to_scaled_int(w_codes)
    if a.shape[-1] > (1 << 15):
        raise ValueError("K above 2**15 breaks the exact-sum bound")
    acc = a @ w.T
    return f64_to_bf16(np.ldexp(acc, -18) * float(np.float32(a_scale)) * float(np.float32(w_scale)))


def qmm(in_bits, amax, w_codes, w_scale, bias_bits=None):
    """``forward_qmm``: quantise a bf16 activation with its recorded abs-max, then
    the scaled FP8 matmul, with an optional bf16 bias per output column.

    [llmq-model] ``forward_qmm(out, inp, weight, bias, ...)`` runs
    ``quantize_with_abs_max`` on ``inp`` and then ``matmul(out, weight,
    inp.Quant, bias, weight.scale(), inp.Quant.scale(), ...)``.
    ``_forward_block`` calls it for the QKV projection (with
    ``Attn_QKV_b``), the attention output projection and both FFN
    projections.  R9: the exact accumulator times both scales is rounded once
    to bf16.  R19: a bias is added to that scaled value before the one
    rounding.  Returns ``(out bits [M, N], codes [M, K], scale)``.
    """
    codes, scale = quantize_with_abs_max(in_bits, amax)
    a = e4m3_to_scaled_int(codes)
    w = e4m3_to_scaled_int(w_codes)
    if a.shape[-1] > (1 << 15):
        raise ValueError("K above 2**15 breaks the exact-sum bound")
    v = np.ldexp(a @ w.T, -18) * float(scale) * float(np.float32(w_scale))
    if bias_bits is not None:
        v = v + bf16_to_f64(bias_bits)[None, :]
    return f64_to_bf16(v), codes, scale


# ------------------------------------------------------------------ A4 (K5/K6)
def silu_f64(z):
    """R10: silu(z) = z * sigmoid(z) = z / (1 + exp(-z)), float64."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(gu_bits, H: int):
    """Step A4 (first half): ``h = bf16(silu(g) * u)`` and its abs-max.

    [llmq-model] ``swiglu_forward(SwiGLu.Value, MlpUp, SwiGLu.Quant.abs_max(),
    B, T, D)`` reads the ``[N, 2H]`` up-projection output; R1: gate is
    ``gu[:, :H]``, up is ``gu[:, H:]``.  Returns ``(h bits [N, H], amax fp32)``.
    """
    gu = np.asarray(gu_bits, dtype=np.uint16)
    g = bf16_to_f64(gu[..., :H])
    u = bf16_to_f64(gu[..., H:2 * H])
    h = f64_to_bf16(silu_f64(g) * u)
    return h, absmax(h)


def swiglu_quant(gu_bits, H: int):
    """Step A4: SwiGLU with abs-max, then requantisation of that bf16 h (R11).

    Returns ``(h bits, hq codes, stats fp32[2] = {abs_max, scale})``
    [llmq-state: two floats per tensor, abs-max first].
    """
    h, amax = swiglu(gu_bits, H)
    hq, scale = quantize_with_abs_max(h, amax)
    return h, hq, np.array([amax, scale], dtype=np.float32)


def swiglu_forward_quant(gu_bits, H: int, amax):
    """Step A4 in the recompute form: SwiGLU quantised with an abs-max given, not recorded.

    [llmq-model] ``_recompute_block``: ``swiglu_forward_quant(SwiGLu.Quant,
    SwiGLu.Quant.scale(), MlpUp, SwiGLu.Quant.abs_max(), B, T, D)`` reads the
    abs-max the forward left in the stats slot and writes the FP8 copy and
    its scale.  h is the bf16 SwiGLU value of ``swiglu`` (R9, R10); it is
    quantised by A2's rule with the given abs-max (R2, R6, R7), and values
    beyond that abs-max saturate at +-448 (R8).  Returns ``(hq codes, scale)``.
    """
    h, _ = swiglu(gu_bits, H)
    return quantize_with_abs_max(h, amax)


# ------------------------------------------------------------------ A1..A5
def ffn_forward(res_bits, x_bits, gain_bits, eps, w1_codes, w1_scale, w2_codes, w2_scale, H: int):
    """The whole prefill FFN chain A1..A5 [llmq-model ``_forward_block``, FFN half].

    Stats are zeroed before the chain (``fill_zero(AbsMaxes)``), so each
    abs-max is the max over the tensor just produced.  Returns a dict with
    every intermediate: r, y, rstd, stats_y, yq, gu, h, stats_h, hq, out.
    """
    r, y, rstd, amax_y = residual_rmsnorm_absmax(res_bits, x_bits, gain_bits, eps)
    yq, sy = quantize_with_abs_max(y, amax_y)
    gu = fp8_gemm_scaled(yq, sy, w1_codes, w1_scale)
    h, hq, stats_h = swiglu_quant(gu, H)
    out = fp8_gemm_scaled(hq, stats_h[1], w2_codes, w2_scale)
    return {
        "r": r, "y": y, "rstd": rstd, "stats_y": np.array([amax_y, sy], dtype=np.float32),
        "yq": yq, "gu": gu, "h": h, "stats_h": stats_h, "hq": hq, "out": out,
    }


def ffn_forward_recompute(res_bits, x_bits, gain_bits, eps, w1_codes, w1_scale, w2_codes,
                          w2_scale, H: int, amax_y, amax_h):
    """The prefill chain with both activation abs-maxes given instead of recorded.

    [llmq-model] ``_recompute_block``, FFN half:
    - the norm is re-run without recording an abs-max
      (``fused_residual_rmsnorm_forward(..., nullptr, eps, ...)``);
    - the up projection's ``forward_qmm`` quantises LN2 with the abs-max its
      stats slot still holds;
    - ``swiglu_forward_quant`` quantises h with the recorded SwiGLU abs-max.

    The recompute block stops at the quantised h.  This chain then applies the
    down projection exactly as the forward does (``forward_qmm`` on the down
    weight with the SwiGLU scale), so it yields the block output.  Given the
    abs-maxes that ``ffn_forward`` recorded, every result equals that forward's.
    Returns r, y, rstd, stats_y, yq, gu, hq, stats_h, out.
    """
    r, y, rstd, _ = residual_rmsnorm_absmax(res_bits, x_bits, gain_bits, eps)
    amax_y, amax_h = np.float32(amax_y), np.float32(amax_h)
    yq, sy = quantize_with_abs_max(y, amax_y)
    gu = fp8_gemm_scaled(yq, sy, w1_codes, w1_scale)
    hq, sh = swiglu_forward_quant(gu, H, amax_h)
    out = fp8_gemm_scaled(hq, sh, w2_codes, w2_scale)
    return {
        "r": r, "y": y, "rstd": rstd, "stats_y": np.array([amax_y, sy], dtype=np.float32),
        "yq": yq, "gu": gu, "hq": hq, "stats_h": np.array([amax_h, sh], dtype=np.float32),
        "out": out,
    }


# ------------------------------------------------------------------ FFN backward (FP8)
def swiglu_backward(dh_bits, gu_bits, H: int):
    """Gradient of ``h = silu(g) * u`` w.r.t. the fused up-projection output.

    [llmq-model] ``_backward_block``: ``swiglu_backward(DMlpUp.Value, DSwiGLU,
    MlpUp, DMlpUp.Quant.abs_max(), B, T, D)``.  R21: ``dg = dh * u *
    sigmoid(g) * (1 + g * (1 - sigmoid(g)))``, ``du = dh * silu(g)`` in
    float64, each rounded once to bf16; R1 layout (gate first).  Returns
    ``(d_gu bits [N, 2H], abs-max fp32)``.
    """
    gu = np.asarray(gu_bits, dtype=np.uint16)
    g = bf16_to_f64(gu[..., :H])
    u = bf16_to_f64(gu[..., H:2 * H])
    dh = bf16_to_f64(dh_bits)
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
    dg = dh * u * sig * (1.0 + g * (1.0 - sig))
    du = dh * (g * sig)
    d = f64_to_bf16(np.concatenate([dg, du], axis=-1))
    return d, absmax(d)


def fp8_gemm_scaled_acc(a_codes, a_scale, w_codes, w_scale, old_bits=None):
    """``fp8_gemm_scaled`` with ``accumulate_gradient`` (R22): ``bf16(old + product)``."""
    if old_bits is None:
        return fp8_gemm_scaled(a_codes, a_scale, w_codes, w_scale)
    a = e4m3_to_scaled_int(a_codes)
    w = e4m3_to_scaled_int(w_codes)
    if a.shape[-1] > (1 << 15):
        raise ValueError("K above 2**15 breaks the exact-sum bound")
    v = np.ldexp(a @ w.T, -18) * float(np.float32(a_scale)) * float(np.float32(w_scale))
    return f64_to_bf16(bf16_to_f64(old_bits) + v)


def backward_qmm(dout_bits, dout_amax, inp_codes, inp_scale, w_codes, w_scale, dw_old_bits=None):
    """The FP8 branch of ``backward_qmm`` for one projection ``out = inp @ W^T``.

    [llmq-model] ``backward_qmm``, FP8 weights: ``quantize_with_abs_max`` of
    dout with its recorded abs-max; ``dinp = matmul(transpose(W), dout_q)``
    with ``W.scale() * dout.scale()`` (reduction over the output channels);
    ``dW (+)= matmul(transpose(inp_q), transpose(dout_q))`` with
    ``inp.scale() * dout.scale()`` (reduction over the tokens), the forward's
    quantised input reused.  Shapes: dout ``[N, OC]``, inp ``[N, IC]``,
    W ``[OC, IC]``.  Returns ``(dinp bits [N, IC], dW bits [OC, IC], dout
    codes, dout scale)``.
    """
    dq, ds = quantize_with_abs_max(dout_bits, dout_amax)
    dinp = fp8_gemm_scaled(dq, ds, np.ascontiguousarray(np.asarray(w_codes).T), w_scale)
    dw = fp8_gemm_scaled_acc(np.ascontiguousarray(dq.T), ds,
                             np.ascontiguousarray(np.asarray(inp_codes).T), inp_scale, dw_old_bits)
    return dinp, dw, dq, ds


def ffn_backward(dout_bits, dout_amax, yq_codes, y_scale, hq_codes, h_scale, w1_codes, w1_scale,
                 w2_codes, w2_scale, H: int, dw1_old=None, dw2_old=None):
    """Backward of the FP8 FFN (after the norm) [llmq-model ``_backward_block``].

    The down projection's ``backward_qmm`` (dout = the block-output gradient,
    inp = the quantised SwiGLU output), ``swiglu_backward`` on the up
    projection's output ``gu`` (recomputed from yq as ``_recompute_block``
    does), then the up projection's ``backward_qmm`` (dout = d_gu with the
    abs-max swiglu_backward recorded, inp = the quantised LN2 output).
    Returns d_ln2, dw1, dw2, dh, gu, d_gu and the two stats pairs.
    """
    dh, dw2, dq, ds = backward_qmm(dout_bits, dout_amax, hq_codes, h_scale, w2_codes, w2_scale, dw2_old)
    gu = fp8_gemm_scaled(yq_codes, y_scale, w1_codes, w1_scale)
    d_gu, amax_dgu = swiglu_backward(dh, gu, H)
    d_ln2, dw1, dguq, sdgu = backward_qmm(d_gu, amax_dgu, yq_codes, y_scale, w1_codes, w1_scale, dw1_old)
    return {
        "dh": dh, "dw2": dw2, "dout_q": dq, "stats_dout": np.array([dout_amax, ds], dtype=np.float32),
        "gu": gu, "d_gu": d_gu, "d_gu_q": dguq,
        "stats_dgu": np.array([amax_dgu, sdgu], dtype=np.float32), "d_ln2": d_ln2, "dw1": dw1,
    }


# ------------------------------------------------------------------ A6..A8
def gemv_row_scaled(x_bits, w_codes, row_scale):
    """``out[r] = bf16(row_scale[r] * sum_k W[r, k] * x[k])`` [metrale-decode ``w8a16_gemv``].

    W8A16: FP8 weight rows, bf16 activation.  The sum is float64 (error at
    most ``K * 2**-53 * sum|terms|``), the row scale multiplies the finished
    sum (R14), one rounding to bf16.
    """
    w = e4m3_decode(w_codes)
    x = bf16_to_f64(x_bits)
    acc = w @ x
    return f64_to_bf16(np.asarray(row_scale, dtype=np.float32).astype(np.float64) * acc)


def gemv_dual(x_bits, wg_codes, sg, wu_codes, su):
    """Step A6 [metrale-decode ``w8a16_gemv_dual``]: gate and up GEMVs of one input."""
    return gemv_row_scaled(x_bits, wg_codes, sg), gemv_row_scaled(x_bits, wu_codes, su)


def silu_mul(g_bits, u_bits):
    """Step A7 [metrale-decode ``silu_mul``]: ``bf16(silu(g) * u)``."""
    return f64_to_bf16(silu_f64(bf16_to_f64(g_bits)) * bf16_to_f64(u_bits))


def decode_forward(x_bits, wg_codes, sg, wu_codes, su, wd_codes, sd):
    """Steps A6..A8, the single-token FP8 decode FFN (split-SiLU arm) [metrale-decode].

    Returns a dict with g, u, h (bf16 bits ``[H]``) and out (bf16 bits ``[C]``).
    """
    g, u = gemv_dual(x_bits, wg_codes, sg, wu_codes, su)
    h = silu_mul(g, u)
    out = gemv_row_scaled(h, wd_codes, sd)
    return {"g": g, "u": u, "h": h, "out": out}
