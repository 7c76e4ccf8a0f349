"""CPU oracle for the FP8 SwiGLU FFN block: prefill chain and single-token decode.

TEST INFRASTRUCTURE: part of the CPU oracle; see ``oracle/__init__.py``.

The arithmetic of every step is in ``ffn_oracle.cpp`` (plain C++17), whose
header lists the pages' functions it follows and the readings it takes
(R1-R22).  These functions only marshal numpy arrays into those calls, allocate
the outputs and name them:

* [llmq-model]  IST-DASLab/llmq "src/models/llama_model.cpp",
  ``LLamaModel::_forward_block`` (FFN half), ``forward_qmm``,
  ``_recompute_block``, ``_backward_block`` / ``backward_qmm``.
* [llmq-state]  IST-DASLab/llmq "src/models/llama_run_state.cpp": buffer
  dtypes and the stats block (abs-max, then scale).
* [metrale-decode]  metrale "layers/dense_ffn_decode.rs",
  ``DenseFfnLayer::forward``, FP8 arm.
"""
from __future__ import annotations

import contextlib

import numpy as np

from ._lib import lib

# Planted mistakes (the pin tests set one to show the pins can fail).
PLANTS = {
    "gate_up_swapped": 1, "e4m3_ties_away": 2, "e4m3_no_saturation": 3, "norm_unrounded_sum": 4,
    "gemm_drops_last_k": 5, "silu_sign": 6, "bf16_truncates": 7, "quant_divides": 8,
    "dsilu_no_correction": 9, "gemv_scale_by_first": 10,
}


@contextlib.contextmanager
def plant(name: str):
    """Run the enclosed oracle calls with one deliberate mistake in the oracle (tests only)."""
    lib().orc_set_plant(PLANTS[name])
    try:
        yield
    finally:
        lib().orc_set_plant(0)


def set_threads(n: int) -> None:
    """Number of OpenMP threads the oracle uses (n <= 0: all processors)."""
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


# ------------------------------------------------------------------ A1 (K1/K2)
def rmsnorm_f64(r_bits, gain_bits, eps: float):
    """Unrounded RMSNorm of bf16 rows: (r * rstd * g in float64, rstd float64)."""
    r = _c(r_bits, np.uint16)
    g = _c(gain_bits, np.uint16)
    C = r.shape[-1]
    N = r.size // C if C else 0
    y = np.empty(r.shape, dtype=np.float64)
    rstd = np.empty(r.shape[:-1], dtype=np.float64)
    lib().orc_rmsnorm_f64(_p(r), _p(g), float(np.float32(eps)), N, C, _p(y), _p(rstd))
    return y, rstd


def residual_rmsnorm_absmax(res_bits, x_bits, gain_bits, eps: float):
    """Step A1, fused residual add + RMSNorm + abs-max [llmq-model
    ``fused_residual_rmsnorm_forward``]; ``res_bits=None`` is ``rmsnorm_forward``.

    Returns ``(r, y, rstd, amax)``: r, y bf16 bits ``[N, C]``, rstd fp32 ``[N]``,
    amax fp32 scalar.
    """
    x = _c(x_bits, np.uint16)
    res = None if res_bits is None else _c(res_bits, np.uint16)
    g = _c(gain_bits, np.uint16)
    C = x.shape[-1]
    N = x.size // C if C else 0
    r = np.empty(x.shape, dtype=np.uint16)
    y = np.empty(x.shape, dtype=np.uint16)
    rstd = np.empty(x.shape[:-1], dtype=np.float32)
    amax = np.zeros(1, dtype=np.float32)
    lib().orc_residual_rmsnorm_absmax(_p(res), _p(x), _p(g), float(np.float32(eps)), N, C, _p(r), _p(y),
                                      _p(rstd), _p(amax))
    return r, y, rstd, amax[0]


def absmax(bits) -> np.float32:
    """Tensor abs-max of bf16 values, as fp32 [llmq-model ``abs_max``]."""
    b = _c(bits, np.uint16)
    return np.float32(lib().orc_absmax_bf16(_p(b), b.size))


# ------------------------------------------------------------------ A2 (K3)
def quantize_with_abs_max(v_bits, amax):
    """Step A2 [llmq-model ``forward_qmm`` -> ``quantize_with_abs_max``]:
    ``(codes uint8, scale fp32)`` with scale = amax / 448 (R2, R6, R7)."""
    v = _c(v_bits, np.uint16)
    codes = np.empty(v.shape, dtype=np.uint8)
    scale = np.zeros(1, dtype=np.float32)
    lib().orc_quantize_with_abs_max(_p(v), v.size, float(np.float32(amax)), _p(codes), _p(scale))
    return codes, scale[0]


def quantize_rows(w_bits):
    """Per-output-row E4M3 record of decode weights [metrale-decode ``row_scale``]:
    ``(codes [R, K], row_scale [R] fp32)``."""
    w = _c(w_bits, np.uint16)
    R, K = w.shape
    codes = np.empty((R, K), dtype=np.uint8)
    scales = np.empty(R, dtype=np.float32)
    lib().orc_quantize_rows(_p(w), R, K, _p(codes), _p(scales))
    return codes, scales


def quantize_tensor(w_bits):
    """Per-tensor E4M3 record of a bf16 tensor: abs-max, then A2."""
    return quantize_with_abs_max(w_bits, absmax(w_bits))


# ------------------------------------------------------------------ A3 / A5 (K4)
def _gemm(a_codes, a_scale, w_codes, w_scale, bias_bits=None, old_bits=None, a_t=False, w_t=False):
    """out = bf16(old + sa * sw * A @ W^T + bias); ``a_t`` / ``w_t`` read the operand transposed."""
    a = _c(a_codes, np.uint8)
    w = _c(w_codes, np.uint8)
    M, K = (a.shape[1], a.shape[0]) if a_t else a.shape
    N, Kw = (w.shape[1], w.shape[0]) if w_t else w.shape
    assert K == Kw, (a.shape, w.shape)
    a_ms, a_ks = (1, M) if a_t else (K, 1)
    b_ns, b_ks = (1, N) if w_t else (K, 1)
    bias = None if bias_bits is None else _c(bias_bits, np.uint16)
    old = None if old_bits is None else _c(old_bits, np.uint16)
    out = np.empty((M, N), dtype=np.uint16)
    rc = lib().orc_fp8_gemm(_p(a), a_ms, a_ks, float(np.float32(a_scale)), _p(w), b_ns, b_ks,
                            float(np.float32(w_scale)), M, N, K, _p(bias), _p(old), _p(out))
    if rc != 0:
        raise ValueError("K too large for the exact int64 sum")
    return out


def fp8_gemm_scaled(a_codes, a_scale, w_codes, w_scale):
    """Steps A3/A5: ``out[m, n] = bf16(a_scale * w_scale * sum_k A[m, k] * W[n, k])``
    [llmq-model ``forward_qmm`` -> ``matmul(..., weight.scale(), inp.Quant.scale(), ..., TN)``];
    the sum exact, one rounding (R9)."""
    return _gemm(a_codes, a_scale, w_codes, w_scale)


def fp8_gemm_exact(a_codes, a_scale, w_codes, w_scale):
    """The unrounded fp64 value ``a_scale * w_scale * sum_k A[m, k] * W[n, k]`` (exact sum)."""
    a = _c(a_codes, np.uint8)
    w = _c(w_codes, np.uint8)
    M, K = a.shape
    N = w.shape[0]
    out = np.empty((M, N), dtype=np.float64)
    rc = lib().orc_fp8_gemm_exact(_p(a), K, 1, float(np.float32(a_scale)), _p(w), K, 1,
                                  float(np.float32(w_scale)), M, N, K, _p(out))
    if rc != 0:
        raise ValueError("K too large for the exact int64 sum")
    return out


def qmm(in_bits, amax, w_codes, w_scale, bias_bits=None):
    """``forward_qmm`` [llmq-model]: quantise with the recorded abs-max, then the
    scaled FP8 matmul, optional bf16 bias added before the one rounding (R19).
    Returns ``(out bits [M, N], codes [M, K], scale)``."""
    codes, scale = quantize_with_abs_max(in_bits, amax)
    return _gemm(codes, scale, w_codes, w_scale, bias_bits=bias_bits), codes, scale


# ------------------------------------------------------------------ A4 (K5/K6)
def silu_f64(z):
    """R10: silu(z) = z / (1 + exp(-z)), float64."""
    v = _c(z, np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    lib().orc_silu(_p(v), _p(out), v.size)
    return out


def swiglu(gu_bits, H: int):
    """Step A4, first half [llmq-model ``swiglu_forward``]: ``h = bf16(silu(g) * u)``
    with gate ``gu[:, :H]`` and up ``gu[:, H:]`` (R1), and its abs-max."""
    gu = _c(gu_bits, np.uint16)
    lead = gu.shape[:-1]
    N = int(np.prod(lead)) if lead else 1
    h = np.empty(lead + (H,), dtype=np.uint16)
    amax = np.zeros(1, dtype=np.float32)
    lib().orc_swiglu(_p(gu), N, H, _p(h), _p(amax))
    return h, amax[0]


def swiglu_quant(gu_bits, H: int):
    """Step A4: SwiGLU with abs-max, then requantisation of that bf16 h (R11).
    Returns ``(h, hq, stats fp32[2] = {abs_max, scale})``."""
    h, amax = swiglu(gu_bits, H)
    hq, scale = quantize_with_abs_max(h, amax)
    return h, hq, np.array([amax, scale], dtype=np.float32)


def swiglu_forward_quant(gu_bits, H: int, amax):
    """Step A4, recompute form [llmq-model ``_recompute_block`` ->
    ``swiglu_forward_quant``]: h quantised with an abs-max given, not recorded."""
    h, _ = swiglu(gu_bits, H)
    return quantize_with_abs_max(h, amax)


# ------------------------------------------------------------------ A1..A5
def ffn_forward(res_bits, x_bits, gain_bits, eps, w1_codes, w1_scale, w2_codes, w2_scale, H: int,
                timing: dict | None = None):
    """The prefill FFN chain A1..A5 [llmq-model ``_forward_block``, FFN half].

    Returns every intermediate: r, y, rstd, stats_y, yq, gu, h, stats_h, hq, out.
    If ``timing`` is a dict, ``timing["seconds"]`` receives the chain's
    steady-clock time measured inside the library.
    """
    x = _c(x_bits, np.uint16)
    res = None if res_bits is None else _c(res_bits, np.uint16)
    g = _c(gain_bits, np.uint16)
    w1 = _c(w1_codes, np.uint8)
    w2 = _c(w2_codes, np.uint8)
    N, C = x.shape
    o = {"r": np.empty((N, C), np.uint16), "y": np.empty((N, C), np.uint16), "rstd": np.empty(N, np.float32),
         "stats_y": np.zeros(2, np.float32), "yq": np.empty((N, C), np.uint8),
         "gu": np.empty((N, 2 * H), np.uint16), "h": np.empty((N, H), np.uint16),
         "stats_h": np.zeros(2, np.float32), "hq": np.empty((N, H), np.uint8),
         "out": np.empty((N, C), np.uint16)}
    sec = np.zeros(1, np.float64)
    rc = lib().orc_ffn_forward(_p(res), _p(x), _p(g), float(np.float32(eps)), _p(w1), float(np.float32(w1_scale)),
                               _p(w2), float(np.float32(w2_scale)), N, C, H, _p(o["r"]), _p(o["y"]),
                               _p(o["rstd"]), _p(o["stats_y"]), _p(o["yq"]), _p(o["gu"]), _p(o["h"]),
                               _p(o["stats_h"]), _p(o["hq"]), _p(o["out"]), _p(sec))
    if rc != 0:
        raise ValueError("K too large for the exact int64 sum")
    if timing is not None:
        timing["seconds"] = float(sec[0])
    return o


def ffn_forward_recompute(res_bits, x_bits, gain_bits, eps, w1_codes, w1_scale, w2_codes,
                          w2_scale, H: int, amax_y, amax_h):
    """The prefill chain with both activation abs-maxes given [llmq-model
    ``_recompute_block``, FFN half, then the forward's down projection].
    Returns r, y, rstd, stats_y, yq, gu, hq, stats_h, out."""
    x = _c(x_bits, np.uint16)
    res = None if res_bits is None else _c(res_bits, np.uint16)
    g = _c(gain_bits, np.uint16)
    w1 = _c(w1_codes, np.uint8)
    w2 = _c(w2_codes, np.uint8)
    N, C = x.shape
    o = {"r": np.empty((N, C), np.uint16), "y": np.empty((N, C), np.uint16), "rstd": np.empty(N, np.float32),
         "stats_y": np.zeros(2, np.float32), "yq": np.empty((N, C), np.uint8),
         "gu": np.empty((N, 2 * H), np.uint16), "hq": np.empty((N, H), np.uint8),
         "stats_h": np.zeros(2, np.float32), "out": np.empty((N, C), np.uint16)}
    rc = lib().orc_ffn_forward_recompute(_p(res), _p(x), _p(g), float(np.float32(eps)), _p(w1),
                                         float(np.float32(w1_scale)), _p(w2), float(np.float32(w2_scale)),
                                         N, C, H, float(np.float32(amax_y)), float(np.float32(amax_h)),
                                         _p(o["r"]), _p(o["y"]), _p(o["rstd"]), _p(o["stats_y"]), _p(o["yq"]),
                                         _p(o["gu"]), _p(o["hq"]), _p(o["stats_h"]), _p(o["out"]))
    if rc != 0:
        raise ValueError("K too large for the exact int64 sum")
    return o


# ------------------------------------------------------------------ FFN backward (FP8)
def swiglu_backward(dh_bits, gu_bits, H: int):
    """[llmq-model ``_backward_block`` -> ``swiglu_backward``], R21:
    ``(d_gu bits [N, 2H], abs-max fp32)``."""
    dh = _c(dh_bits, np.uint16)
    gu = _c(gu_bits, np.uint16)
    lead = gu.shape[:-1]
    N = int(np.prod(lead)) if lead else 1
    d = np.empty(gu.shape, dtype=np.uint16)
    amax = np.zeros(1, dtype=np.float32)
    lib().orc_swiglu_backward(_p(dh), _p(gu), N, H, _p(d), _p(amax))
    return d, amax[0]


def fp8_gemm_scaled_acc(a_codes, a_scale, w_codes, w_scale, old_bits=None):
    """``fp8_gemm_scaled`` with ``accumulate_gradient`` (R22): ``bf16(old + product)``."""
    return _gemm(a_codes, a_scale, w_codes, w_scale, old_bits=old_bits)


def backward_qmm(dout_bits, dout_amax, inp_codes, inp_scale, w_codes, w_scale, dw_old_bits=None):
    """The FP8 branch of ``backward_qmm`` [llmq-model] for ``out = inp @ W^T``:
    dout ``[N, OC]``, inp ``[N, IC]``, W ``[OC, IC]``.  Returns ``(dinp [N, IC],
    dW [OC, IC], dout codes, dout scale)``."""
    dout = _c(dout_bits, np.uint16)
    inp = _c(inp_codes, np.uint8)
    w = _c(w_codes, np.uint8)
    N, OC = dout.shape
    IC = w.shape[1]
    old = None if dw_old_bits is None else _c(dw_old_bits, np.uint16)
    dinp = np.empty((N, IC), np.uint16)
    dw = np.empty((OC, IC), np.uint16)
    dq = np.empty((N, OC), np.uint8)
    ds = np.zeros(1, np.float32)
    rc = lib().orc_backward_qmm(_p(dout), float(np.float32(dout_amax)), _p(inp), float(np.float32(inp_scale)),
                                _p(w), float(np.float32(w_scale)), N, OC, IC, _p(old), _p(dinp), _p(dw), _p(dq),
                                _p(ds))
    if rc != 0:
        raise ValueError("K too large for the exact int64 sum")
    return dinp, dw, dq, ds[0]


def ffn_backward(dout_bits, dout_amax, yq_codes, y_scale, hq_codes, h_scale, w1_codes, w1_scale,
                 w2_codes, w2_scale, H: int, dw1_old=None, dw2_old=None):
    """Backward of the FP8 FFN after the norm [llmq-model ``_backward_block``].
    Returns dh, dw2, dout_q, stats_dout, gu, d_gu, d_gu_q, stats_dgu, d_ln2, dw1."""
    dout = _c(dout_bits, np.uint16)
    yq = _c(yq_codes, np.uint8)
    hq = _c(hq_codes, np.uint8)
    w1 = _c(w1_codes, np.uint8)
    w2 = _c(w2_codes, np.uint8)
    N, C = dout.shape
    o1 = None if dw1_old is None else _c(dw1_old, np.uint16)
    o2 = None if dw2_old is None else _c(dw2_old, np.uint16)
    o = {"dh": np.empty((N, H), np.uint16), "dw2": np.empty((C, H), np.uint16),
         "dout_q": np.empty((N, C), np.uint8), "stats_dout": np.zeros(2, np.float32),
         "gu": np.empty((N, 2 * H), np.uint16), "d_gu": np.empty((N, 2 * H), np.uint16),
         "d_gu_q": np.empty((N, 2 * H), np.uint8), "stats_dgu": np.zeros(2, np.float32),
         "d_ln2": np.empty((N, C), np.uint16), "dw1": np.empty((2 * H, C), np.uint16)}
    rc = lib().orc_ffn_backward(_p(dout), float(np.float32(dout_amax)), _p(yq), float(np.float32(y_scale)), _p(hq),
                                float(np.float32(h_scale)), _p(w1), float(np.float32(w1_scale)), _p(w2),
                                float(np.float32(w2_scale)), N, C, H, _p(o1), _p(o2), _p(o["dh"]), _p(o["dw2"]),
                                _p(o["dout_q"]), _p(o["stats_dout"]), _p(o["gu"]), _p(o["d_gu"]),
                                _p(o["d_gu_q"]), _p(o["stats_dgu"]), _p(o["d_ln2"]), _p(o["dw1"]))
    if rc != 0:
        raise ValueError("K too large for the exact int64 sum")
    return o


# ------------------------------------------------------------------ A6..A8
def gemv_row_scaled(x_bits, w_codes, row_scale):
    """``out[r] = bf16(row_scale[r] * sum_k W[r, k] * x[k])`` [metrale-decode ``w8a16_gemv``], R14."""
    x = _c(x_bits, np.uint16)
    w = _c(w_codes, np.uint8)
    s = _c(row_scale, np.float32)
    R, K = w.shape
    out = np.empty(R, np.uint16)
    lib().orc_gemv_row_scaled(_p(x), _p(w), _p(s), R, K, _p(out))
    return out


def gemv_exact(x_bits, w_codes, row_scale):
    """The unrounded fp64 value ``row_scale[r] * sum_k W[r, k] * x[k]``."""
    x = _c(x_bits, np.uint16)
    w = _c(w_codes, np.uint8)
    s = _c(row_scale, np.float32)
    R, K = w.shape
    out = np.empty(R, np.float64)
    lib().orc_gemv_exact(_p(x), _p(w), _p(s), R, K, _p(out))
    return out


def gemv_dual(x_bits, wg_codes, sg, wu_codes, su):
    """Step A6 [metrale-decode ``w8a16_gemv_dual``]: gate and up GEMVs of one input."""
    return gemv_row_scaled(x_bits, wg_codes, sg), gemv_row_scaled(x_bits, wu_codes, su)


def silu_mul(g_bits, u_bits):
    """Step A7 [metrale-decode ``silu_mul``]: ``bf16(silu(g) * u)``."""
    g = _c(g_bits, np.uint16)
    u = _c(u_bits, np.uint16)
    h = np.empty(g.shape, np.uint16)
    lib().orc_silu_mul(_p(g), _p(u), g.size, _p(h))
    return h


def decode_forward(x_bits, wg_codes, sg, wu_codes, su, wd_codes, sd):
    """Steps A6..A8, the single-token FP8 decode FFN, split-SiLU arm [metrale-decode].
    Returns g, u, h (bf16 bits ``[H]``) and out (``[C]``)."""
    x = _c(x_bits, np.uint16)
    wg, wu, wd = _c(wg_codes, np.uint8), _c(wu_codes, np.uint8), _c(wd_codes, np.uint8)
    sg, su, sd = _c(sg, np.float32), _c(su, np.float32), _c(sd, np.float32)
    H, C = wg.shape
    o = {"g": np.empty(H, np.uint16), "u": np.empty(H, np.uint16), "h": np.empty(H, np.uint16),
         "out": np.empty(C, np.uint16)}
    lib().orc_decode_forward(_p(x), _p(wg), _p(sg), _p(wu), _p(su), _p(wd), _p(sd), C, H, _p(o["g"]),
                             _p(o["u"]), _p(o["h"]), _p(o["out"]))
    return o
