"""Python binding of libqffn (FP8 SwiGLU FFN block for one GB300).

Argument marshalling only: each function here has the name of a C entry
point of ``include/qffn.h``, turns torch tensors (or raw integer device
addresses) into pointers, passes the current torch CUDA stream unless one is
given, and raises ``QffnError`` on a non-zero status.  Every step of the
block runs in the CUDA kernels of ``libqffn.so``; there is no fallback.  If
the library is missing the import fails (run ``build()`` first).
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as LIB_PATH
from ._build import build

__all__ = [
    "QffnError", "lib", "build", "LIB_PATH", "STATUS",
    "qffn_status_string", "qffn_abi_version", "qffn_check_status", "qffn_selftest_bounded_wait",
    "qffn_gemm_clock_sample",
    "qffn_rmsnorm_absmax", "qffn_absmax", "qffn_quantize", "qffn_quantize_rows",
    "qffn_fp8_gemm_scaled", "qffn_qmm", "qffn_gate_up_swiglu", "qffn_swiglu_quant",
    "qffn_swiglu_forward_quant", "qffn_gate_up_swiglu_quant",
    "qffn_forward_workspace_size", "qffn_forward_workspace_offsets", "qffn_forward",
    "qffn_forward_recompute", "qffn_transpose_e4m3", "qffn_swiglu_backward",
    "qffn_backward_qmm_workspace_size", "qffn_backward_qmm", "qffn_ffn_backward_workspace_size",
    "qffn_ffn_backward_workspace_offsets", "qffn_ffn_backward", "qffn_gate_up_swiglu_backward",
    "qffn_gemv_dual", "qffn_gemv", "qffn_gemv_silu_input", "qffn_silu_mul", "qffn_decode_workspace_size",
    "qffn_decode_workspace_offsets", "qffn_decode_forward", "qffn_decode_forward_ex", "qffn_decode_forward_gu",
    "qffn_decode_forward_noalloc", "QFFN_DECODE_WEIGHTS_STABLE",
]

QFFN_DECODE_WEIGHTS_STABLE = 1

STATUS = {0: "QFFN_OK", 1: "QFFN_ERR_INVALID_ARG", 2: "QFFN_ERR_UNSUPPORTED_SHAPE",
          3: "QFFN_ERR_MISALIGNED", 4: "QFFN_ERR_CUDA", 5: "QFFN_ERR_TIMEOUT"}

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is not built; run transformer_ffn_block_gb300._build.build() "
        "(or __graft_entry__.build()) first")

lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_S = ctypes.c_int

_SIGS = {
    "qffn_status_string": ([_S], ctypes.c_char_p),
    "qffn_abi_version": ([], ctypes.c_int),
    "qffn_check_status": ([_P], _S),
    "qffn_selftest_bounded_wait": ([_P, _S, _I64, _P], _S),
    "qffn_gemm_clock_sample": ([_P, _P], _S),
    "qffn_rmsnorm_absmax": ([_P, _P, _P, _P, _P, _P, _P, _F, _I64, _I64, _P], _S),
    "qffn_absmax": ([_P, _P, _I64, _P], _S),
    "qffn_quantize": ([_P, _P, _P, _I64, _P], _S),
    "qffn_quantize_rows": ([_P, _P, _P, _I64, _I64, _P], _S),
    "qffn_fp8_gemm_scaled": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _P], _S),
    "qffn_qmm": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P], _S),
    "qffn_gate_up_swiglu": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P], _S),
    "qffn_swiglu_quant": ([_P, _P, _P, _P, _I64, _I64, _P], _S),
    "qffn_swiglu_forward_quant": ([_P, _P, _P, _I64, _I64, _P], _S),
    "qffn_gate_up_swiglu_quant": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P], _S),
    "qffn_forward_workspace_size": ([_I64, _I64, _I64, _I64], _SZ),
    "qffn_forward_workspace_offsets": ([_I64, _I64, _I64, _I64, ctypes.POINTER(_SZ)], _S),
    "qffn_forward": ([_P, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P, _P, _P,
                      _I64, _I64, _I64, _I64, _P, _SZ, _P], _S),
    "qffn_forward_recompute": ([_P, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P, _P, _P,
                                _I64, _I64, _I64, _I64, _P, _SZ, _P], _S),
    "qffn_transpose_e4m3": ([_P, _P, _I64, _I64, _P], _S),
    "qffn_swiglu_backward": ([_P, _P, _P, _P, _I64, _I64, _P], _S),
    "qffn_backward_qmm_workspace_size": ([_I64, _I64, _I64], _SZ),
    "qffn_backward_qmm": ([_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _S, _P, _SZ, _P], _S),
    "qffn_ffn_backward_workspace_size": ([_I64, _I64, _I64], _SZ),
    "qffn_gate_up_swiglu_backward": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P], _S),
    "qffn_ffn_backward_workspace_offsets": ([_I64, _I64, _I64, ctypes.POINTER(_SZ)], _S),
    "qffn_ffn_backward": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                           _I64, _I64, _I64, _S, _P, _SZ, _P], _S),
    "qffn_gemv_dual": ([_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P], _S),
    "qffn_gemv": ([_P, _P, _P, _P, _I64, _I64, _P], _S),
    "qffn_gemv_silu_input": ([_P, _P, _P, _P, _P, _I64, _I64, _P], _S),
    "qffn_silu_mul": ([_P, _P, _I64, _P], _S),
    "qffn_decode_workspace_size": ([_I64, _I64], _SZ),
    "qffn_decode_workspace_offsets": ([_I64, _I64, _P], _S),
    "qffn_decode_forward": ([_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P], _S),
    "qffn_decode_forward_ex": ([_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, ctypes.c_uint, _P], _S),
    "qffn_decode_forward_gu": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P], _S),
    "qffn_decode_forward_noalloc": ([_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P], _S),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


class QffnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({qffn_status_string(status)})")


def _ptr(t):
    """torch tensor -> device address; int -> itself; None -> NULL."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != 0:
        raise QffnError(fn, status)


def qffn_status_string(status: int) -> str:
    return lib.qffn_status_string(status).decode()


def qffn_abi_version() -> int:
    return lib.qffn_abi_version()


def qffn_check_status(stream=None):
    _check("qffn_check_status", lib.qffn_check_status(_stream(stream)))


def qffn_selftest_bounded_wait(out, arrive, limit_ns, stream=None):
    _check("qffn_selftest_bounded_wait", lib.qffn_selftest_bounded_wait(
        _ptr(out), int(bool(arrive)), int(limit_ns), _stream(stream)))


def qffn_gemm_clock_sample(stream=None):
    """(SM clock cycles, nanoseconds) of the first CTA of the most recent GEMM launch."""
    out = (ctypes.c_uint64 * 2)()
    _check("qffn_gemm_clock_sample", lib.qffn_gemm_clock_sample(
        ctypes.cast(out, ctypes.c_void_p), _stream(stream)))
    return int(out[0]), int(out[1])


def qffn_rmsnorm_absmax(res_out, y, rstd, stats, res_in, x, gain, eps, N, C, stream=None):
    _check("qffn_rmsnorm_absmax", lib.qffn_rmsnorm_absmax(
        _ptr(res_out), _ptr(y), _ptr(rstd), _ptr(stats), _ptr(res_in), _ptr(x), _ptr(gain),
        float(eps), int(N), int(C), _stream(stream)))


def qffn_absmax(stats, inp, n, stream=None):
    _check("qffn_absmax", lib.qffn_absmax(_ptr(stats), _ptr(inp), int(n), _stream(stream)))


def qffn_quantize(q, stats, inp, n, stream=None):
    _check("qffn_quantize", lib.qffn_quantize(_ptr(q), _ptr(stats), _ptr(inp), int(n), _stream(stream)))


def qffn_quantize_rows(q, row_scale, w, rows, cols, stream=None):
    _check("qffn_quantize_rows", lib.qffn_quantize_rows(
        _ptr(q), _ptr(row_scale), _ptr(w), int(rows), int(cols), _stream(stream)))


def qffn_fp8_gemm_scaled(out, a, a_scale, w, w_scale, M, N, K, stream=None):
    _check("qffn_fp8_gemm_scaled", lib.qffn_fp8_gemm_scaled(
        _ptr(out), _ptr(a), _ptr(a_scale), _ptr(w), _ptr(w_scale), int(M), int(N), int(K),
        _stream(stream)))


def qffn_qmm(out, q, stats, inp, bias, w, w_scale, M, N, K, stream=None):
    _check("qffn_qmm", lib.qffn_qmm(
        _ptr(out), _ptr(q), _ptr(stats), _ptr(inp), _ptr(bias), _ptr(w), _ptr(w_scale),
        int(M), int(N), int(K), _stream(stream)))


def qffn_gate_up_swiglu(h, stats_h, yq, y_scale, w1, w1_scale, N, C, H, stream=None):
    _check("qffn_gate_up_swiglu", lib.qffn_gate_up_swiglu(
        _ptr(h), _ptr(stats_h), _ptr(yq), _ptr(y_scale), _ptr(w1), _ptr(w1_scale),
        int(N), int(C), int(H), _stream(stream)))


def qffn_swiglu_quant(h, hq, stats, gate_up, N, H, stream=None):
    _check("qffn_swiglu_quant", lib.qffn_swiglu_quant(
        _ptr(h), _ptr(hq), _ptr(stats), _ptr(gate_up), int(N), int(H), _stream(stream)))


def qffn_swiglu_forward_quant(hq, stats, gate_up, N, H, stream=None):
    _check("qffn_swiglu_forward_quant", lib.qffn_swiglu_forward_quant(
        _ptr(hq), _ptr(stats), _ptr(gate_up), int(N), int(H), _stream(stream)))


def qffn_gate_up_swiglu_quant(hq, stats_h, yq, y_scale, w1, w1_scale, N, C, H, stream=None):
    _check("qffn_gate_up_swiglu_quant", lib.qffn_gate_up_swiglu_quant(
        _ptr(hq), _ptr(stats_h), _ptr(yq), _ptr(y_scale), _ptr(w1), _ptr(w1_scale),
        int(N), int(C), int(H), _stream(stream)))


def qffn_forward_workspace_size(B, T, C, H) -> int:
    return int(lib.qffn_forward_workspace_size(int(B), int(T), int(C), int(H)))


def qffn_forward_workspace_offsets(B, T, C, H) -> list[int]:
    off = (_SZ * 4)()
    _check("qffn_forward_workspace_offsets",
           lib.qffn_forward_workspace_offsets(int(B), int(T), int(C), int(H), off))
    return [int(v) for v in off]


def qffn_forward(res_out, out, rstd, stats_y, stats_h, res_in, x, gain, eps, w1, w1_scale,
                 w2, w2_scale, B, T, C, H, workspace, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("qffn_forward", lib.qffn_forward(
        _ptr(res_out), _ptr(out), _ptr(rstd), _ptr(stats_y), _ptr(stats_h), _ptr(res_in),
        _ptr(x), _ptr(gain), float(eps), _ptr(w1), _ptr(w1_scale), _ptr(w2), _ptr(w2_scale),
        int(B), int(T), int(C), int(H), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def qffn_forward_recompute(res_out, out, rstd, stats_y, stats_h, res_in, x, gain, eps, w1,
                           w1_scale, w2, w2_scale, B, T, C, H, workspace, workspace_bytes=None,
                           stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("qffn_forward_recompute", lib.qffn_forward_recompute(
        _ptr(res_out), _ptr(out), _ptr(rstd), _ptr(stats_y), _ptr(stats_h), _ptr(res_in),
        _ptr(x), _ptr(gain), float(eps), _ptr(w1), _ptr(w1_scale), _ptr(w2), _ptr(w2_scale),
        int(B), int(T), int(C), int(H), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def qffn_transpose_e4m3(out, inp, rows, cols, stream=None):
    _check("qffn_transpose_e4m3", lib.qffn_transpose_e4m3(
        _ptr(out), _ptr(inp), int(rows), int(cols), _stream(stream)))


def qffn_swiglu_backward(d_gate_up, stats, dh, gate_up, N, H, stream=None):
    _check("qffn_swiglu_backward", lib.qffn_swiglu_backward(
        _ptr(d_gate_up), _ptr(stats), _ptr(dh), _ptr(gate_up), int(N), int(H), _stream(stream)))


def qffn_backward_qmm_workspace_size(N, IC, OC) -> int:
    return int(lib.qffn_backward_qmm_workspace_size(int(N), int(IC), int(OC)))


def qffn_backward_qmm(dinp, dw, stats_dout, dout, inp_q, inp_scale, w, w_scale, N, IC, OC,
                      accumulate, workspace, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("qffn_backward_qmm", lib.qffn_backward_qmm(
        _ptr(dinp), _ptr(dw), _ptr(stats_dout), _ptr(dout), _ptr(inp_q), _ptr(inp_scale), _ptr(w),
        _ptr(w_scale), int(N), int(IC), int(OC), int(bool(accumulate)), _ptr(workspace),
        int(workspace_bytes), _stream(stream)))


def qffn_ffn_backward_workspace_size(N, C, H) -> int:
    return int(lib.qffn_ffn_backward_workspace_size(int(N), int(C), int(H)))


def qffn_gate_up_swiglu_backward(d_gate_up, stats, dh, yq, y_scale, w1, w1_scale, N, C, H,
                                 stream=None):
    _check("qffn_gate_up_swiglu_backward", lib.qffn_gate_up_swiglu_backward(
        _ptr(d_gate_up), _ptr(stats), _ptr(dh), _ptr(yq), _ptr(y_scale), _ptr(w1), _ptr(w1_scale),
        int(N), int(C), int(H), _stream(stream)))


def qffn_ffn_backward_workspace_offsets(N, C, H) -> list[int]:
    off = (_SZ * 2)()
    _check("qffn_ffn_backward_workspace_offsets",
           lib.qffn_ffn_backward_workspace_offsets(int(N), int(C), int(H), off))
    return [int(v) for v in off]


def qffn_ffn_backward(d_ln2, dw1, dw2, stats_dout, stats_dgu, dout, yq, y_scale, hq, h_scale, w1,
                      w1_scale, w2, w2_scale, N, C, H, accumulate, workspace, workspace_bytes=None,
                      stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("qffn_ffn_backward", lib.qffn_ffn_backward(
        _ptr(d_ln2), _ptr(dw1), _ptr(dw2), _ptr(stats_dout), _ptr(stats_dgu), _ptr(dout), _ptr(yq),
        _ptr(y_scale), _ptr(hq), _ptr(h_scale), _ptr(w1), _ptr(w1_scale), _ptr(w2), _ptr(w2_scale),
        int(N), int(C), int(H), int(bool(accumulate)), _ptr(workspace), int(workspace_bytes),
        _stream(stream)))


def qffn_gemv_dual(g, u, x, w_gate, s_gate, w_up, s_up, H, C, stream=None):
    _check("qffn_gemv_dual", lib.qffn_gemv_dual(
        _ptr(g), _ptr(u), _ptr(x), _ptr(w_gate), _ptr(s_gate), _ptr(w_up), _ptr(s_up),
        int(H), int(C), _stream(stream)))


def qffn_gemv(out, x, w, row_scale, rows, cols, stream=None):
    _check("qffn_gemv", lib.qffn_gemv(
        _ptr(out), _ptr(x), _ptr(w), _ptr(row_scale), int(rows), int(cols), _stream(stream)))


def qffn_gemv_silu_input(out, g, u, w, row_scale, rows, cols, stream=None):
    _check("qffn_gemv_silu_input", lib.qffn_gemv_silu_input(
        _ptr(out), _ptr(g), _ptr(u), _ptr(w), _ptr(row_scale), int(rows), int(cols),
        _stream(stream)))


def qffn_silu_mul(g, u, n, stream=None):
    _check("qffn_silu_mul", lib.qffn_silu_mul(_ptr(g), _ptr(u), int(n), _stream(stream)))


def qffn_decode_workspace_size(C, H) -> int:
    return int(lib.qffn_decode_workspace_size(int(C), int(H)))


def qffn_decode_workspace_offsets(C, H):
    """Byte offsets of h and u in the decode workspace."""
    off = (ctypes.c_size_t * 2)()
    _check("qffn_decode_workspace_offsets", lib.qffn_decode_workspace_offsets(int(C), int(H), off))
    return [int(off[0]), int(off[1])]


def qffn_decode_forward(out, x, w_gate, s_gate, w_up, s_up, w_down, s_down, C, H, workspace,
                        workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("qffn_decode_forward", lib.qffn_decode_forward(
        _ptr(out), _ptr(x), _ptr(w_gate), _ptr(s_gate), _ptr(w_up), _ptr(s_up), _ptr(w_down),
        _ptr(s_down), int(C), int(H), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def qffn_decode_forward_ex(out, x, w_gate, s_gate, w_up, s_up, w_down, s_down, C, H, workspace, flags,
                           workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("qffn_decode_forward_ex", lib.qffn_decode_forward_ex(
        _ptr(out), _ptr(x), _ptr(w_gate), _ptr(s_gate), _ptr(w_up), _ptr(s_up), _ptr(w_down),
        _ptr(s_down), int(C), int(H), _ptr(workspace), int(workspace_bytes), int(flags), _stream(stream)))


def qffn_decode_forward_gu(out, x, w_gu, gu_row_scale, w_down, s_down, C, H, workspace,
                           workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("qffn_decode_forward_gu", lib.qffn_decode_forward_gu(
        _ptr(out), _ptr(x), _ptr(w_gu), _ptr(gu_row_scale), _ptr(w_down), _ptr(s_down), int(C), int(H),
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def qffn_decode_forward_noalloc(out, x, w_gate, s_gate, w_up, s_up, w_down, s_down, C, H,
                                stream=None):
    """qffn_decode_forward for callers that cannot allocate: the scratch is a fixed array
    inside the library (C, H <= 32768); calls overlapping on the GPU race on it."""
    _check("qffn_decode_forward_noalloc", lib.qffn_decode_forward_noalloc(
        _ptr(out), _ptr(x), _ptr(w_gate), _ptr(s_gate), _ptr(w_up), _ptr(s_up), _ptr(w_down),
        _ptr(s_down), int(C), int(H), _stream(stream)))
