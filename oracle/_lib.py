"""Build and load the C++ oracle library (``liboracle.so``).

TEST INFRASTRUCTURE: part of the CPU oracle; see ``oracle/__init__.py``.

The library is compiled in-tree from ``ffn_oracle.cpp`` with the host C++
compiler (C++17, OpenMP, no floating-point contraction) the first time it is
needed or whenever the source is newer than the built file.  This module
only declares the C signatures for ``ctypes``; it does no arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ffn_oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")
CXXFLAGS = ["-std=c++17", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so if it is missing or older than its source; return its path."""
    with _lock:
        if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            cxx = os.environ.get("CXX") or shutil.which("g++") or shutil.which("c++")
            if cxx is None:
                raise RuntimeError("no C++ compiler found to build the oracle")
            tmp = LIB + f".tmp{os.getpid()}"
            r = subprocess.run([cxx, *CXXFLAGS, SRC, "-o", tmp], capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("building the oracle failed:\n" + r.stdout + r.stderr)
            os.replace(tmp, LIB)
    return LIB


_P = ctypes.c_void_p
_I = ctypes.c_int64
_F = ctypes.c_float

_SIGNATURES = {
    "orc_set_plant": (None, [ctypes.c_int]),
    "orc_get_plant": (ctypes.c_int, []),
    "orc_set_threads": (None, [ctypes.c_int]),
    "orc_max_threads": (ctypes.c_int, []),
    "orc_bf16_decode": (None, [_P, _P, _I]),
    "orc_bf16_round": (None, [_P, _P, _I]),
    "orc_e4m3_decode": (None, [_P, _P, _I]),
    "orc_e4m3_scaled_int": (None, [_P, _P, _I]),
    "orc_e4m3_round": (None, [_P, _P, _I]),
    "orc_silu": (None, [_P, _P, _I]),
    "orc_rmsnorm_f64": (None, [_P, _P, _F, _I, _I, _P, _P]),
    "orc_residual_rmsnorm_absmax": (None, [_P, _P, _P, _F, _I, _I, _P, _P, _P, _P]),
    "orc_absmax_bf16": (_F, [_P, _I]),
    "orc_quantize_with_abs_max": (None, [_P, _I, _F, _P, _P]),
    "orc_quantize_rows": (None, [_P, _I, _I, _P, _P]),
    "orc_fp8_gemm": (ctypes.c_int, [_P, _I, _I, _F, _P, _I, _I, _F, _I, _I, _I, _P, _P, _P]),
    "orc_fp8_gemm_exact": (ctypes.c_int, [_P, _I, _I, _F, _P, _I, _I, _F, _I, _I, _I, _P]),
    "orc_swiglu": (None, [_P, _I, _I, _P, _P]),
    "orc_silu_mul": (None, [_P, _P, _I, _P]),
    "orc_swiglu_backward": (None, [_P, _P, _I, _I, _P, _P]),
    "orc_ffn_forward": (ctypes.c_int, [_P, _P, _P, _F, _P, _F, _P, _F, _I, _I, _I,
                                       _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "orc_ffn_forward_recompute": (ctypes.c_int, [_P, _P, _P, _F, _P, _F, _P, _F, _I, _I, _I, _F, _F,
                                                 _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "orc_backward_qmm": (ctypes.c_int, [_P, _F, _P, _F, _P, _F, _I, _I, _I, _P, _P, _P, _P, _P]),
    "orc_ffn_backward": (ctypes.c_int, [_P, _F, _P, _F, _P, _F, _P, _F, _P, _F, _I, _I, _I, _P, _P,
                                        _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "orc_gemv_row_scaled": (None, [_P, _P, _P, _I, _I, _P]),
    "orc_gemv_exact": (None, [_P, _P, _P, _I, _I, _P]),
    "orc_decode_forward": (None, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P]),
}


def lib() -> ctypes.CDLL:
    """The loaded oracle library (built first if needed)."""
    global _lib
    if _lib is None:
        path = build()
        l = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib
