"""Codecs of the FFN block's two storage formats (oracle side).

TEST INFRASTRUCTURE: part of the CPU oracle; see ``oracle/__init__.py``.

The arithmetic lives in ``ffn_oracle.cpp`` (C++17): bf16 (binary32 with the
low 16 mantissa bits dropped) and OCP FP8 E4M3 ("fn": bias 7, subnormals
``m * 2**-9``, NaN at ``S.1111.111``, no infinity, largest finite 448),
decoded from their bit fields and encoded by rounding to nearest, ties to
even, on the format's grid (E4M3 saturating at +-448).  These functions
only marshal numpy arrays into those calls.
"""
from __future__ import annotations

import numpy as np

from ._lib import lib

E4M3_MAX = 448.0


def _p(a):
    return a.ctypes.data


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().orc_bf16_decode(_p(b), _p(out), b.size)
    return out


def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float32 values."""
    return bf16_to_f64(bits).astype(np.float32)       # exact: a bf16 value is a float32 value


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even), one rounding."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_bf16_round(_p(v), _p(out), v.size)
    return out


def f32_to_bf16(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even)."""
    return f64_to_bf16(np.asarray(x, dtype=np.float32).astype(np.float64))


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 bit patterns (uint8) -> exact float64 values (NaN for 0x7F/0xFF)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().orc_e4m3_decode(_p(c), _p(out), c.size)
    return out


def e4m3_to_scaled_int(codes) -> np.ndarray:
    """E4M3 values times 2**9, as float64 holding the integers (|v| <= 229376)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.int32)
    lib().orc_e4m3_scaled_int(_p(c), _p(out), c.size)
    return out.astype(np.float64)


def e4m3_encode(v) -> np.ndarray:
    """Round float values to E4M3 codes: nearest, ties to even, satfinite."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint8)
    lib().orc_e4m3_round(_p(a), _p(out), a.size)
    return out
