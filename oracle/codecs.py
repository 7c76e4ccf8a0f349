"""Software codecs for the two storage formats of the FFN block (oracle side).

TEST INFRASTRUCTURE: part of the CPU oracle; see ``oracle/__init__.py``.

* bf16 -- the model dtype of every activation buffer in the trainer
  (llmq "llama_run_state.cpp", ``allocate_basic_fwd_tensors``: ln2, mlp_up,
  swiglu and mlp_down are ``Config.DType``).  Format: IEEE-754 binary32 with
  the low 16 mantissa bits dropped (1 sign, 8 exponent bits with bias 127,
  7 stored mantissa bits).  Rounding: to nearest, ties to even.
* e4m3 -- the FP8 ``matmul_dtype`` of the quantised copies ``ln2.q`` and
  ``swiglu.q`` (``allocate_fwd_quant_tensors``) and of the decode weights
  (metrale "dense_ffn_decode.rs", ``fp8w.*_proj.weight``).  Format: OCP
  8-bit floating point E4M3 ("fn" flavour): 1 sign, 4 exponent bits with
  bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
  ``m * 2**-9``; the all-ones pattern ``S.1111.111`` is NaN; there is no
  infinity, so the largest finite magnitude is ``1.75 * 2**8 = 448``.
  Encoding rounds to nearest, ties to even, and saturates to +-448
  ("satfinite") instead of overflowing.

Everything here is written from those format definitions with power-of-two
scalings (``np.ldexp``), ``np.frexp`` and ``np.rint`` (round half to even);
no hardware conversion routine is imitated.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0

# Element-wise conversions of large arrays run over flat slices of this many
# elements, only to bound the size of the float64 temporaries.
_CHUNK = 1 << 22


def _chunked(fn, x, out_dtype):
    x = np.asarray(x)
    if x.size <= _CHUNK:
        return fn(x)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=out_dtype)
    for i in range(0, flat.size, _CHUNK):
        out[i:i + _CHUNK] = fn(flat[i:i + _CHUNK])
    return out.reshape(x.shape)


# --------------------------------------------------------------------- bf16
def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float32 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even), one rounding."""
    return _chunked(_f64_to_bf16, x, np.uint16)


def _f64_to_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even), one rounding.

    A bf16 normal number has 8 significant bits, so in the binade
    ``[2**(e-1), 2**e)`` (``np.frexp`` exponent ``e``) the spacing is
    ``2**(e-8)``; below the smallest normal ``2**-126`` the spacing stays at
    the subnormal quantum ``2**-133``.  Dividing by the spacing, rounding to
    an integer with ties to even and multiplying back gives the rounded value
    exactly; magnitudes that round past the largest finite bf16 become inf.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)
        q_exp = np.maximum(e - 8, -133)
        q = np.ldexp(np.rint(np.ldexp(x, -q_exp)), q_exp)
        f32 = q.astype(np.float32)  # exact: q has at most 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def f32_to_bf16(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even)."""
    return f64_to_bf16(np.asarray(x, dtype=np.float32).astype(np.float64))


# --------------------------------------------------------------------- e4m3
def _e4m3_field_value(codes) -> np.ndarray:
    """E4M3 bit patterns -> exact float64 values, from the sign/exponent/mantissa fields."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    # normal: (1 + m/8) * 2**(e-7) = (8 + m) * 2**(e-10); subnormal: m * 2**-9
    mag = np.where(e == 0, np.ldexp(m.astype(np.float64), -9),
                   np.ldexp((8 + m).astype(np.float64), e - 10))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


# value of every one of the 256 codes, by the field definition above
_E4M3_VALUES = _e4m3_field_value(np.arange(256, dtype=np.uint8))


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 bit patterns (uint8) -> exact float64 values (NaN for 0x7F/0xFF)."""
    return _E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def e4m3_to_scaled_int(codes) -> np.ndarray:
    """E4M3 values times 2**9, as float64 holding integers (|v| <= 229376).

    Every finite E4M3 value is an integer multiple of the smallest subnormal
    ``2**-9``; the largest, 448, is ``229376 * 2**-9``.
    """
    return np.ldexp(e4m3_decode(codes), 9)


def e4m3_encode(v) -> np.ndarray:
    """Round float values to E4M3 codes: nearest, ties to even, satfinite."""
    return _chunked(_e4m3_encode, v, np.uint8)


def _e4m3_encode(v) -> np.ndarray:
    """Round float values to E4M3 codes: nearest, ties to even, satfinite.

    For ``|v|`` in the binade ``[2**E, 2**(E+1))`` with ``E >= -6`` the
    spacing of E4M3 values is ``2**(E-3)`` (3 mantissa bits); below the
    smallest normal ``2**-6`` it is the subnormal quantum ``2**-9``.  The
    magnitude is rounded on that grid (ties to even) and clamped to 448.
    NaN inputs give the NaN code 0x7F (with the input's sign bit).
    """
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(a)            # a = f * 2**e, f in [0.5, 1)  => E = e - 1
        q_exp = np.maximum(e - 1, -6) - 3
        q = np.ldexp(np.rint(np.ldexp(a, -q_exp)), q_exp)
        q = np.minimum(q, E4M3_MAX)
        # encode the rounded magnitude
        sub = q < 2.0 ** -6
        code_sub = np.ldexp(q, 9)                      # 0..7
        _, e2 = np.frexp(np.where(sub, 1.0, q))
        E2 = e2 - 1
        mant = np.ldexp(np.where(sub, 1.0, q), -E2) * 8 - 8   # 0..7
        code_norm = (E2 + 7) * 8 + mant
    code = np.where(sub, code_sub, code_norm).astype(np.int64)
    code = np.where(nan, 0x7F, code)
    code = np.where(neg, code | 0x80, code)
    return code.astype(np.uint8)
