"""Helpers shared by the GPU parity tests (host <-> device marshalling, tolerances)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def dev(a, dtype=None):
    """numpy array -> contiguous CUDA tensor with the same bits."""
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = t.view(torch.int16)
    if dtype is not None and t.dtype != dtype:
        t = t.view(dtype)
    return t.to(DEV)


def host(t, np_dtype=None):
    a = t.detach().cpu().numpy()
    if np_dtype is not None:
        a = a.view(np_dtype)
    return a


def bf(t):
    """CUDA int16 tensor of bf16 bits -> numpy uint16."""
    return host(t, np.uint16)


def empty_bf16(*shape):
    return torch.empty(*shape, dtype=torch.int16, device=DEV)


def empty_u8(*shape):
    return torch.empty(*shape, dtype=torch.uint8, device=DEV)


def bf16_ulp_diff(a_bits, b_bits):
    """Distance in bf16 units in the last place between two bf16 bit arrays (finite values)."""
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    # map sign-magnitude to a monotone integer line
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)


def e4m3_step_diff(a, b):
    """Distance in E4M3 code steps (finite codes)."""
    a = a.astype(np.int32)
    b = b.astype(np.int32)
    a = np.where(a & 0x80, -(a & 0x7F), a)
    b = np.where(b & 0x80, -(b & 0x7F), b)
    return np.abs(a - b)


def assert_out_close(got_bits, want_bits, rel_l2=1e-2, max_abs_rms=5e-2):
    """The block-output acceptance rule: relative L2 <= 1e-2 and max|err| <= 5e-2 * rms(want)."""
    g = oracle.bf16_to_f64(got_bits)
    w = oracle.bf16_to_f64(want_bits)
    err = g - w
    nw = np.linalg.norm(w)
    rel = np.linalg.norm(err) / nw if nw > 0 else np.linalg.norm(err)
    rms = np.sqrt(np.mean(w * w)) if w.size else 0.0
    mx = np.max(np.abs(err)) if err.size else 0.0
    assert rel <= rel_l2, f"relative L2 {rel:.3e} > {rel_l2}"
    assert mx <= max_abs_rms * rms + 0.0, f"max abs err {mx:.3e} > {max_abs_rms} * rms {rms:.3e}"
    return rel, mx, rms


def sync():
    torch.cuda.synchronize()


def check_dot_outputs(got_bits, want_bits, absdot, K, max_mismatch):
    """Outputs of fp32-accumulated dot products against the exact-then-rounded values:
    |got - want| <= 1 bf16 ulp + K * 2**-22 * absdot (absdot = scale * sum|terms|), and at
    most `max_mismatch` of the outputs differ at all."""
    g = oracle.bf16_to_f64(got_bits)
    w = oracle.bf16_to_f64(want_bits)
    big = np.maximum(np.abs(g), np.abs(w))
    ulp = np.ldexp(1.0, np.frexp(np.maximum(big, 1e-30))[1] - 8)
    bound = ulp + K * 2.0 ** -22 * absdot
    err = np.abs(g - w)
    frac = float(np.mean(got_bits != want_bits))
    assert np.all(err <= bound), (float(np.max(err / bound)), frac)
    assert frac <= max_mismatch, frac
    return frac
