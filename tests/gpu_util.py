"""Helpers shared by the GPU parity tests (host <-> device marshalling, tolerances)."""
from __future__ import annotations

import os

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


# Accumulation error per step, relative to the sum of |terms|.  The decode GEMVs
# accumulate exact products with round-to-nearest fp32 FMAs (at most half a unit
# in the last place, 2**-24, per step).  The tensor cores' FP8 accumulation is
# bounded here by a whole unit, 2**-23, per step (it is not documented as
# round-to-nearest, and measured errors exceed the 2**-24 bound).
ACC_REL_FMA = 2.0 ** -24
ACC_REL_TENSOR = 2.0 ** -23


def _bf16_spacing(v):
    """Spacing of bf16 values in the binade of |v| (the subnormal quantum below 2**-126)."""
    e = np.frexp(np.maximum(np.abs(v), 2.0 ** -126))[1]
    return np.ldexp(1.0, e - 8)


def check_dot_outputs(got_bits, exact, absdot, K, max_mismatch, acc_rel=ACC_REL_TENSOR, want_bits=None):
    """bf16 results of fp32-accumulated dot products against the exact value.

    ``exact`` is the unrounded fp64 value the oracle rounds once (the exact sum
    times the scales, plus a bias or a previous gradient where there is one);
    ``absdot`` = scales * sum |terms|; ``K`` terms per output.
    Rule 1, every output: the result is the bf16 rounding of a value within the
    accumulation bound of the exact one,
        |got - exact| <= spacing(got) / 2 + 2**-24 |got| + (K acc_rel + 2**-22) absdot
    (the 2**-24 |got| for the fp32 value that is rounded to bf16, the 2**-22
    absdot for the fp32 multiplications by the scales).
    Rule 2: at most ``max_mismatch`` of the outputs differ from the oracle's
    result ``want_bits`` (by default the bf16 rounding of ``exact``); one
    differing output is always allowed, so that a check of a few hundred
    outputs does not turn a fraction into a bar of zero.
    Returns the mismatch fraction."""
    exact = np.asarray(exact, dtype=np.float64)
    g = oracle.bf16_to_f64(got_bits)
    want = oracle.f64_to_bf16(exact) if want_bits is None else np.asarray(want_bits)
    bound = 0.5 * _bf16_spacing(g) + 2.0 ** -24 * np.abs(g) + (K * acc_rel + 2.0 ** -22) * absdot
    err = np.abs(g - exact)
    frac = float(np.mean(got_bits != want)) if want.size else 0.0
    ok = err <= bound
    if os.environ.get("QFFN_REPORT_PARITY"):
        print(f"[parity] K={K} outputs={got_bits.size} mismatch={frac:.2e} "
              f"max err/bound={float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0:.3f}")
    assert np.all(ok), (float(np.max(err / np.maximum(bound, 1e-300))), int(np.sum(~ok)), frac)
    n_diff = int(np.sum(got_bits != want)) if want.size else 0
    assert n_diff <= max(1, int(max_mismatch * want.size)), (frac, max_mismatch, K)
    return frac


def gemm_mismatch_bar(K):
    """Fraction of GEMM outputs that may differ from the exactly rounded value.

    An output differs when the exact value lies closer to a bf16 rounding
    boundary than the accumulation error.  Measured on the 8B, Qwen2.5-7B-shaped
    and Llama-3.2-1B workloads: at most 1e-4 for K <= 4096, 0.06% at K = 8192,
    0.11% at K = 14336 and 0.16% at K = 18944 (the long down projections, whose
    SwiGLU inputs cancel more).  The bar is 0.1% up to K = 8192 and 0.2% above.
    """
    return 1e-3 if K <= 8192 else 2e-3


def absdot_gemm(a_codes, sa, b_codes, sb):
    """scales * sum |terms| of out = A . B^T (the size of the accumulation error bound)."""
    return (np.abs(oracle.e4m3_decode(a_codes)) @ np.abs(oracle.e4m3_decode(b_codes)).T) * float(sa) * float(sb)


def check_codes_rule(got, want, max_frac=1e-3):
    """The FP8 code rule: at most 0.1% of E4M3 codes differ, each by at most one code step."""
    d = e4m3_step_diff(got, want)
    frac = float((d > 0).mean()) if d.size else 0.0
    assert frac <= max_frac and (d.max() if d.size else 0) <= 1, (frac, int(d.max()) if d.size else 0)
    return frac
