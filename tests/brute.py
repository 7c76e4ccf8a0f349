"""Brute-force exact arithmetic for tiny inputs: an independent check of the oracle.

Nothing here shares code with ``oracle/``.  Values are Python ``Fraction``s
(exact) or 60-digit ``Decimal``s where a square root or an exponential is
needed; rounding to bf16 / E4M3 is done by searching the list of every
representable value (built from the bit fields) for the nearest one, with
ties going to the value whose last mantissa bit is 0.  It is slow and only
meant for a few hundred values at a time.
"""
from __future__ import annotations

import bisect
from decimal import Decimal, getcontext
from fractions import Fraction

getcontext().prec = 60


def _bf16_value(bits: int) -> Fraction | None:
    s = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if e == 0xFF:
        return None                                   # inf / nan
    if e == 0:
        return s * Fraction(m, 128) * Fraction(2) ** -126
    return s * (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)


def _e4m3_value(code: int) -> Fraction | None:
    s = -1 if code & 0x80 else 1
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 15 and m == 7:
        return None                                   # nan
    if e == 0:
        return s * Fraction(m, 8) * Fraction(2) ** -6
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


# positive finite values with their codes, sorted
_BF16_POS = sorted((v, b) for b in range(0x0000, 0x7F80) if (v := _bf16_value(b)) is not None)
_E4M3_POS = sorted((v, c) for c in range(0x00, 0x7F) if (v := _e4m3_value(c)) is not None)
_BF16_VALS = [v for v, _ in _BF16_POS]
_E4M3_VALS = [v for v, _ in _E4M3_POS]


def bf16_value(bits: int) -> Fraction:
    v = _bf16_value(int(bits))
    if v is None:
        raise ValueError("non-finite bf16")
    return v


def e4m3_value(code: int) -> Fraction:
    v = _e4m3_value(int(code))
    if v is None:
        raise ValueError("nan e4m3")
    return v


def _nearest(vals, table, a: Fraction, sign_bit: int, top_bit_mask: int):
    i = bisect.bisect_left(vals, a)
    if i < len(vals) and vals[i] == a:
        return table[i][1] | sign_bit
    lo = table[i - 1] if i > 0 else None
    hi = table[i] if i < len(vals) else None
    if hi is None:
        return None
    if lo is None:
        return hi[1] | sign_bit
    dl, dh = a - lo[0], hi[0] - a
    if dl < dh:
        return lo[1] | sign_bit
    if dh < dl:
        return hi[1] | sign_bit
    # tie: even last mantissa bit
    return (lo[1] if lo[1] % 2 == 0 else hi[1]) | sign_bit


def round_bf16(v) -> int:
    """Exact value -> nearest bf16 bits (ties to even).  Overflow is not handled."""
    v = Fraction(v)
    sign = 0x8000 if v < 0 else 0
    r = _nearest(_BF16_VALS, _BF16_POS, abs(v), sign, 0)
    if r is None:
        raise OverflowError
    return r


def round_e4m3_satfinite(v) -> int:
    """Exact value -> nearest E4M3 code (ties to even), clamped to +-448."""
    v = Fraction(v)
    sign = 0x80 if v < 0 else 0
    a = abs(v)
    if a >= 448:
        return 0x7E | sign
    return _nearest(_E4M3_VALS, _E4M3_POS, a, sign, 0)


def to_fraction(d: Decimal) -> Fraction:
    return Fraction(d)


def f32(v) -> Fraction:
    """Round an exact value to binary32 (nearest even) by brute force on the binade."""
    v = Fraction(v)
    if v == 0:
        return Fraction(0)
    s = -1 if v < 0 else 1
    a = abs(v)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    # a in [1, 2): 24 significant bits
    e_eff = max(e, -126)
    q = Fraction(2) ** (e_eff - 23)
    n = abs(v) / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return s * fl * q


# ------------------------------------------------------------------ block steps
def rmsnorm_row(res_bits, x_bits, gain_bits, eps) -> tuple[list[int], list[int], Decimal]:
    """One row of fused residual + RMSNorm: (r bits, y bits, rstd as Decimal)."""
    if res_bits is None:
        r = [int(b) for b in x_bits]
    else:
        r = [round_bf16(bf16_value(a) + bf16_value(b)) for a, b in zip(res_bits, x_bits)]
    rv = [bf16_value(b) for b in r]
    ms = sum(v * v for v in rv) / len(rv)
    eps_f = Fraction(float(eps))
    denom = Decimal(ms.numerator) / Decimal(ms.denominator) + Decimal(eps_f.numerator) / Decimal(eps_f.denominator)
    rstd = Decimal(1) / denom.sqrt()
    rstd_f = Fraction(rstd)
    y = [round_bf16(v * rstd_f * bf16_value(g)) for v, g in zip(rv, gain_bits)]
    return r, y, rstd


def quantize(v_bits, amax_f32: float) -> tuple[list[int], Fraction]:
    """Per-tensor E4M3 quantisation with fp32 scale and fp32 element products."""
    amax = Fraction(float(amax_f32))
    if amax == 0:
        return [0 for _ in v_bits], Fraction(1)
    scale = f32(amax / 448)
    inv = f32(Fraction(448) / amax)
    codes = [round_e4m3_satfinite(f32(bf16_value(b) * inv)) for b in v_bits]
    return codes, scale


def gemm(a_codes, a_scale, w_codes, w_scale):
    """out[m][n] = bf16(sa * sw * sum_k A[m][k] * W[n][k]), exact sums."""
    sa, sw = Fraction(float(a_scale)), Fraction(float(w_scale))
    out = []
    for arow in a_codes:
        av = [e4m3_value(c) for c in arow]
        orow = []
        for wrow in w_codes:
            acc = sum(x * e4m3_value(c) for x, c in zip(av, wrow))
            orow.append(round_bf16(acc * sa * sw))
        out.append(orow)
    return out


def gemm_bias(a_codes, a_scale, w_codes, w_scale, bias_bits):
    """out[m][n] = bf16(sa * sw * sum_k A[m][k] * W[n][k] + bias[n]), exact sums, one rounding."""
    sa, sw = Fraction(float(a_scale)), Fraction(float(w_scale))
    bias = [bf16_value(b) for b in bias_bits]
    out = []
    for arow in a_codes:
        av = [e4m3_value(c) for c in arow]
        out.append([round_bf16(sum(x * e4m3_value(c) for x, c in zip(av, wrow)) * sa * sw + b)
                    for wrow, b in zip(w_codes, bias)])
    return out


def silu_times(g_bits: int, u_bits: int) -> int:
    g = Decimal(bf16_value(g_bits).numerator) / Decimal(bf16_value(g_bits).denominator)
    u = bf16_value(u_bits)
    s = g / (Decimal(1) + (-g).exp())
    return round_bf16(Fraction(s) * u)


def _dec(f: Fraction) -> Decimal:
    return Decimal(f.numerator) / Decimal(f.denominator)


def swiglu_grad(dh_bits: int, g_bits: int, u_bits: int) -> tuple[int, int]:
    """(dg, du) of h = silu(g) * u, from the closed-form derivative, each rounded once."""
    g, u, dh = _dec(bf16_value(g_bits)), bf16_value(u_bits), bf16_value(dh_bits)
    sig = Decimal(1) / (Decimal(1) + (-g).exp())
    dsilu = sig * (Decimal(1) + g * (Decimal(1) - sig))
    return round_bf16(Fraction(dsilu) * u * dh), round_bf16(Fraction(g * sig) * dh)


def silu_times_u_fd(g_bits: int, u_bits: int, dh_bits: int) -> int:
    """dh * d/dg [silu(g) * u] by a central difference (60-digit decimals, step 1e-18), rounded once."""
    g, u, dh = _dec(bf16_value(g_bits)), _dec(bf16_value(u_bits)), _dec(bf16_value(dh_bits))
    eps = Decimal(10) ** -18

    def f(z):
        return z / (Decimal(1) + (-z).exp()) * u
    return round_bf16(Fraction((f(g + eps) - f(g - eps)) / (2 * eps) * dh))


def gemm_acc(a_codes, a_scale, w_codes, w_scale, old_bits):
    """out[m][n] = bf16(old[m][n] + sa * sw * sum_k A[m][k] * W[n][k]), one rounding."""
    sa, sw = Fraction(float(a_scale)), Fraction(float(w_scale))
    out = []
    for arow, orow_old in zip(a_codes, old_bits):
        av = [e4m3_value(c) for c in arow]
        out.append([round_bf16(bf16_value(o) + sum(x * e4m3_value(c) for x, c in zip(av, wrow)) * sa * sw)
                    for wrow, o in zip(w_codes, orow_old)])
    return out


def gemv(x_bits, w_codes, row_scales):
    xv = [bf16_value(b) for b in x_bits]
    out = []
    for wrow, s in zip(w_codes, row_scales):
        acc = sum(e4m3_value(c) * x for c, x in zip(wrow, xv))
        out.append(round_bf16(Fraction(float(s)) * acc))
    return out
