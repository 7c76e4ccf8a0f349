"""Pins for the oracle's FFN steps (CPU only).

Every step is checked against something other than itself: hand-worked
values (``tests/golden``), closed forms and invariants, and the exact
brute-force arithmetic of ``tests/brute.py`` on tiny inputs.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import brute
import oracle
from ffn_inputs import random_bf16, random_codes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf(vals):
    return oracle.f64_to_bf16(np.asarray(vals, dtype=np.float64))


def _mixed_bf16(shape, seed):
    """bf16 values spread over several decades, both signs."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(shape) * 10.0 ** rng.integers(-3, 3, shape)
    return _bf(v)


# ------------------------------------------------------------------ A1 RMSNorm
def test_rmsnorm_golden_hand_worked():
    with open(os.path.join(GOLDEN, "rmsnorm_hand.txt")) as f:
        rows = [l for l in f.read().splitlines() if l.strip() and not l.startswith("#")]
    for line in rows:
        lhs, rhs = line.split("|")
        r0, r1, g0, g1, eps = (float(t) for t in lhs.split())
        y0, y1, rstd = (float(t) for t in rhs.split())
        r, y, got_rstd, amax = oracle.residual_rmsnorm_absmax(None, _bf([[r0, r1]]), _bf([g0, g1]), eps)
        np.testing.assert_array_equal(oracle.bf16_to_f64(y)[0], [y0, y1])
        assert got_rstd[0] == np.float32(rstd)
        assert amax == np.float32(max(abs(y0), abs(y1)))


@pytest.mark.parametrize("with_res", [True, False])
def test_rmsnorm_matches_brute_force(with_res):
    N, C = 5, 24
    res = _mixed_bf16((N, C), 11) if with_res else None
    x = _mixed_bf16((N, C), 12)
    gain = _bf(1 + 0.1 * np.random.default_rng(13).standard_normal(C))
    eps = 1e-5
    r, y, rstd, amax = oracle.residual_rmsnorm_absmax(res, x, gain, eps)
    for i in range(N):
        br, by, brstd = brute.rmsnorm_row(None if res is None else res[i], x[i], gain, np.float32(eps))
        assert list(r[i]) == br
        assert list(y[i]) == by
        assert rstd[i] == np.float32(float(brstd))
    assert amax == np.float32(max(abs(float(brute.bf16_value(b))) for b in y.ravel()))


def test_rmsnorm_reads_rounded_residual():
    """R3: the norm reads bf16(res + x), not the unrounded sum (brute force decides)."""
    # x much smaller than res, so the rounding of the stored sum moves y
    rng = np.random.default_rng(21)
    for trial in range(200):
        C = 6
        res = _bf(rng.standard_normal((1, C)) * 3)
        x = _bf(rng.standard_normal((1, C)) * 0.01)
        gain = _bf(np.ones(C))
        r, y, _, _ = oracle.residual_rmsnorm_absmax(res, x, gain, 1e-5)
        _, by, _ = brute.rmsnorm_row(res[0], x[0], gain, np.float32(1e-5))
        assert list(y[0]) == by


def test_rmsnorm_unit_rms_invariant():
    x = random_bf16((64, 512), seed=3)
    gain = _bf(np.ones(512))
    for eps in (1e-5, 1e-2, 0.0):
        y64, rstd = oracle.rmsnorm_f64(x, gain, eps)
        ms = np.mean(oracle.bf16_to_f64(x) ** 2, axis=1)
        np.testing.assert_allclose(np.mean(y64 ** 2, axis=1), ms / (ms + np.float32(eps)), rtol=1e-12)


def test_rmsnorm_constant_row_closed_form():
    for c in (0.5, 3.0, -7.25, 1e-3):
        x = _bf(np.full((1, 128), c))
        cb = float(oracle.bf16_to_f64(x)[0, 0])
        eps = 1e-5
        _, y, _, _ = oracle.residual_rmsnorm_absmax(None, x, _bf(np.ones(128)), eps)
        want = cb / np.sqrt(cb * cb + float(np.float32(eps)))
        assert np.all(y == oracle.f64_to_bf16(np.array([want]))[0])


def test_residual_sum_is_single_rounding_of_exact_sum():
    a = random_bf16((200, 64), seed=8)
    b = random_bf16((200, 64), seed=9, std=0.3)
    r, _, _, _ = oracle.residual_rmsnorm_absmax(a, b, _bf(np.ones(64)), 1e-5)
    for i in range(0, 200, 37):
        for j in range(0, 64, 5):
            exact = brute.bf16_value(a[i, j]) + brute.bf16_value(b[i, j])
            assert int(r[i, j]) == brute.round_bf16(exact)


# ------------------------------------------------------------------ A2 quantize
def test_quantize_matches_brute_force():
    v = _mixed_bf16((300,), 31)
    amax = oracle.absmax(v)
    codes, scale = oracle.quantize_with_abs_max(v, amax)
    bcodes, bscale = brute.quantize(list(v), float(amax))
    assert list(codes) == bcodes
    assert Fraction(float(scale)) == bscale


def test_quantize_invariants():
    v = random_bf16((4096,), seed=33)
    amax = oracle.absmax(v)
    codes, scale = oracle.quantize_with_abs_max(v, amax)
    assert scale == np.float32(amax / np.float32(448))
    vals = oracle.bf16_to_f64(v)
    i = int(np.argmax(np.abs(vals)))
    assert codes[i] in (0x7E, 0xFE)
    # |dequant(q) - x*inv| <= half an E4M3 step at x*inv (scaled units)
    inv = float(np.float32(448) / np.float32(amax))
    scaled = (vals.astype(np.float32) * np.float32(inv)).astype(np.float64)
    deq = oracle.e4m3_decode(codes)
    step = np.where(np.abs(scaled) < 2 ** -6, 2.0 ** -9,
                    2.0 ** (np.floor(np.log2(np.maximum(np.abs(scaled), 2 ** -6))) - 3))
    assert np.all(np.abs(deq - scaled) <= step / 2 + 0.0)
    assert np.all(np.abs(deq) <= 448)


def test_quantize_zero_tensor():
    codes, scale = oracle.quantize_with_abs_max(np.zeros(100, np.uint16), np.float32(0))
    assert scale == np.float32(1.0)
    assert not codes.any()


def test_quantize_rows_equals_per_row_tensor_quantization():
    w = random_bf16((37, 96), seed=41, std=0.02)
    w[5] = 0                                   # an all-zero row
    codes, scales = oracle.quantize_rows(w)
    for i in range(37):
        c, s = oracle.quantize_with_abs_max(w[i], oracle.absmax(w[i]))
        np.testing.assert_array_equal(codes[i], c)
        assert scales[i] == s
    assert scales[5] == 1.0 and not codes[5].any()


# ------------------------------------------------------------------ A3/A5 GEMM
def test_gemm_matches_brute_force_nonsquare():
    a = random_codes((3, 40), seed=51)
    w = random_codes((5, 40), seed=52)
    sa, sw = np.float32(0.013), np.float32(0.0007)
    out = oracle.fp8_gemm_scaled(a, sa, w, sw)
    assert out.shape == (3, 5)
    assert out.tolist() == brute.gemm(a.tolist(), sa, w.tolist(), sw)


def test_gemm_identity_weight_closed_form():
    """W = 448 * I (code 0x7E on the diagonal): out = bf16(dequant(A) * sA * 448 * sW)."""
    K = 64
    a = random_codes((7, K), seed=53)
    w = np.zeros((K, K), np.uint8)
    np.fill_diagonal(w, 0x7E)
    sa, sw = np.float32(0.25), np.float32(1 / 448.0)
    out = oracle.fp8_gemm_scaled(a, sa, w, sw)
    want = oracle.f64_to_bf16(oracle.e4m3_decode(a) * 0.25 * 448.0 * float(np.float32(1 / 448.0)))
    # compared as values: a -0 code gives a +0 sum (IEEE: -0 + +0 = +0)
    np.testing.assert_array_equal(oracle.bf16_to_f64(out), oracle.bf16_to_f64(want))


def test_gemm_exact_at_largest_magnitudes():
    """All-448 operands at K = 2**14: the exact sum 448*448*K must come out exactly."""
    K = 1 << 14
    a = np.full((1, K), 0x7E, np.uint8)
    w = np.full((2, K), 0x7E, np.uint8)
    w[1, ::2] = 0xFE
    acc = oracle.e4m3_to_scaled_int(a) @ oracle.e4m3_to_scaled_int(w).T
    assert acc[0, 0] == 229376.0 ** 2 * K
    assert acc[0, 1] == 0.0
    out = oracle.fp8_gemm_scaled(a, np.float32(1), w, np.float32(1))
    assert oracle.bf16_to_f64(out)[0, 0] == 448.0 * 448.0 * K


# ------------------------------------------------------------------ A4 SwiGLU
def test_silu_identities():
    z = np.linspace(-30, 30, 1001)
    s = oracle.silu_f64(z)
    np.testing.assert_allclose(s - oracle.silu_f64(-z), z, rtol=0, atol=1e-12)
    assert oracle.silu_f64(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(oracle.silu_f64(np.array([40.0, 100.0])), [40.0, 100.0], rtol=1e-15)
    assert abs(oracle.silu_f64(np.array([-800.0]))[0]) == 0.0


def test_swiglu_matches_brute_force_and_gate_is_first_half():
    H = 12
    gu = _mixed_bf16((3, 2 * H), 61)
    h, amax = oracle.swiglu(gu, H)
    for i in range(3):
        for j in range(H):
            assert int(h[i, j]) == brute.silu_times(gu[i, j], gu[i, H + j])
    swapped = np.concatenate([gu[:, H:], gu[:, :H]], axis=1)
    assert not np.array_equal(oracle.swiglu(swapped, H)[0], h)
    assert amax == oracle.absmax(h)


def test_swiglu_quant_equals_two_pass():
    H = 256
    gu = random_bf16((16, 2 * H), seed=63, std=2.0)
    h, hq, stats = oracle.swiglu_quant(gu, H)
    h2, amax = oracle.swiglu(gu, H)
    q2, s2 = oracle.quantize_with_abs_max(h2, amax)
    np.testing.assert_array_equal(h, h2)
    np.testing.assert_array_equal(hq, q2)
    assert stats[0] == amax and stats[1] == s2


# ------------------------------------------------------------------ A1..A5 chain
def test_ffn_forward_tiny_brute_force_chain():
    """Whole prefill chain at N=2, C=8, H=4 against the brute-force steps."""
    N, C, H = 2, 8, 4
    res = _mixed_bf16((N, C), 71)
    x = _mixed_bf16((N, C), 72)
    gain = _bf(1 + 0.1 * np.random.default_rng(73).standard_normal(C))
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), 74, std=0.02))
    w2q, w2s = oracle.quantize_tensor(random_bf16((C, H), 75, std=0.02))
    eps = np.float32(1e-5)
    o = oracle.ffn_forward(res, x, gain, eps, w1q, w1s, w2q, w2s, H)

    ys = []
    for i in range(N):
        br, by, _ = brute.rmsnorm_row(res[i], x[i], gain, eps)
        assert list(o["r"][i]) == br
        ys.extend(by)
    amax_y = max(abs(brute.bf16_value(b)) for b in ys)
    yq, sy = brute.quantize(ys, float(amax_y))
    assert Fraction(float(o["stats_y"][0])) == amax_y and Fraction(float(o["stats_y"][1])) == sy
    yq = [yq[i * C:(i + 1) * C] for i in range(N)]
    assert o["yq"].tolist() == yq
    gu = brute.gemm(yq, float(sy), w1q.tolist(), w1s)
    assert o["gu"].tolist() == gu
    h = [[brute.silu_times(gu[i][j], gu[i][H + j]) for j in range(H)] for i in range(N)]
    assert o["h"].tolist() == h
    flat = [b for row in h for b in row]
    amax_h = max(abs(brute.bf16_value(b)) for b in flat)
    hq, sh = brute.quantize(flat, float(amax_h))
    hq = [hq[i * H:(i + 1) * H] for i in range(N)]
    assert o["hq"].tolist() == hq
    assert o["out"].tolist() == brute.gemm(hq, float(sh), w2q.tolist(), w2s)


# ------------------------------------------------------------------ A6..A8 decode
def test_decode_golden_hand_worked():
    vals = {}
    with open(os.path.join(GOLDEN, "decode_hand.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                vals[k] = [float(t) for t in v]
    x = _bf([1.0, -2.0])
    wg = np.array([[0x38, 0x40]], np.uint8)
    wu = np.array([[0x30, 0x38]], np.uint8)
    wd = np.array([[0x38], [0xB8]], np.uint8)
    o = oracle.decode_forward(x, wg, np.float32([0.5]), wu, np.float32([1.0]), wd, np.float32([2.0, 0.25]))
    for k in ("g", "u", "h", "out"):
        np.testing.assert_array_equal(oracle.bf16_to_f64(o[k]), vals[k])


def test_decode_matches_brute_force():
    C, H = 32, 6
    x = _mixed_bf16((C,), 81)
    wg, sg = random_codes((H, C), 82), np.float32(np.random.default_rng(83).uniform(1e-4, 1e-2, H))
    wu, su = random_codes((H, C), 84), np.float32(np.random.default_rng(85).uniform(1e-4, 1e-2, H))
    wd, sd = random_codes((C, H), 86), np.float32(np.random.default_rng(87).uniform(1e-4, 1e-2, C))
    o = oracle.decode_forward(x, wg, sg, wu, su, wd, sd)
    assert o["g"].tolist() == brute.gemv(x.tolist(), wg.tolist(), sg.tolist())
    assert o["u"].tolist() == brute.gemv(x.tolist(), wu.tolist(), su.tolist())
    assert o["h"].tolist() == [brute.silu_times(a, b) for a, b in zip(o["g"], o["u"])]
    assert o["out"].tolist() == brute.gemv(o["h"].tolist(), wd.tolist(), sd.tolist())


def test_decode_equals_prefill_gemm_semantics_at_one_token():
    """With x exactly an E4M3 value times a power of two and equal row scales, the
    row-scaled GEMV equals the per-tensor scaled FP8 GEMM at N = 1."""
    C, H = 128, 16
    xq = random_codes((1, C), 91)
    sx = np.float32(2.0 ** -5)
    x = oracle.f64_to_bf16(oracle.e4m3_decode(xq)[0] * float(sx))     # exact in bf16
    w = random_codes((H, C), 92)
    sw = np.float32(0.00123)
    g = oracle.gemv_row_scaled(x, w, np.full(H, sw, np.float32))
    np.testing.assert_array_equal(g, oracle.fp8_gemm_scaled(xq, sx, w, sw)[0])


# ------------------------------------------------------------------ recompute form (given abs-max)
def test_swiglu_forward_quant_given_absmax_matches_brute_force():
    """A4 with the abs-max given: the codes of the exact-arithmetic quantiser, also
    when the given abs-max is below the true one (every element beyond it saturates)."""
    H = 16
    gu = _mixed_bf16((4, 2 * H), 91)
    h, amax = oracle.swiglu(gu, H)
    # Fractions have no signed zero: an input of -0.0 (silu underflow) keeps its
    # sign in the E4M3 encoding (code 0x80) where the brute force says 0.
    negzero = [int(b) == 0x8000 for b in h.ravel()]
    for given in (amax, np.float32(amax * np.float32(0.25)), np.float32(amax * np.float32(3.0))):
        hq, scale = oracle.swiglu_forward_quant(gu, H, given)
        bq, bs = brute.quantize(list(h.ravel()), float(given))
        bq = [0x80 if nz else c for c, nz in zip(bq, negzero)]
        assert list(hq.ravel()) == bq
        assert Fraction(float(scale)) == bs
    # below the true abs-max: saturated codes are exactly the elements whose
    # fp32-scaled value is at or above 432 (the tie between 416 and 448 rounds to 448)
    given = np.float32(amax * np.float32(0.25))
    hq, _ = oracle.swiglu_forward_quant(gu, H, given)
    inv = Fraction(float(np.float32(448) / given))
    big = [abs(brute.f32(brute.bf16_value(int(b)) * inv)) >= 432 for b in h.ravel()]
    sat = [int(c) & 0x7F == 0x7E for c in hq.ravel()]
    assert any(big) and big == sat


def test_swiglu_forward_quant_zero_absmax():
    gu = _mixed_bf16((2, 16), 92)
    hq, scale = oracle.swiglu_forward_quant(gu, 8, np.float32(0))
    assert scale == np.float32(1.0) and not hq.any()


def test_recompute_with_recorded_absmax_equals_forward():
    """Re-running the chain with the abs-maxes a forward recorded reproduces it."""
    N, C, H = 24, 64, 128
    res, x = random_bf16((N, C), 93), random_bf16((N, C), 94)
    gain = _bf(1 + 0.1 * np.random.default_rng(95).standard_normal(C))
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), 96, std=0.02))
    w2q, w2s = oracle.quantize_tensor(random_bf16((C, H), 97, std=0.02))
    eps = np.float32(1e-5)
    f = oracle.ffn_forward(res, x, gain, eps, w1q, w1s, w2q, w2s, H)
    r = oracle.ffn_forward_recompute(res, x, gain, eps, w1q, w1s, w2q, w2s, H,
                                     f["stats_y"][0], f["stats_h"][0])
    for k in ("r", "y", "rstd", "stats_y", "yq", "gu", "hq", "stats_h", "out"):
        np.testing.assert_array_equal(r[k], f[k], err_msg=k)


def test_recompute_tiny_brute_force_chain():
    """Recompute chain at N=2, C=8, H=4 with abs-maxes unrelated to the data
    (one above, one below the recorded values) against the brute-force steps."""
    N, C, H = 2, 8, 4
    res, x = _mixed_bf16((N, C), 101), _mixed_bf16((N, C), 102)
    gain = _bf(1 + 0.1 * np.random.default_rng(103).standard_normal(C))
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), 104, std=0.02))
    w2q, w2s = oracle.quantize_tensor(random_bf16((C, H), 105, std=0.02))
    eps = np.float32(1e-5)
    f = oracle.ffn_forward(res, x, gain, eps, w1q, w1s, w2q, w2s, H)
    ay = np.float32(f["stats_y"][0] * np.float32(1.5))
    ah = np.float32(f["stats_h"][0] * np.float32(0.5))
    o = oracle.ffn_forward_recompute(res, x, gain, eps, w1q, w1s, w2q, w2s, H, ay, ah)
    ys = []
    for i in range(N):
        _, by, _ = brute.rmsnorm_row(res[i], x[i], gain, eps)
        ys.extend(by)
    yq, sy = brute.quantize(ys, float(ay))
    assert o["yq"].tolist() == [yq[i * C:(i + 1) * C] for i in range(N)]
    assert Fraction(float(o["stats_y"][1])) == sy
    gu = brute.gemm(o["yq"].tolist(), float(sy), w1q.tolist(), w1s)
    assert o["gu"].tolist() == gu
    h = [brute.silu_times(gu[i][j], gu[i][H + j]) for i in range(N) for j in range(H)]
    hq, sh = brute.quantize(h, float(ah))
    assert o["hq"].tolist() == [hq[i * H:(i + 1) * H] for i in range(N)]
    assert Fraction(float(o["stats_h"][1])) == sh
    assert o["out"].tolist() == brute.gemm(o["hq"].tolist(), float(sh), w2q.tolist(), w2s)


# ------------------------------------------------------------------ forward_qmm (attention projections)
def test_qmm_matches_brute_force_with_bias():
    """Quantise with the recorded abs-max, scaled FP8 matmul, bias before the one rounding."""
    M, K, N = 3, 24, 5
    x = _mixed_bf16((M, K), 111)
    amax = oracle.absmax(x)
    wq, ws = oracle.quantize_tensor(random_bf16((N, K), 112, std=0.02))
    bias = _mixed_bf16((N,), 113)
    out, codes, scale = oracle.qmm(x, amax, wq, ws, bias)
    bq, bs = brute.quantize(list(x.ravel()), float(amax))
    assert list(codes.ravel()) == bq and Fraction(float(scale)) == bs
    rows = [bq[i * K:(i + 1) * K] for i in range(M)]
    assert out.tolist() == brute.gemm_bias(rows, float(bs), wq.tolist(), ws, list(bias))
    # no bias: the plain scaled matmul of the same codes
    out0, _, _ = oracle.qmm(x, amax, wq, ws)
    assert out0.tolist() == brute.gemm(rows, float(bs), wq.tolist(), ws)
    assert not np.array_equal(out0, out)


def test_qmm_identity_weight_closed_form():
    """W = 448 * I with scale 1/448: out = bf16(dequant(q) * scale + bias)."""
    K = 32
    x = _mixed_bf16((4, K), 114)
    amax = oracle.absmax(x)
    w = np.zeros((K, K), np.uint8)
    np.fill_diagonal(w, 0x7E)
    bias = _mixed_bf16((K,), 115)
    out, codes, scale = oracle.qmm(x, amax, w, np.float32(1 / 448.0), bias)
    want = oracle.f64_to_bf16(oracle.e4m3_decode(codes) * float(scale) * 448.0 * float(np.float32(1 / 448.0))
                              + oracle.bf16_to_f64(bias)[None, :])
    np.testing.assert_array_equal(out, want)


# ------------------------------------------------------------------ FFN backward (FP8)
def test_swiglu_backward_matches_brute_force_and_layout():
    H = 10
    gu = _mixed_bf16((3, 2 * H), 121)
    dh = _mixed_bf16((3, H), 122)
    d, amax = oracle.swiglu_backward(dh, gu, H)
    for i in range(3):
        for j in range(H):
            dg, du = brute.swiglu_grad(dh[i, j], gu[i, j], gu[i, H + j])
            assert int(d[i, j]) == dg and int(d[i, H + j]) == du
    assert amax == oracle.absmax(d)


def test_swiglu_backward_derivative_by_finite_difference():
    """The gate gradient is dh times the derivative of silu(g) * u, checked by a
    central difference (not by the closed form)."""
    H = 64
    gu = random_bf16((4, 2 * H), seed=123, std=2.0)
    dh = random_bf16((4, H), seed=124)
    d, _ = oracle.swiglu_backward(dh, gu, H)
    fd = np.array([[brute.silu_times_u_fd(gu[i, j], gu[i, H + j], dh[i, j]) for j in range(H)]
                   for i in range(4)], dtype=np.uint16)
    from gpu_util import bf16_ulp_diff
    diff = bf16_ulp_diff(d[:, :H], fd)
    assert diff.max() <= 1 and (diff == 0).mean() >= 0.98
    # du is dh * silu(g), the forward's product with u replaced by dh
    np.testing.assert_array_equal(d[:, H:], oracle.swiglu(np.concatenate([gu[:, :H], dh], axis=1), H)[0])


def test_backward_qmm_matches_brute_force():
    """dgrad over the output channels, wgrad over the tokens, and wgrad accumulation."""
    N, IC, OC = 4, 16, 6
    dout = _mixed_bf16((N, OC), 125)
    amax = oracle.absmax(dout)
    inq, ins = oracle.quantize_tensor(_mixed_bf16((N, IC), 126))
    wq, ws = oracle.quantize_tensor(random_bf16((OC, IC), 127, std=0.02))
    old = _mixed_bf16((OC, IC), 128)
    dinp, dw, dq, ds = oracle.backward_qmm(dout, amax, inq, ins, wq, ws)
    _, dwa, _, _ = oracle.backward_qmm(dout, amax, inq, ins, wq, ws, old)
    bq, bs = brute.quantize(list(dout.ravel()), float(amax))
    rows = [bq[i * OC:(i + 1) * OC] for i in range(N)]
    assert dq.tolist() == rows and Fraction(float(ds)) == bs
    wt = [list(c) for c in zip(*wq.tolist())]                 # W^T: [IC][OC]
    assert dinp.tolist() == brute.gemm(rows, float(bs), wt, ws)
    dqt = [list(c) for c in zip(*rows)]                        # dout_q^T: [OC][N]
    int_ = [list(c) for c in zip(*inq.tolist())]               # inp^T: [IC][N]
    assert dw.tolist() == brute.gemm(dqt, float(bs), int_, ins)
    assert dwa.tolist() == brute.gemm_acc(dqt, float(bs), int_, ins, old.tolist())


def test_ffn_backward_tiny_brute_force_chain():
    N, C, H = 3, 8, 4
    dout = _mixed_bf16((N, C), 131)
    yq, sy = oracle.quantize_tensor(_mixed_bf16((N, C), 132))
    hq, sh = oracle.quantize_tensor(_mixed_bf16((N, H), 133))
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), 134, std=0.02))
    w2q, w2s = oracle.quantize_tensor(random_bf16((C, H), 135, std=0.02))
    amax = oracle.absmax(dout)
    o = oracle.ffn_backward(dout, amax, yq, sy, hq, sh, w1q, w1s, w2q, w2s, H)
    T = lambda m: [list(c) for c in zip(*m)]
    dq, ds = brute.quantize(list(dout.ravel()), float(amax))
    dq = [dq[i * C:(i + 1) * C] for i in range(N)]
    dh = brute.gemm(dq, float(ds), T(w2q.tolist()), w2s)
    assert o["dh"].tolist() == dh
    assert o["dw2"].tolist() == brute.gemm(T(dq), float(ds), T(hq.tolist()), sh)
    gu = brute.gemm(yq.tolist(), sy, w1q.tolist(), w1s)
    assert o["gu"].tolist() == gu
    dgu = [[0] * (2 * H) for _ in range(N)]
    for i in range(N):
        for j in range(H):
            dgu[i][j], dgu[i][H + j] = brute.swiglu_grad(dh[i][j], gu[i][j], gu[i][H + j])
    assert o["d_gu"].tolist() == dgu
    amax_g = max(abs(brute.bf16_value(b)) for row in dgu for b in row)
    assert Fraction(float(o["stats_dgu"][0])) == amax_g
    gq, gs = brute.quantize([b for row in dgu for b in row], float(amax_g))
    gq = [gq[i * 2 * H:(i + 1) * 2 * H] for i in range(N)]
    assert o["d_ln2"].tolist() == brute.gemm(gq, float(gs), T(w1q.tolist()), w1s)
    assert o["dw1"].tolist() == brute.gemm(T(gq), float(gs), T(yq.tolist()), sy)
