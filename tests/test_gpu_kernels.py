"""Stage-wise GPU parity: each CUDA kernel, through the C ABI, against the oracle.

Every kernel is fed seeded inputs (or the GPU's own upstream tensors, so an
earlier 1-ulp difference does not propagate) and compared element by element:
integer/byte results bit-exact, bf16 results within the stated ulps.
"""
import numpy as np
import pytest
import torch

import oracle
from ffn_inputs import random_bf16, random_codes
from gpu_util import (ACC_REL_FMA, absdot_gemm, assert_out_close, bf, bf16_ulp_diff, check_dot_outputs, dev,
                      empty_bf16, empty_u8, gemm_mismatch_bar, host, sync)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import transformer_ffn_block_gb300 as q
    return q


def _mixed(shape, seed, spread=2):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(shape) * 10.0 ** rng.integers(-spread, spread + 1, shape)
    return oracle.f64_to_bf16(v)


# ------------------------------------------------------------------ A1
@pytest.mark.parametrize("N,C", [(1, 8), (3, 24), (64, 256), (257, 2048), (33, 3584), (5, 16384), (130, 4096)])
@pytest.mark.parametrize("with_res", [True, False])
def test_rmsnorm_absmax(q, N, C, with_res):
    res = random_bf16((N, C), seed=N * 7 + C) if with_res else None
    x = random_bf16((N, C), seed=N * 11 + C + 1)
    gain = oracle.f64_to_bf16(1 + 0.1 * np.random.default_rng(C).standard_normal(C))
    eps = 1e-5
    r_ref, y_ref, rstd_ref, amax_ref = oracle.residual_rmsnorm_absmax(res, x, gain, eps)

    res_out = empty_bf16(N, C) if with_res else None
    y = empty_bf16(N, C)
    rstd = torch.empty(N, dtype=torch.float32, device="cuda")
    stats = torch.full((2,), 123.0, dtype=torch.float32, device="cuda")
    q.qffn_rmsnorm_absmax(res_out, y, rstd, stats, None if res is None else dev(res), dev(x),
                          dev(gain), eps, N, C)
    sync()
    if with_res:
        np.testing.assert_array_equal(bf(res_out), r_ref)          # bit-exact
    yg = bf(y)
    # y is rounded once from an almost exact value: bit-identical to the oracle
    np.testing.assert_array_equal(yg, y_ref)
    np.testing.assert_allclose(host(rstd), rstd_ref, rtol=2.0 ** -23, atol=0)
    st = host(stats)
    assert st[0] == amax_ref
    assert st[1] == 123.0                                           # scale slot untouched


def test_rmsnorm_in_place_and_no_stats(q):
    N, C = 17, 512
    res = random_bf16((N, C), 1)
    x = random_bf16((N, C), 2)
    gain = random_bf16((C,), 3)
    r_ref, y_ref, _, _ = oracle.residual_rmsnorm_absmax(res, x, gain, 1e-6)
    xd = dev(x)
    y = empty_bf16(N, C)
    rstd = torch.empty(N, dtype=torch.float32, device="cuda")
    q.qffn_rmsnorm_absmax(xd, y, rstd, None, dev(res), xd, dev(gain), 1e-6, N, C)   # res_out aliases x
    sync()
    np.testing.assert_array_equal(bf(xd), r_ref)
    np.testing.assert_array_equal(bf(y), y_ref)


def test_rmsnorm_empty(q):
    stats = torch.full((2,), 5.0, dtype=torch.float32, device="cuda")
    y = empty_bf16(1, 256)
    rstd = torch.empty(1, dtype=torch.float32, device="cuda")
    q.qffn_rmsnorm_absmax(None, y, rstd, stats, None, y, y, 1e-5, 0, 256)
    sync()
    assert host(stats)[0] == 0.0


# ------------------------------------------------------------------ abs-max, A2
@pytest.mark.parametrize("n", [0, 1, 7, 8, 15, 16, 17, 4096, 100003, 1 << 22])
def test_absmax_and_quantize(q, n):
    v = _mixed((n,), n + 3)
    stats = torch.full((2,), 7.0, dtype=torch.float32, device="cuda")
    codes = empty_u8(max(n, 1))
    vd = dev(v) if n else empty_bf16(1)
    q.qffn_absmax(stats, vd, n)
    q.qffn_quantize(codes, stats, vd, n)
    sync()
    st = host(stats)
    amax = oracle.absmax(v)
    assert st[0] == amax
    ref_codes, ref_scale = oracle.quantize_with_abs_max(v, amax)
    assert st[1] == ref_scale
    np.testing.assert_array_equal(host(codes)[:n], ref_codes)


def test_quantize_zero_tensor_gives_zero_codes(q):
    n = 4096 + 5
    v = np.zeros(n, np.uint16)
    v[::3] = 0x8000                                  # -0.0 as well
    stats = torch.zeros(2, dtype=torch.float32, device="cuda")
    codes = torch.full((n,), 0x55, dtype=torch.uint8, device="cuda")
    vd = dev(v)
    q.qffn_absmax(stats, vd, n)
    q.qffn_quantize(codes, stats, vd, n)
    sync()
    assert host(stats).tolist() == [0.0, 1.0]
    assert not host(codes).any()


def test_quantize_saturation_edge(q):
    # values whose scaled product lands exactly on E4M3 ties and on 448
    v = oracle.f64_to_bf16(np.array([448.0, 1.0625, 1.1875, -3 * 2.0 ** -10, 2.0 ** -10, 0.0, -0.0, 447.0] * 4))
    stats = torch.tensor([448.0, 0.0], dtype=torch.float32, device="cuda")
    codes = empty_u8(v.size)
    q.qffn_quantize(codes, stats, dev(v), v.size)
    sync()
    ref, scale = oracle.quantize_with_abs_max(v, np.float32(448.0))
    np.testing.assert_array_equal(host(codes), ref)
    assert host(stats)[1] == scale == np.float32(1.0)


@pytest.mark.parametrize("rows,cols", [(1, 16), (37, 96), (300, 4096), (64, 14336)])
def test_quantize_rows(q, rows, cols):
    w = random_bf16((rows, cols), seed=rows + cols, std=0.02)
    w[rows // 2] = 0
    codes = empty_u8(rows, cols)
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    q.qffn_quantize_rows(codes, scales, dev(w), rows, cols)
    sync()
    rc, rs = oracle.quantize_rows(w)
    np.testing.assert_array_equal(host(codes), rc)
    np.testing.assert_array_equal(host(scales), rs)


# ------------------------------------------------------------------ A3/A5 GEMM
def _gemm_check(got, want, a, sa, w, sw, max_mismatch=None):
    """Every output within the accumulation bound of the exact value, and at most
    the K-dependent fraction differing from the exact-then-rounded value."""
    K = a.shape[1]
    return check_dot_outputs(got, oracle.fp8_gemm_exact(a, sa, w, sw), absdot_gemm(a, sa, w, sw), K,
                             gemm_mismatch_bar(K) if max_mismatch is None else max_mismatch, want_bits=want)


GEMM_SHAPES = [
    (1, 32, 16), (64, 256, 128), (128, 256, 128), (129, 288, 144), (300, 512, 512),
    (256, 768, 256), (200, 256, 4096), (130, 512, 14336), (1000, 1024, 2048),
    # more tiles than SM pairs with a short last wave, which runs as half tiles
    # (N = 128): 80 tiles, and 78 tiles whose split ones sit on a ragged
    # column edge (N = 416)
    (20480, 256, 64), (9984, 416, 96)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_fp8_gemm_scaled(q, M, N, K):
    """Activations and weights quantised from Gaussian data, as in the block."""
    a, sa = oracle.quantize_tensor(random_bf16((M, K), seed=M * 3 + K))
    w, sw = oracle.quantize_tensor(random_bf16((N, K), seed=N * 5 + K + 1, std=0.02))
    want = oracle.fp8_gemm_scaled(a, sa, w, sw)
    out = empty_bf16(M, N)
    scales = torch.tensor([sa, sw], dtype=torch.float32, device="cuda")
    q.qffn_fp8_gemm_scaled(out, dev(a), scales[0:1], dev(w), scales[1:2], M, N, K)
    q.qffn_check_status()
    sync()
    _gemm_check(bf(out), want, a, sa, w, sw)


@pytest.mark.parametrize("M,N,K", [(129, 288, 144), (200, 256, 4096), (64, 256, 14336)])
def test_fp8_gemm_random_codes_error_bound(q, M, N, K):
    """Uniformly random codes (heavy cancellation): every output within the accumulation
    bound of the exact value; the fraction of flipped roundings is not bounded here."""
    a = random_codes((M, K), seed=M * 3 + K)
    w = random_codes((N, K), seed=N * 5 + K + 1)
    sa, sw = np.float32(0.5 / 448), np.float32(0.02 / 448)
    want = oracle.fp8_gemm_scaled(a, sa, w, sw)
    out = empty_bf16(M, N)
    scales = torch.tensor([sa, sw], dtype=torch.float32, device="cuda")
    q.qffn_fp8_gemm_scaled(out, dev(a), scales[0:1], dev(w), scales[1:2], M, N, K)
    sync()
    _gemm_check(bf(out), want, a, sa, w, sw, max_mismatch=1.0)


def test_fp8_gemm_identity_weight(q):
    """W = 448 * I: out = bf16(dequant(A) * sA * 448 * sW) exactly."""
    M, K = 77, 256
    a = random_codes((M, K), 5)
    w = np.zeros((K, K), np.uint8)
    np.fill_diagonal(w, 0x7E)
    scales = torch.tensor([0.25, 1 / 448.0], dtype=torch.float32, device="cuda")
    out = empty_bf16(M, K)
    q.qffn_fp8_gemm_scaled(out, dev(a), scales[0:1], dev(w), scales[1:2], M, K, K)
    sync()
    want = oracle.fp8_gemm_scaled(a, np.float32(0.25), w, np.float32(1 / 448.0))
    np.testing.assert_array_equal(oracle.bf16_to_f64(bf(out)), oracle.bf16_to_f64(want))


def test_gemm_clock_sample(q):
    """The clock sample of a GEMM launch: positive SM cycles and nanoseconds whose ratio
    (the mean SM clock of the launch) lies in the part's range, and a later launch
    replaces the sample."""
    M = N = K = 2048
    a = random_codes((M, K), seed=91)
    w = random_codes((N, K), seed=92)
    scales = torch.tensor([0.5, 0.25], dtype=torch.float32, device="cuda")
    out = empty_bf16(M, N)
    q.qffn_fp8_gemm_scaled(out, dev(a), scales[0:1], dev(w), scales[1:2], M, N, K)
    cyc, ns = q.qffn_gemm_clock_sample()
    assert cyc > 0 and ns > 0
    assert 0.3 < cyc / ns < 2.5, (cyc, ns)
    out2 = empty_bf16(4 * M, N)
    q.qffn_fp8_gemm_scaled(out2, dev(np.concatenate([a] * 4)), scales[0:1], dev(w), scales[1:2], 4 * M, N, K)
    cyc2, ns2 = q.qffn_gemm_clock_sample()
    assert (cyc2, ns2) != (cyc, ns) and 0.3 < cyc2 / ns2 < 2.5, (cyc2, ns2)


# ------------------------------------------------------------------ A3+A4 fused
@pytest.mark.parametrize("N,C,H", [(64, 256, 768), (1, 128, 128), (200, 384, 256), (513, 2048, 1024),
                                   # 80 tiles: the last wave runs as half tiles (64 gate +
                                   # 64 up columns), the second with a ragged last M-block
                                   (5120, 64, 512), (4900, 96, 512),
                                   # K > 2048: the eight-column epilogue step (the shapes
                                   # above take the sixteen-column one), whole and half tiles
                                   (130, 2176, 384), (5120, 2304, 512)])
def test_gate_up_swiglu(q, N, C, H):
    """The fused epilogue equals SwiGLU applied to the GPU's own unfused gate|up GEMM
    (same accumulators, same bf16 rounding of g and u), within 1 ulp of the fp64 silu."""
    yq, sy = oracle.quantize_tensor(random_bf16((N, C), seed=N + C))
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), seed=H + C, std=0.02))
    scales = torch.tensor([sy, w1s], dtype=torch.float32, device="cuda")
    yqd, w1d = dev(yq), dev(w1q)
    h = empty_bf16(N, H)
    stats = torch.full((2,), 9.0, dtype=torch.float32, device="cuda")
    q.qffn_gate_up_swiglu(h, stats, yqd, scales[0:1], w1d, scales[1:2], N, C, H)
    gu = empty_bf16(N, 2 * H)
    q.qffn_fp8_gemm_scaled(gu, yqd, scales[0:1], w1d, scales[1:2], N, 2 * H, C)
    q.qffn_check_status()
    sync()
    hg = bf(h)
    h_stage, _ = oracle.swiglu(bf(gu), H)
    assert bf16_ulp_diff(hg, h_stage).max() <= 1
    st = host(stats)
    assert st[0] == np.float32(np.max(np.abs(oracle.bf16_to_f64(hg))))
    assert st[1] == 9.0
    # against the exact oracle end to end: the block-output tolerance
    h_ref, _ = oracle.swiglu(oracle.fp8_gemm_scaled(yq, sy, w1q, w1s), H)
    assert_out_close(hg, h_ref)


def test_gate_up_swiglu_gate_is_first_half(q):
    """Swapping the gate and up halves of W1 must change h (gate = rows [0, H))."""
    N, C, H = 64, 256, 256
    yq = random_codes((N, C), 1)
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), 2, std=0.02))
    want = oracle.swiglu(oracle.fp8_gemm_scaled(yq, np.float32(0.01), w1q, w1s), H)[0]
    scales = torch.tensor([0.01, w1s], dtype=torch.float32, device="cuda")
    h = empty_bf16(N, H)
    stats = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_gate_up_swiglu(h, stats, dev(yq), scales[0:1], dev(w1q), scales[1:2], N, C, H)
    sync()
    assert_out_close(bf(h), want)
    swapped = oracle.swiglu(oracle.fp8_gemm_scaled(yq, np.float32(0.01), np.concatenate([w1q[H:], w1q[:H]]), w1s), H)[0]
    with pytest.raises(AssertionError):
        assert_out_close(bf(h), swapped)


# ------------------------------------------------------------------ A4 standalone
@pytest.mark.parametrize("N,H", [(1, 8), (64, 768), (333, 1024), (16, 14336)])
def test_swiglu_quant(q, N, H):
    gu = _mixed((N, 2 * H), N + H, spread=1)
    h_ref, amax_ref = oracle.swiglu(gu, H)
    h = empty_bf16(N, H)
    hq = empty_u8(N, H)
    stats = torch.zeros(2, dtype=torch.float32, device="cuda")
    gud = dev(gu)
    q.qffn_swiglu_quant(h, hq, stats, gud, N, H)
    hq2 = empty_u8(N, H)
    stats2 = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_swiglu_quant(None, hq2, stats2, gud, N, H)          # recompute form
    sync()
    hg = bf(h)
    assert bf16_ulp_diff(hg, h_ref).max() <= 1
    st = host(stats)
    assert st[0] == np.float32(np.max(np.abs(oracle.bf16_to_f64(hg))))
    codes, scale = oracle.quantize_with_abs_max(hg, st[0])
    assert st[1] == scale
    np.testing.assert_array_equal(host(hq), codes)
    np.testing.assert_array_equal(host(hq2), host(hq))
    np.testing.assert_array_equal(host(stats2), st)


# ------------------------------------------------------------------ A6..A8
@pytest.mark.parametrize("rows,cols", [(1, 16), (100, 4096), (4096, 14336), (777, 640), (64, 32768)])
def test_gemv_and_dual_bit_identical(q, rows, cols):
    x = random_bf16((cols,), seed=cols)
    wg = random_codes((rows, cols), seed=rows + 1)
    wu = random_codes((rows, cols), seed=rows + 2)
    rng = np.random.default_rng(rows)
    sg = rng.uniform(1e-5, 1e-4, rows).astype(np.float32)
    su = rng.uniform(1e-5, 1e-4, rows).astype(np.float32)
    g = empty_bf16(rows)
    u = empty_bf16(rows)
    g1 = empty_bf16(rows)
    u1 = empty_bf16(rows)
    xd, wgd, wud, sgd, sud = dev(x), dev(wg), dev(wu), dev(sg), dev(su)
    q.qffn_gemv_dual(g, u, xd, wgd, sgd, wud, sud, rows, cols)
    q.qffn_gemv(g1, xd, wgd, sgd, rows, cols)
    q.qffn_gemv(u1, xd, wud, sud, rows, cols)
    sync()
    # the per-projection arm agrees bit for bit with the dual arm
    np.testing.assert_array_equal(bf(g1), bf(g))
    np.testing.assert_array_equal(bf(u1), bf(u))
    gr, ur = oracle.gemv_dual(x, wg, sg, wu, su)
    xa = np.abs(oracle.bf16_to_f64(x))
    for got, want, wq, sc in ((bf(g), gr, wg, sg), (bf(u), ur, wu, su)):
        absdot = (np.abs(oracle.e4m3_decode(wq)) @ xa) * sc.astype(np.float64)
        check_dot_outputs(got, oracle.gemv_exact(x, wq, sc), absdot, cols, 1e-3, acc_rel=ACC_REL_FMA,
                          want_bits=want)


@pytest.mark.parametrize("n", [8, 14336, 8 * 1001])
def test_silu_mul(q, n):
    g = _mixed((n,), n, spread=1)
    u = _mixed((n,), n + 1, spread=1)
    gd = dev(g)
    q.qffn_silu_mul(gd, dev(u), n)
    sync()
    assert bf16_ulp_diff(bf(gd), oracle.silu_mul(g, u)).max() <= 1
