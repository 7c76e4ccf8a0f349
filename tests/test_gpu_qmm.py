"""GPU parity of forward_qmm (qffn_qmm): quantisation with the recorded abs-max, then
the scaled FP8 matmul with an optional bias -- the attention projections of the
block (QKV of LN1, the attention output projection), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from ffn_inputs import random_bf16
from gpu_util import bf, check_dot_outputs, dev, empty_bf16, empty_u8, gemm_mismatch_bar, host, sync

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import transformer_ffn_block_gb300 as q
    return q


def _run(q, x, bias, wq, ws):
    M, K = x.shape
    N = wq.shape[0]
    xd = dev(x)
    stats = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_absmax(stats, xd, x.size)
    out = empty_bf16(M, N)
    qbuf = empty_u8(M, K)
    wsc = torch.tensor([ws], dtype=torch.float32, device="cuda")
    q.qffn_qmm(out, qbuf, stats, xd, None if bias is None else dev(bias), dev(wq), wsc, M, N, K)
    q.qffn_check_status()
    sync()
    return bf(out), host(qbuf), host(stats)


@pytest.mark.parametrize("M,N,K,with_bias", [(64, 384, 256, True), (129, 288, 144, False),
                                             (1000, 3072, 2048, True), (300, 4096, 4096, False)])
def test_qmm_parity(q, M, N, K, with_bias):
    x = random_bf16((M, K), seed=M + N + K)
    wq, ws = oracle.quantize_tensor(random_bf16((N, K), seed=N * 3 + K, std=0.02))
    bias = random_bf16((N,), seed=N + 7, std=0.5) if with_bias else None
    out, codes, st = _run(q, x, bias, wq, ws)
    amax = oracle.absmax(x)
    want, rcodes, rscale = oracle.qmm(x, amax, wq, ws, bias)
    assert st[0] == amax and st[1] == rscale                 # abs-max and scale bit-exact
    np.testing.assert_array_equal(codes, rcodes)             # codes bit-exact
    absdot = (np.abs(oracle.e4m3_decode(rcodes)) @ np.abs(oracle.e4m3_decode(wq)).T) \
        * float(rscale) * float(ws)
    exact = oracle.fp8_gemm_exact(rcodes, rscale, wq, ws)
    if bias is not None:
        exact = exact + oracle.bf16_to_f64(bias)[None, :]
    check_dot_outputs(out, exact, absdot, K, gemm_mismatch_bar(K), want_bits=want)


def test_qmm_bias_is_added_per_column(q):
    """A bias of 2^k on column n shifts exactly that column (closed form on a zero input
    is bias itself: abs-max 0 gives zero codes and the matmul adds nothing)."""
    M, N, K = 8, 64, 32
    x = np.zeros((M, K), np.uint16)
    wq, ws = oracle.quantize_tensor(random_bf16((N, K), seed=3, std=0.02))
    bias = oracle.f64_to_bf16(np.ldexp(1.0, np.arange(N) % 7 - 3) * np.where(np.arange(N) % 2, -1, 1))
    out, codes, st = _run(q, x, bias, wq, ws)
    assert not codes.any() and st[1] == np.float32(1.0)
    np.testing.assert_array_equal(out, np.broadcast_to(bias, (M, N)))


def test_attention_qkv_projection_8b_sampled(q):
    """LN1 (fused residual + RMSNorm + abs-max) into the QKV projection at the
    Llama-3-8B shape (N=16384 tokens, C=4096, 4096 + 2*1024 outputs), checked on
    sampled rows stage by stage against the oracle fed the GPU's own y."""
    N, C, NQKV = 16384, 4096, 6144
    res, x = random_bf16((N, C), seed=201), random_bf16((N, C), seed=202)
    gain = oracle.f64_to_bf16(1 + 0.1 * np.random.default_rng(203).standard_normal(C))
    wq, ws = oracle.quantize_tensor(random_bf16((NQKV, C), seed=204, std=0.02))
    r, y = empty_bf16(N, C), empty_bf16(N, C)
    rstd = torch.empty(N, dtype=torch.float32, device="cuda")
    stats = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_rmsnorm_absmax(r, y, rstd, stats, dev(res), dev(x), dev(gain), 1e-5, N, C)
    out, qbuf = empty_bf16(N, NQKV), empty_u8(N, C)
    wsc = torch.tensor([ws], dtype=torch.float32, device="cuda")
    q.qffn_qmm(out, qbuf, stats, y, None, dev(wq), wsc, N, NQKV, C)
    q.qffn_check_status()
    sync()
    st = host(stats)
    yb = bf(y)
    assert st[0] == np.float32(np.max(np.abs(oracle.bf16_to_f64(yb))))
    rows = np.random.default_rng(5).choice(N, 48, replace=False)
    rows.sort()
    # LN1 on the sampled rows: bit-exact
    rr, ry, _, _ = oracle.residual_rmsnorm_absmax(res[rows], x[rows], gain, np.float32(1e-5))
    np.testing.assert_array_equal(bf(r)[rows], rr)
    np.testing.assert_array_equal(yb[rows], ry)
    # quantisation and matmul of those rows with the recorded abs-max
    want, rcodes, rscale = oracle.qmm(yb[rows], st[0], wq, ws)
    assert st[1] == rscale
    np.testing.assert_array_equal(host(qbuf)[rows], rcodes)
    absdot = (np.abs(oracle.e4m3_decode(rcodes)) @ np.abs(oracle.e4m3_decode(wq)).T) * float(rscale) * float(ws)
    check_dot_outputs(bf(out)[rows], oracle.fp8_gemm_exact(rcodes, rscale, wq, ws), absdot, C, gemm_mismatch_bar(C),
                      want_bits=want)
