"""GPU parity of the single-token FP8 decode FFN (A6..A8) through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from ffn_inputs import DECODE, DecodeConfig, decode_inputs
from gpu_util import (ACC_REL_FMA, assert_out_close, bf, bf16_ulp_diff, check_dot_outputs, dev, empty_bf16,
                      host, sync)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import transformer_ffn_block_gb300 as q
    return q


def _records_on_gpu(q, w_bits):
    rows, cols = w_bits.shape
    codes = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    q.qffn_quantize_rows(codes, scales, dev(w_bits), rows, cols)
    return codes, scales


def run_decode(q, cfg):
    di = decode_inputs(cfg)
    recs = {k: _records_on_gpu(q, di[k]) for k in ("w_gate", "w_up", "w_down")}
    out = empty_bf16(cfg.C)
    ws = torch.zeros(q.qffn_decode_workspace_size(cfg.C, cfg.H), dtype=torch.uint8, device="cuda")
    x = dev(di["x"])
    q.qffn_decode_forward(out, x, *recs["w_gate"], *recs["w_up"], *recs["w_down"], cfg.C, cfg.H, ws)
    sync()
    return di, recs, out, ws, x


@pytest.mark.parametrize("C,H", [(4096, 14336), (256, 768), (16, 16), (2048, 8192), (3584, 18944)])
def test_decode_forward(q, C, H):
    cfg = DECODE["llama3-8b-decode"] if (C, H) == (4096, 14336) else DecodeConfig("d", C=C, H=H, seed=C + H)
    di, recs, out, ws, x = run_decode(q, cfg)
    ref_rec = {k: oracle.quantize_rows(di[k]) for k in ("w_gate", "w_up", "w_down")}
    for k in ref_rec:                                   # the GPU builds the same records
        np.testing.assert_array_equal(host(recs[k][0]), ref_rec[k][0])
        np.testing.assert_array_equal(host(recs[k][1]), ref_rec[k][1])
    ref = oracle.decode_forward(di["x"], *ref_rec["w_gate"], *ref_rec["w_up"], *ref_rec["w_down"])
    assert_out_close(bf(out), ref["out"])
    # stage-wise: g and u from the dual entry point against the exact dual GEMV;
    # the workspace holds h (gate buffer) and u as the split-SiLU arm leaves them
    g = empty_bf16(cfg.H)
    u = empty_bf16(cfg.H)
    q.qffn_gemv_dual(g, u, x, *recs["w_gate"], *recs["w_up"], cfg.H, cfg.C)
    sync()
    gb, ub = bf(g), bf(u)
    xa = np.abs(oracle.bf16_to_f64(di["x"]))
    for got, want, (wq, ws_) in ((gb, ref["g"], ref_rec["w_gate"]), (ub, ref["u"], ref_rec["w_up"])):
        absdot = (np.abs(oracle.e4m3_decode(wq)) @ xa) * ws_.astype(np.float64)
        check_dot_outputs(got, oracle.gemv_exact(di["x"], wq, ws_), absdot, cfg.C, 1e-3, acc_rel=ACC_REL_FMA,
                          want_bits=want)
    off_h, off_u = q.qffn_decode_workspace_offsets(cfg.C, cfg.H)
    h_ws = bf(ws[off_h:off_h + 2 * cfg.H].view(torch.int16))
    np.testing.assert_array_equal(bf(ws[off_u:off_u + 2 * cfg.H].view(torch.int16)), ub)
    assert bf16_ulp_diff(h_ws, oracle.silu_mul(gb, ub)).max() <= 1
    out_stage = oracle.gemv_row_scaled(h_ws, *ref_rec["w_down"])
    absdot = (np.abs(oracle.e4m3_decode(ref_rec["w_down"][0])) @ np.abs(oracle.bf16_to_f64(h_ws))) \
        * ref_rec["w_down"][1].astype(np.float64)
    check_dot_outputs(bf(out), oracle.gemv_exact(h_ws, *ref_rec["w_down"]), absdot, cfg.H, 1e-3,
                      acc_rel=ACC_REL_FMA, want_bits=out_stage)
    # h in the workspace is exactly what the silu_mul entry point makes of g, u
    g2 = g.clone()
    q.qffn_silu_mul(g2, u, cfg.H)
    sync()
    np.testing.assert_array_equal(bf(g2), h_ws)


ARM_SHAPES = [(4096, 14336), (256, 768), (16, 16), (3584, 18944)]


def _cfg(C, H, salt):
    return DECODE["llama3-8b-decode"] if (C, H) == (4096, 14336) else DecodeConfig("a", C=C, H=H, seed=C * salt + H)


def _oracle_decode(di):
    rec = {k: oracle.quantize_rows(di[k]) for k in ("w_gate", "w_up", "w_down")}
    return oracle.decode_forward(di["x"], *rec["w_gate"], *rec["w_up"], *rec["w_down"]), rec


def _check_against_oracle(out, di, ref, rec, gb, ub):
    """An arm's output: the block-output rule against the oracle's decode, and the down
    GEMV stage within its bound of the exact value on the arm's own h = silu(g) * u."""
    assert_out_close(bf(out), ref["out"])
    h = oracle.silu_mul(gb, ub)
    absdot = (np.abs(oracle.e4m3_decode(rec["w_down"][0])) @ np.abs(oracle.bf16_to_f64(h))) \
        * rec["w_down"][1].astype(np.float64)
    check_dot_outputs(bf(out), oracle.gemv_exact(h, *rec["w_down"]), absdot, h.size, 1e-3,
                      acc_rel=ACC_REL_FMA, want_bits=oracle.gemv_row_scaled(h, *rec["w_down"]))


@pytest.mark.parametrize("C,H", ARM_SHAPES)
def test_decode_per_projection_arm(q, C, H):
    """PerProjection arm (separate gate and up GEMVs, silu_mul, down GEMV): the same
    bits as the whole decode, and each stage against the oracle."""
    cfg = _cfg(C, H, 5)
    di, recs, out, ws, x = run_decode(q, cfg)
    ref, rec = _oracle_decode(di)
    g = empty_bf16(cfg.H)
    u = empty_bf16(cfg.H)
    o2 = empty_bf16(cfg.C)
    q.qffn_gemv(g, x, *recs["w_gate"], cfg.H, cfg.C)
    q.qffn_gemv(u, x, *recs["w_up"], cfg.H, cfg.C)
    sync()
    gb, ub = bf(g), bf(u)
    xa = np.abs(oracle.bf16_to_f64(di["x"]))
    for got, want, (wq, sc) in ((gb, ref["g"], rec["w_gate"]), (ub, ref["u"], rec["w_up"])):
        absdot = (np.abs(oracle.e4m3_decode(wq)) @ xa) * sc.astype(np.float64)
        check_dot_outputs(got, oracle.gemv_exact(di["x"], wq, sc), absdot, cfg.C, 1e-3, acc_rel=ACC_REL_FMA,
                          want_bits=want)
    q.qffn_silu_mul(g, u, cfg.H)
    q.qffn_gemv(o2, g, *recs["w_down"], cfg.C, cfg.H)
    sync()
    assert torch.equal(o2, out)
    _check_against_oracle(o2, di, ref, rec, gb, ub)


@pytest.mark.parametrize("C,H", ARM_SHAPES)
def test_decode_fused_silu_input_arm(q, C, H):
    """Fused-SiLU-input arm (dual GEMV, then the down GEMV forming silu(g)*u from g and
    u itself): the bits of the whole decode, g and u untouched, and against the oracle."""
    cfg = _cfg(C, H, 3)
    di, recs, out, ws, x = run_decode(q, cfg)
    ref, rec = _oracle_decode(di)
    g = empty_bf16(cfg.H)
    u = empty_bf16(cfg.H)
    q.qffn_gemv_dual(g, u, x, *recs["w_gate"], *recs["w_up"], cfg.H, cfg.C)
    g0, u0 = g.clone(), u.clone()
    o2 = empty_bf16(cfg.C)
    q.qffn_gemv_silu_input(o2, g, u, *recs["w_down"], cfg.C, cfg.H)
    sync()
    assert torch.equal(o2, out)
    assert torch.equal(g, g0) and torch.equal(u, u0)
    _check_against_oracle(o2, di, ref, rec, bf(g), bf(u))


def test_decode_in_cuda_graph(q):
    """The two launches (the second a programmatic dependent launch) captured in a CUDA
    graph replay to the same bits."""
    cfg = DECODE["llama3-8b-decode"]
    di, recs, out, ws, x = run_decode(q, cfg)
    out2 = empty_bf16(cfg.C)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        q.qffn_decode_forward(out2, x, *recs["w_gate"], *recs["w_up"], *recs["w_down"], cfg.C,
                              cfg.H, ws, stream=s)
    for _ in range(3):
        out2.zero_()
        graph.replay()
    sync()
    assert torch.equal(out2, out)


def test_decode_right_after_quantize_rows_on_one_stream(q):
    """Weights built by qffn_quantize_rows and used by the very next launch on the same
    stream, no synchronisation between: the decode (without the stable-weights flag it
    reads nothing before the preceding kernel has finished) reads the new weights and
    matches the oracle."""
    cfg = DecodeConfig("fresh", C=2048, H=8192, seed=77)
    di = decode_inputs(cfg)
    ref, rec = _oracle_decode(di)
    s = torch.cuda.Stream()
    wb = {k: dev(di[k]) for k in ("w_gate", "w_up", "w_down")}
    x = dev(di["x"])
    sync()
    recs = {}
    for k, (rows, cols) in (("w_gate", (cfg.H, cfg.C)), ("w_up", (cfg.H, cfg.C)), ("w_down", (cfg.C, cfg.H))):
        recs[k] = (torch.full((rows, cols), 0x7E, dtype=torch.uint8, device="cuda"),
                   torch.full((rows,), 1.0, dtype=torch.float32, device="cuda"))
    ws = torch.zeros(q.qffn_decode_workspace_size(cfg.C, cfg.H), dtype=torch.uint8, device="cuda")
    out = empty_bf16(cfg.C)
    sync()
    with torch.cuda.stream(s):
        for k in ("w_gate", "w_up", "w_down"):
            rows, cols = di[k].shape
            q.qffn_quantize_rows(*recs[k], wb[k], rows, cols, stream=s)
        q.qffn_decode_forward(out, x, *recs["w_gate"], *recs["w_up"], *recs["w_down"], cfg.C, cfg.H, ws, stream=s)
    sync()
    q.qffn_check_status()
    assert_out_close(bf(out), ref["out"])
    # the same bits as a decode on weights that were complete long before
    o2 = empty_bf16(cfg.C)
    q.qffn_decode_forward(o2, x, *recs["w_gate"], *recs["w_up"], *recs["w_down"], cfg.C, cfg.H, ws)
    sync()
    assert torch.equal(o2, out)


@pytest.mark.parametrize("C,H", [(4096, 14336), (256, 768)])
def test_decode_variants_give_the_same_bits(q, C, H):
    """qffn_decode_forward_ex with the stable-weights flag (early weight streaming) and
    qffn_decode_forward_gu (one fused [2H, C] gate|up record) give the bits of
    qffn_decode_forward."""
    cfg = _cfg(C, H, 11)
    di, recs, out, ws, x = run_decode(q, cfg)
    o1 = empty_bf16(cfg.C)
    for _ in range(2):
        q.qffn_decode_forward_ex(o1, x, *recs["w_gate"], *recs["w_up"], *recs["w_down"], cfg.C, cfg.H, ws,
                                 q.QFFN_DECODE_WEIGHTS_STABLE)
    sync()
    assert torch.equal(o1, out)
    w_gu = torch.cat([recs["w_gate"][0], recs["w_up"][0]], dim=0).contiguous()
    s_gu = torch.cat([recs["w_gate"][1], recs["w_up"][1]], dim=0).contiguous()
    o2 = empty_bf16(cfg.C)
    q.qffn_decode_forward_gu(o2, x, w_gu, s_gu, *recs["w_down"], cfg.C, cfg.H, ws)
    sync()
    q.qffn_check_status()
    assert torch.equal(o2, out)


def test_decode_workspace_reused_across_shapes(q):
    """One workspace serves calls of different shapes in turn."""
    shapes = [(4096, 14336), (256, 768), (16, 16), (4096, 14336)]
    big = max(q.qffn_decode_workspace_size(C, H) for C, H in shapes)
    shared = torch.zeros(big, dtype=torch.uint8, device="cuda")
    for C, H in shapes:
        di, recs, out, ws, x = run_decode(q, _cfg(C, H, 13))
        o = empty_bf16(C)
        q.qffn_decode_forward(o, x, *recs["w_gate"], *recs["w_up"], *recs["w_down"], C, H, shared)
        sync()
        q.qffn_check_status()
        assert torch.equal(o, out), (C, H)
