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
    ws = torch.empty(q.qffn_decode_workspace_size(cfg.C, cfg.H), dtype=torch.uint8, device="cuda")
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
    vec = (2 * cfg.H + 255) // 256 * 256
    h_ws = bf(ws[:2 * cfg.H].view(torch.int16))
    np.testing.assert_array_equal(bf(ws[vec:vec + 2 * cfg.H].view(torch.int16)), ub)
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


def test_decode_per_projection_arm_bit_identical(q):
    """PerProjection arm (separate gate and up GEMVs, silu_mul, down GEMV) gives the
    same bits as the dual + split-SiLU arm."""
    cfg = DECODE["llama3-8b-decode"]
    di, recs, out, ws, x = run_decode(q, cfg)
    g = empty_bf16(cfg.H)
    u = empty_bf16(cfg.H)
    o2 = empty_bf16(cfg.C)
    q.qffn_gemv(g, x, *recs["w_gate"], cfg.H, cfg.C)
    q.qffn_gemv(u, x, *recs["w_up"], cfg.H, cfg.C)
    q.qffn_silu_mul(g, u, cfg.H)
    q.qffn_gemv(o2, g, *recs["w_down"], cfg.C, cfg.H)
    sync()
    assert torch.equal(o2, out)


def test_decode_in_cuda_graph(q):
    """The three launches (the last two programmatic dependent launches) captured in a
    CUDA graph replay to the same bits."""
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


@pytest.mark.parametrize("C,H", [(4096, 14336), (256, 768), (16, 16)])
def test_decode_fused_silu_input_arm_bit_identical(q, C, H):
    """Fused-SiLU-input arm (dual GEMV, then the down GEMV forming silu(g)*u from g and
    u itself) gives the bits of the split-SiLU decode and leaves g and u untouched."""
    cfg = DECODE["llama3-8b-decode"] if (C, H) == (4096, 14336) else DecodeConfig("f", C=C, H=H, seed=C * 3 + H)
    di, recs, out, ws, x = run_decode(q, cfg)
    g = empty_bf16(cfg.H)
    u = empty_bf16(cfg.H)
    q.qffn_gemv_dual(g, u, x, *recs["w_gate"], *recs["w_up"], cfg.H, cfg.C)
    g0, u0 = g.clone(), u.clone()
    o2 = empty_bf16(cfg.C)
    q.qffn_gemv_silu_input(o2, g, u, *recs["w_down"], cfg.C, cfg.H)
    sync()
    assert torch.equal(o2, out)
    assert torch.equal(g, g0) and torch.equal(u, u0)
