"""GPU parity of the recompute form (activation abs-maxes given, not recorded):
the E4M3 SwiGLU epilogue of the gate|up GEMM, the elementwise
swiglu_forward_quant, and the whole chain qffn_forward_recompute, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from ffn_inputs import PREFILL, prefill_inputs, random_bf16
from gpu_util import (assert_out_close, bf, check_codes_rule, dev, e4m3_step_diff, empty_bf16, empty_u8,
                      host, sync)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import transformer_ffn_block_gb300 as q
    return q


def _gate_up_inputs(N, C, H, seed):
    yq, sy = oracle.quantize_tensor(random_bf16((N, C), seed=seed))
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), seed=seed + 1, std=0.02))
    scales = torch.tensor([sy, w1s], dtype=torch.float32, device="cuda")
    return dev(yq), dev(w1q), scales


@pytest.mark.parametrize("N,C,H", [(64, 256, 768), (1, 128, 128), (200, 384, 256), (513, 2048, 1024),
                                   (300, 4096, 14336),
                                   # the last wave as half tiles, one with a ragged last M-block
                                   (5120, 64, 512), (4900, 96, 512),
                                   # K > 2048 (the eight-column epilogue step), half tiles
                                   (5120, 2304, 512)])
def test_gate_up_swiglu_quant_equals_two_pass(q, N, C, H):
    """E4M3 straight from the epilogue == quantize of the bf16 h the SwiGLU epilogue
    writes, with the abs-max that call recorded (codes and scale bit for bit)."""
    yqd, w1d, scales = _gate_up_inputs(N, C, H, N + C + H)
    h = empty_bf16(N, H)
    stats = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_gate_up_swiglu(h, stats, yqd, scales[0:1], w1d, scales[1:2], N, C, H)
    hq_ref = empty_u8(N, H)
    q.qffn_quantize(hq_ref, stats, h, N * H)
    stats2 = stats.clone()
    stats2[1] = -7.0
    hq = empty_u8(N, H)
    q.qffn_gate_up_swiglu_quant(hq, stats2, yqd, scales[0:1], w1d, scales[1:2], N, C, H)
    q.qffn_check_status()
    sync()
    np.testing.assert_array_equal(host(hq), host(hq_ref))
    np.testing.assert_array_equal(host(stats2), host(stats))
    # and against the oracle's quantiser on the GPU's own h
    codes, scale = oracle.quantize_with_abs_max(bf(h), host(stats)[0])
    np.testing.assert_array_equal(host(hq), codes)
    assert host(stats2)[1] == scale


@pytest.mark.parametrize("factor", [0.25, 4.0, 0.0])
def test_gate_up_swiglu_quant_given_absmax_not_recorded(q, factor):
    """A given abs-max unrelated to the data is used as given: below the true one
    elements saturate at +-448, above it the codes shrink; 0 gives zero codes, scale 1."""
    N, C, H = 130, 512, 384
    yqd, w1d, scales = _gate_up_inputs(N, C, H, 17)
    h = empty_bf16(N, H)
    stats = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_gate_up_swiglu(h, stats, yqd, scales[0:1], w1d, scales[1:2], N, C, H)
    sync()
    given = np.float32(host(stats)[0] * np.float32(factor))
    st = torch.tensor([given, -1.0], dtype=torch.float32, device="cuda")
    hq = empty_u8(N, H)
    q.qffn_gate_up_swiglu_quant(hq, st, yqd, scales[0:1], w1d, scales[1:2], N, C, H)
    sync()
    codes, scale = oracle.quantize_with_abs_max(bf(h), given)
    np.testing.assert_array_equal(host(hq), codes)
    assert host(st)[0] == given and host(st)[1] == scale
    if factor == 0.25:
        assert np.any((host(hq) & 0x7F) == 0x7E)
    if factor == 0.0:
        assert not host(hq).any() and scale == np.float32(1.0)


@pytest.mark.parametrize("N,H", [(1, 8), (64, 768), (333, 1024), (16, 14336)])
def test_swiglu_forward_quant_given_absmax(q, N, H):
    """The elementwise recompute form: with the recorded abs-max it reproduces the
    two-pass codes; with another abs-max it is the oracle's quantiser applied to h."""
    rng = np.random.default_rng(N * 7 + H)
    gu = oracle.f64_to_bf16(rng.standard_normal((N, 2 * H)) * 10.0 ** rng.integers(-1, 2, (N, 2 * H)))
    gud = dev(gu)
    h = empty_bf16(N, H)
    hq = empty_u8(N, H)
    stats = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_swiglu_quant(h, hq, stats, gud, N, H)
    sync()
    st = host(stats)
    for given in (st[0], np.float32(st[0] * np.float32(0.3))):
        s2 = torch.tensor([given, -1.0], dtype=torch.float32, device="cuda")
        hq2 = empty_u8(N, H)
        q.qffn_swiglu_forward_quant(hq2, s2, gud, N, H)
        sync()
        codes, scale = oracle.quantize_with_abs_max(bf(h), given)
        np.testing.assert_array_equal(host(hq2), codes)
        assert host(s2)[1] == scale
        # the fp64 oracle's h may differ from the GPU's by one bf16 ulp: codes by <= 1 step
        rq, rs = oracle.swiglu_forward_quant(gu, H, given)
        assert rs == scale
        assert e4m3_step_diff(host(hq2), rq).max() <= 1
        if given == st[0]:                                   # the recorded abs-max
            np.testing.assert_array_equal(host(hq2), host(hq))


def _forward_pair(q, cfg, inp, ay=None, ah=None):
    """qffn_forward, then qffn_forward_recompute with its recorded abs-maxes (or the
    ones given).  Returns both results' tensors."""
    N, C, H = cfg.N, cfg.C, cfg.H
    w1s_ = torch.zeros(2, dtype=torch.float32, device="cuda")
    w2s_ = torch.zeros(2, dtype=torch.float32, device="cuda")
    w1 = empty_u8(2 * H, C)
    w2 = empty_u8(C, H)
    for w, src, st in ((w1, inp["w1"], w1s_), (w2, inp["w2"], w2s_)):
        wb = dev(src)
        q.qffn_absmax(st, wb, src.size)
        q.qffn_quantize(w, st, wb, src.size)
    res, x, gain = dev(inp["res"]), dev(inp["x"]), dev(inp["gain"])
    ws_bytes = q.qffn_forward_workspace_size(cfg.B, cfg.T, C, H)
    off = q.qffn_forward_workspace_offsets(cfg.B, cfg.T, C, H)
    outs = []
    for mode in ("forward", "recompute"):
        res_out, out = empty_bf16(N, C), empty_bf16(N, C)
        rstd = torch.empty(N, dtype=torch.float32, device="cuda")
        ws = torch.full((ws_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
        if mode == "forward":
            stats = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")
            q.qffn_forward(res_out, out, rstd, stats[0:2], stats[2:4], res, x, gain, inp["eps"],
                           w1, w1s_[1:2], w2, w2s_[1:2], cfg.B, cfg.T, C, H, ws)
        else:
            rec = host(outs[0]["stats"])
            stats = torch.tensor([rec[0] if ay is None else ay, -1.0, rec[2] if ah is None else ah, -1.0],
                                 dtype=torch.float32, device="cuda")
            q.qffn_forward_recompute(res_out, out, rstd, stats[0:2], stats[2:4], res, x, gain,
                                     inp["eps"], w1, w1s_[1:2], w2, w2s_[1:2], cfg.B, cfg.T, C, H, ws)
        q.qffn_check_status()
        sync()
        outs.append(dict(res_out=bf(res_out), out=bf(out), rstd=host(rstd), stats=stats,
                         y=bf(ws[off[0]:off[0] + N * C * 2].view(torch.int16)).reshape(N, C),
                         yq=host(ws[off[1]:off[1] + N * C]).reshape(N, C),
                         hq=host(ws[off[3]:off[3] + N * H]).reshape(N, H),
                         h_slot=host(ws[off[2]:off[2] + N * H * 2])))
    outs[1]["stats"] = host(outs[1]["stats"])
    outs[0]["stats"] = host(outs[0]["stats"])
    return outs, (w1, w1s_, w2, w2s_)


@pytest.mark.parametrize("name", ["tiny", "llama3.2-1b", "llama3-8b"])
def test_forward_recompute_with_recorded_absmax_equals_forward(q, name):
    """Given the abs-maxes qffn_forward recorded, the recompute chain reproduces
    every output of that forward bit for bit, and leaves the h slot untouched."""
    cfg = PREFILL[name]
    f, r = _forward_pair(q, cfg, prefill_inputs(cfg))[0]
    for k in ("res_out", "out", "rstd", "y", "yq", "hq", "stats"):
        np.testing.assert_array_equal(r[k], f[k], err_msg=k)
    assert np.all(r["h_slot"] == 0xAB)


def test_forward_recompute_given_absmax_against_oracle(q):
    """Abs-maxes unrelated to the data (y: 1.5x, h: 0.5x the recorded ones): yq bit-exact,
    hq equal to the oracle's quantiser on the GPU's own h, out within the block tolerance."""
    cfg = PREFILL["tiny"]
    inp = prefill_inputs(cfg)
    w1q, w1s = oracle.quantize_tensor(inp["w1"])
    w2q, w2s = oracle.quantize_tensor(inp["w2"])
    fwd = oracle.ffn_forward(inp["res"], inp["x"], inp["gain"], inp["eps"], w1q, w1s, w2q, w2s, cfg.H)
    ay = np.float32(fwd["stats_y"][0] * np.float32(1.5))
    ah = np.float32(fwd["stats_h"][0] * np.float32(0.5))
    (f, r), (w1, w1s_, w2, w2s_) = _forward_pair(q, cfg, inp, ay=ay, ah=ah)
    ref = oracle.ffn_forward_recompute(inp["res"], inp["x"], inp["gain"], inp["eps"], w1q, w1s, w2q,
                                       w2s, cfg.H, ay, ah)
    np.testing.assert_array_equal(r["y"], ref["y"])
    np.testing.assert_array_equal(r["yq"], ref["yq"])
    np.testing.assert_array_equal(r["stats"][0:2], ref["stats_y"])
    np.testing.assert_array_equal(r["stats"][2:4], ref["stats_h"])
    # stage-wise: h from the GPU's SwiGLU epilogue on the same yq, quantised by the oracle
    N, C, H = cfg.N, cfg.C, cfg.H
    h = empty_bf16(N, H)
    st = torch.zeros(2, dtype=torch.float32, device="cuda")
    ysc = torch.tensor([ref["stats_y"][1]], dtype=torch.float32, device="cuda")
    q.qffn_gate_up_swiglu(h, st, dev(r["yq"]), ysc, w1, w1s_[1:2], N, C, H)
    sync()
    codes, _ = oracle.quantize_with_abs_max(bf(h), ah)
    np.testing.assert_array_equal(r["hq"], codes)
    check_codes_rule(r["hq"], ref["hq"])
    assert np.any((r["hq"] & 0x7F) == 0x7E)                 # h beyond the given abs-max saturates
    assert_out_close(r["out"], ref["out"])
