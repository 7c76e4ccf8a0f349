"""End-to-end GPU parity of qffn_forward (the whole prefill chain A1..A5).

The tiny, Llama-3.2-1B and ragged workloads are compared with the oracle over
every element.  The Qwen2.5-7B-shaped and Llama-3-8B workloads run at full
size: the norm, the quantised y and both per-tensor abs-maxes are compared
with the oracle's own over the whole tensor, and sampled rows stage by stage
(each stage fed the GPU's own upstream tensor) and end to end.
"""
import numpy as np
import pytest
import torch

import oracle
from ffn_inputs import PREFILL, PrefillConfig, prefill_inputs
from gpu_util import (absdot_gemm, assert_out_close, bf, bf16_ulp_diff, check_codes_rule, check_dot_outputs,
                      dev, empty_bf16, gemm_mismatch_bar, host, sync)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import transformer_ffn_block_gb300 as q
    return q


def _gpu_weight_record(q, w_bits):
    """Per-tensor E4M3 record built on the GPU (qffn_absmax + qffn_quantize)."""
    wd = dev(w_bits)
    stats = torch.zeros(2, dtype=torch.float32, device="cuda")
    codes = torch.empty(w_bits.shape, dtype=torch.uint8, device="cuda")
    q.qffn_absmax(stats, wd, w_bits.size)
    q.qffn_quantize(codes, stats, wd, w_bits.size)
    return codes, stats


def run_forward(q, cfg, inp, with_res=True):
    N, C, H = cfg.N, cfg.C, cfg.H
    w1, s1 = _gpu_weight_record(q, inp["w1"])
    w2, s2 = _gpu_weight_record(q, inp["w2"])
    res_out = empty_bf16(N, C) if with_res else None
    out = empty_bf16(N, C)
    rstd = torch.empty(N, dtype=torch.float32, device="cuda")
    stats = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")
    ws_bytes = q.qffn_forward_workspace_size(cfg.B, cfg.T, C, H)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    q.qffn_forward(res_out, out, rstd, stats[0:2], stats[2:4], dev(inp["res"]) if with_res else None,
                   dev(inp["x"]), dev(inp["gain"]), inp["eps"], w1, s1[1:2], w2, s2[1:2],
                   cfg.B, cfg.T, C, H, ws)
    q.qffn_check_status()
    sync()
    off = q.qffn_forward_workspace_offsets(cfg.B, cfg.T, C, H)
    y = ws[off[0]:off[0] + N * C * 2].view(torch.int16).view(N, C)
    yq = ws[off[1]:off[1] + N * C].view(N, C)
    h = ws[off[2]:off[2] + N * H * 2].view(torch.int16).view(N, H)
    hq = ws[off[3]:off[3] + N * H].view(N, H)
    return dict(res_out=res_out, out=out, rstd=rstd, stats=stats, y=y, yq=yq, h=h, hq=hq,
                w1=w1, s1=s1, w2=w2, s2=s2)


def check_gemm_stage(got, a, sa, w, sw):
    """A GEMM stage fed the GPU's own operand codes: every output within the
    accumulation bound of the exact value, and at most the K-dependent fraction
    of outputs differing from the exactly rounded one."""
    K = a.shape[1]
    check_dot_outputs(got, oracle.fp8_gemm_exact(a, sa, w, sw), absdot_gemm(a, sa, w, sw), K,
                      gemm_mismatch_bar(K))


def check_h_stage(q, g, yq_rows, h_rows, st, w1q, w1s, H):
    """h rows against SwiGLU of the GPU's unfused gate|up GEMM on the same yq rows."""
    M, C = yq_rows.shape
    gu = empty_bf16(M, 2 * H)
    yqd = dev(yq_rows)
    q.qffn_fp8_gemm_scaled(gu, yqd, g["stats"][1:2], g["w1"], g["s1"][1:2], M, 2 * H, C)
    sync()
    gub = bf(gu)
    h_from_gu, _ = oracle.swiglu(gub, H)
    assert bf16_ulp_diff(h_rows, h_from_gu).max() <= 1
    check_gemm_stage(gub, yq_rows, st[1], w1q, w1s)


def check_full(q, cfg, with_res=True):
    inp = prefill_inputs(cfg)
    g = run_forward(q, cfg, inp, with_res)
    w1q, w1s = oracle.quantize_tensor(inp["w1"])
    w2q, w2s = oracle.quantize_tensor(inp["w2"])
    # the GPU builds the same weight records bit for bit
    np.testing.assert_array_equal(host(g["w1"]), w1q)
    np.testing.assert_array_equal(host(g["w2"]), w2q)
    assert host(g["s1"])[1] == w1s and host(g["s2"])[1] == w2s
    ref = oracle.ffn_forward(inp["res"] if with_res else None, inp["x"], inp["gain"], inp["eps"],
                             w1q, w1s, w2q, w2s, cfg.H)
    st = host(g["stats"])
    y, yq, h, hq = bf(g["y"]), host(g["yq"]), bf(g["h"]), host(g["hq"])

    # A1, A2: bit-exact
    if with_res:
        np.testing.assert_array_equal(bf(g["res_out"]), ref["r"])
    np.testing.assert_array_equal(y, ref["y"])
    np.testing.assert_allclose(host(g["rstd"]), ref["rstd"], rtol=2.0 ** -23, atol=0)
    np.testing.assert_array_equal(st[0:2], ref["stats_y"])                     # abs-max, scale
    np.testing.assert_array_equal(yq, ref["yq"])                               # codes
    # A3+A4 stage-wise: the fused h equals SwiGLU of the GPU's own unfused gate|up GEMM
    # of its own yq (within 1 ulp of the fp64 silu); that GEMM is within the fp32
    # accumulation bound of the exact product
    check_h_stage(q, g, yq, h, st, w1q, w1s, cfg.H)
    assert st[2] == np.float32(np.max(np.abs(oracle.bf16_to_f64(h))))
    codes, scale = oracle.quantize_with_abs_max(h, st[2])
    np.testing.assert_array_equal(hq, codes)
    assert st[3] == scale
    # end to end against the oracle: abs-max and scale of h bit-exact, the FP8 code rule
    np.testing.assert_array_equal(st[2:4], ref["stats_h"])
    check_codes_rule(hq, ref["hq"])
    # A5 from the GPU's own hq
    out = bf(g["out"])
    check_gemm_stage(out, hq, st[3], w2q, w2s)
    # the acceptance rule against the end-to-end oracle
    return assert_out_close(out, ref["out"])


def oracle_whole_amax_h(q, g, yq, sy, w1q, w1s, H, chunk=1024):
    """The oracle's own abs-max of h over the whole tensor, found without the oracle
    computing every row.

    The GPU's unfused gate|up GEMM gives g', u' for every element.  The exact
    values lie within the accumulation bound of those (the rule the GEMM stage
    checks), with sum|terms| bounded by Cauchy-Schwarz: sa sw |yq row| |w1 row|.
    From that, each element gets an upper bound UB on the oracle's |h| (using
    |silu(z)| <= max(|z|, 0.28)).  The oracle computes in full the row holding
    the GPU's largest |h| (a lower bound A0 on its own abs-max) and then every
    row with an element whose UB reaches A0; no other row can hold its maximum.
    Returns (oracle abs-max, number of rows the oracle computed)."""
    N, C = yq.shape
    ya = np.sqrt(np.sum(oracle.e4m3_decode(yq) ** 2, axis=1))                # [N]
    wa = np.sqrt(np.sum(oracle.e4m3_decode(w1q) ** 2, axis=1))               # [2H]
    k = (C * 2.0 ** -23 + 2.0 ** -22) * float(sy) * float(w1s)
    lift = 1.0 + 2.0 ** -8                                                   # one bf16 rounding up
    ub_row = np.zeros(N)
    for r0 in range(0, N, chunk):
        r1 = min(N, r0 + chunk)
        gu = empty_bf16(r1 - r0, 2 * H)
        q.qffn_fp8_gemm_scaled(gu, dev(yq[r0:r1]), g["stats"][1:2], g["w1"], g["s1"][1:2], r1 - r0, 2 * H, C)
        sync()
        v = oracle.bf16_to_f64(bf(gu))
        del gu
        bnd = k * ya[r0:r1, None] * wa[None, :]
        bnd += 0.5 * np.ldexp(1.0, np.frexp(np.maximum(np.abs(v), 2.0 ** -126))[1] - 8) + 2.0 ** -24 * np.abs(v)
        mag = (np.abs(v) + bnd) * lift
        ub = np.maximum(mag[:, :H], 0.2785) * mag[:, H:] * lift * lift
        ub_row[r0:r1] = ub.max(axis=1)
        del v, bnd, mag, ub
    gpu_arg = int(torch.argmax(g["h"].view(torch.bfloat16).float().abs().amax(dim=1)).item())

    def oracle_rows_max(rows):
        gu_o = oracle.fp8_gemm_scaled(yq[rows], sy, w1q, w1s)
        return float(oracle.swiglu(gu_o, H)[1])

    a0 = oracle_rows_max(np.array([gpu_arg]))
    cand = np.nonzero(ub_row >= a0)[0]
    return max(a0, oracle_rows_max(cand)), len(cand)


def check_sampled(q, cfg, rows):
    """Full-size workload in the benchmark's launch configuration: whole-tensor checks
    of A1, A2 and of both abs-maxes against the oracle's own, then sampled rows stage
    by stage and end to end."""
    inp = prefill_inputs(cfg)
    g = run_forward(q, cfg, inp)
    N, H = cfg.N, cfg.H
    st = host(g["stats"])
    w1q, w1s = oracle.quantize_tensor(inp["w1"])
    w2q, w2s = oracle.quantize_tensor(inp["w2"])
    np.testing.assert_array_equal(host(g["w1"]), w1q)
    np.testing.assert_array_equal(host(g["w2"]), w2q)
    # A1 and A2 over the whole tensor, against the oracle's own norm and abs-max
    r_ref, y_ref, rstd_ref, amax_y = oracle.residual_rmsnorm_absmax(inp["res"], inp["x"], inp["gain"], inp["eps"])
    np.testing.assert_array_equal(bf(g["res_out"]), r_ref)
    np.testing.assert_array_equal(bf(g["y"]), y_ref)
    np.testing.assert_allclose(host(g["rstd"]), rstd_ref, rtol=2.0 ** -23, atol=0)
    yq_ref, sy_ref = oracle.quantize_with_abs_max(y_ref, amax_y)
    assert st[0] == amax_y and st[1] == sy_ref
    yq = host(g["yq"])
    np.testing.assert_array_equal(yq, yq_ref)
    del r_ref, y_ref
    # the abs-max of h: the GPU's equals the max of its own h and the oracle's own
    # whole-tensor abs-max, bit for bit
    assert st[2] == torch.max(torch.abs(g["h"].view(torch.bfloat16).float())).item()
    amax_h, n_rows = oracle_whole_amax_h(q, g, yq, sy_ref, w1q, w1s, H)
    assert st[2] == amax_h, (st[2], amax_h, n_rows)
    assert st[3] == np.float32(amax_h / np.float32(448))
    # sampled rows, stage by stage
    h = bf(g["h"])[rows]
    check_h_stage(q, g, yq[rows], h, st, w1q, w1s, H)
    hq = host(g["hq"])[rows]
    np.testing.assert_array_equal(hq, oracle.quantize_with_abs_max(h, st[2])[0])
    out = bf(g["out"])[rows]
    check_gemm_stage(out, hq, st[3], w2q, w2s)
    # end to end on the sampled rows: the oracle's chain with its own abs-maxes
    gu_ref = oracle.fp8_gemm_scaled(yq_ref[rows], sy_ref, w1q, w1s)
    h_ref, _ = oracle.swiglu(gu_ref, H)
    hq_ref, sh_ref = oracle.quantize_with_abs_max(h_ref, amax_h)
    check_codes_rule(hq, hq_ref)
    out_ref = oracle.fp8_gemm_scaled(hq_ref, sh_ref, w2q, w2s)
    assert_out_close(out, out_ref)


@pytest.mark.parametrize("name", ["tiny", "llama3.2-1b"])
def test_forward_full_parity(q, name):
    check_full(q, PREFILL[name])


def _sample_rows(N, extra, seed=0):
    return np.unique(np.concatenate([[0, 1, 127, 128, N // 2 - 1, N - 2, N - 1],
                                     np.random.default_rng(seed).integers(0, N, extra)]))


def test_forward_qwen_outliers_sampled(q):
    """Qwen2.5-7B shape, 0.1% outliers x20: stresses the abs-max scaling end to end."""
    cfg = PREFILL["qwen2.5-7b"]
    check_sampled(q, cfg, _sample_rows(cfg.N, 57))


@pytest.mark.parametrize("B,T,C,H", [(1, 1, 128, 128), (3, 43, 256, 384), (1, 129, 384, 512),
                                     (2, 200, 1024, 2816)])
def test_forward_ragged_shapes(q, B, T, C, H):
    check_full(q, PrefillConfig("ragged", B=B, T=T, C=C, H=H, eps=1e-5, seed=B * T + C))


def test_forward_without_residual(q):
    check_full(q, PREFILL["tiny"], with_res=False)


def test_forward_zero_input(q):
    cfg = PrefillConfig("zeros", B=1, T=70, C=256, H=256, eps=1e-5)
    inp = prefill_inputs(cfg)
    inp["res"][:] = 0
    inp["x"][:] = 0
    g = run_forward(q, cfg, inp)
    st = host(g["stats"])
    assert st.tolist() == [0.0, 1.0, 0.0, 1.0]
    assert not host(g["yq"]).any() and not host(g["hq"]).any()
    assert not np.any(oracle.bf16_to_f64(bf(g["out"])))


def test_forward_empty(q):
    cfg = PrefillConfig("empty", B=0, T=16, C=256, H=256, eps=1e-5)
    stats = torch.full((4,), 3.0, dtype=torch.float32, device="cuda")
    w = torch.zeros(2 * 256 * 256, dtype=torch.uint8, device="cuda")
    sc = torch.ones(2, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(q.qffn_forward_workspace_size(0, 16, 256, 256), 256), dtype=torch.uint8, device="cuda")
    dummy = empty_bf16(8)
    q.qffn_forward(dummy, dummy, sc, stats[0:2], stats[2:4], dummy, dummy, dummy, 1e-5, w, sc[0:1],
                   w, sc[1:2], 0, 16, 256, 256, ws)
    sync()
    assert host(stats)[[0, 2]].tolist() == [0.0, 0.0]


def test_forward_repeatable(q):
    """Two calls on the same inputs give identical bits (stats re-zeroed each call)."""
    cfg = PREFILL["tiny"]
    inp = prefill_inputs(cfg)
    a = run_forward(q, cfg, inp)
    b = run_forward(q, cfg, inp)
    for k in ("out", "res_out", "h", "hq", "stats"):
        assert torch.equal(a[k], b[k]), k


def test_forward_llama3_8b_sampled(q):
    """Full Llama-3-8B shape (N=16384, C=4096, H=14336) in the launch configuration the
    benchmark times: whole-tensor A1/A2 and both abs-maxes against the oracle's own,
    sampled rows stage by stage and end to end."""
    cfg = PREFILL["llama3-8b"]
    check_sampled(q, cfg, _sample_rows(cfg.N, 57))


@pytest.mark.parametrize("B,T,C,H", [(2, 32, 256, 768), (3, 43, 256, 384), (1, 300, 2176, 384)])
def test_forward_graph_capture_equals_eager(q, B, T, C, H):
    """qffn_forward and qffn_forward_recompute captured in a CUDA graph (their
    programmatic dependent launches and the abs-max memset become graph nodes) and
    replayed twice give the eager call's bits in every output and workspace tap.
    The shapes take both SwiGLU epilogue steps (K <= 2048 and K > 2048)."""
    cfg = PrefillConfig("graph", B=B, T=T, C=C, H=H, eps=1e-5, seed=B + T + C)
    inp = prefill_inputs(cfg)
    N = cfg.N
    w1, s1 = _gpu_weight_record(q, inp["w1"])
    w2, s2 = _gpu_weight_record(q, inp["w2"])
    res, x, gain = dev(inp["res"]), dev(inp["x"]), dev(inp["gain"])
    ws_bytes = q.qffn_forward_workspace_size(B, T, C, H)

    def buffers():
        return dict(res_out=empty_bf16(N, C), out=empty_bf16(N, C),
                    rstd=torch.empty(N, dtype=torch.float32, device="cuda"),
                    stats=torch.full((4,), -1.0, dtype=torch.float32, device="cuda"),
                    ws=torch.full((ws_bytes,), 0xAB, dtype=torch.uint8, device="cuda"))

    def fwd(b, stream=None):
        q.qffn_forward(b["res_out"], b["out"], b["rstd"], b["stats"][0:2], b["stats"][2:4], res, x, gain,
                       cfg.eps, w1, s1[1:2], w2, s2[1:2], B, T, C, H, b["ws"], stream=stream)

    def rec(b, stream=None):
        q.qffn_forward_recompute(b["res_out"], b["out"], b["rstd"], b["stats"][0:2], b["stats"][2:4], res, x,
                                 gain, cfg.eps, w1, s1[1:2], w2, s2[1:2], B, T, C, H, b["ws"], stream=stream)

    def snap(b):
        return {k: host(v).copy() for k, v in b.items()}

    eager = buffers()
    fwd(eager)
    q.qffn_check_status()
    sync()
    want = snap(eager)
    eager_rec = buffers()
    eager_rec["stats"].copy_(torch.tensor([want["stats"][0], -1.0, want["stats"][2], -1.0]))
    rec(eager_rec)
    q.qffn_check_status()
    sync()
    want_rec = snap(eager_rec)
    for call, ref, given in ((fwd, want, None), (rec, want_rec, want["stats"])):
        b = buffers()
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            call(b, stream=stream)
        for _ in range(2):
            b["ws"].fill_(0xAB)              # as before the eager call: the recompute form leaves the h slot
            for k in ("res_out", "out", "rstd"):
                b[k].fill_(-7)
            b["stats"].copy_(torch.tensor([-1.0] * 4) if given is None
                             else torch.tensor([given[0], -1.0, given[2], -1.0]))
            graph.replay()
            sync()
            got = snap(b)
            for k in ref:
                assert np.array_equal(got[k], ref[k]), (call.__name__, k)
        q.qffn_check_status()


def test_forward_two_streams_concurrently(q):
    """Two forwards with their own inputs, outputs and workspaces enqueued on two
    streams at once (the kernels may interleave on the device) give the bits each
    gives alone."""
    cfgs = [PrefillConfig("concurrent", B=2, T=96, C=512, H=768, eps=1e-5, seed=s) for s in (5, 6)]
    runs = []
    for cfg in cfgs:
        inp = prefill_inputs(cfg)
        w1, s1 = _gpu_weight_record(q, inp["w1"])
        w2, s2 = _gpu_weight_record(q, inp["w2"])
        N, C, H = cfg.N, cfg.C, cfg.H
        ws_bytes = q.qffn_forward_workspace_size(cfg.B, cfg.T, C, H)
        args = dict(res=dev(inp["res"]), x=dev(inp["x"]), gain=dev(inp["gain"]), w1=w1, s1=s1, w2=w2, s2=s2)

        def buffers(N=N, C=C, ws_bytes=ws_bytes):
            return dict(res_out=empty_bf16(N, C), out=empty_bf16(N, C),
                        rstd=torch.empty(N, dtype=torch.float32, device="cuda"),
                        stats=torch.full((4,), -1.0, dtype=torch.float32, device="cuda"),
                        ws=torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda"))

        runs.append((cfg, args, buffers))

    def fwd(cfg, a, b, stream):
        q.qffn_forward(b["res_out"], b["out"], b["rstd"], b["stats"][0:2], b["stats"][2:4], a["res"], a["x"],
                       a["gain"], cfg.eps, a["w1"], a["s1"][1:2], a["w2"], a["s2"][1:2], cfg.B, cfg.T, cfg.C,
                       cfg.H, b["ws"], stream=stream)

    alone = []
    for cfg, a, buffers in runs:
        b = buffers()
        fwd(cfg, a, b, None)
        sync()
        alone.append({k: host(v).copy() for k, v in b.items()})
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    bufs = [buffers() for _, _, buffers in runs]
    for rep in range(3):
        for (cfg, a, _), b, s in zip(runs, bufs, streams):
            fwd(cfg, a, b, s)
    sync()
    q.qffn_check_status()
    for want, b in zip(alone, bufs):
        for k, v in want.items():
            assert np.array_equal(host(b[k]), v), k
