"""GPU parity of the FP8 FFN backward (transpose, swiglu_backward, backward_qmm and the
chain qffn_ffn_backward) through the C ABI, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from ffn_inputs import random_bf16, random_codes
from gpu_util import (assert_out_close, bf, bf16_ulp_diff, check_dot_outputs, dev, empty_bf16,
                      empty_u8, gemm_mismatch_bar, host, sync)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import transformer_ffn_block_gb300 as q
    return q


def _mixed(shape, seed, spread=1):
    rng = np.random.default_rng(seed)
    return oracle.f64_to_bf16(rng.standard_normal(shape) * 10.0 ** rng.integers(-spread, spread + 1, shape))


def _absdot(a_codes, sa, b_codes, sb):
    """scale * sum |terms| of out = A . B^T (the fp32 accumulation bound's magnitude)."""
    return (np.abs(oracle.e4m3_decode(a_codes)) @ np.abs(oracle.e4m3_decode(b_codes)).T) * float(sa) * float(sb)


def _check_gemm(got, want, a, sa, b, sb, old=None, max_mismatch=None):
    """got and the oracle's want are bf16(old + sa sb A B^T): every output within the
    accumulation bound of the exact value, at most the K-dependent fraction differing."""
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    exact = oracle.fp8_gemm_exact(a, sa, b, sb)
    if old is not None:
        exact = oracle.bf16_to_f64(old) + exact
    K = a.shape[1]
    return check_dot_outputs(got, exact, _absdot(a, sa, b, sb), K,
                             gemm_mismatch_bar(K) if max_mismatch is None else max_mismatch, want_bits=want)


@pytest.mark.parametrize("R,C", [(16, 16), (48, 80), (64, 128), (1040, 336), (4096, 14336)])
def test_transpose_e4m3(q, R, C):
    a = random_codes((R, C), seed=R + C)
    out = empty_u8(C, R)
    q.qffn_transpose_e4m3(out, dev(a), R, C)
    sync()
    np.testing.assert_array_equal(host(out), a.T)


def _check_swiglu_grad(got, want):
    """<= 1 bf16 ulp, except where silu'(g) is near its root (g ~ -1.28): there the
    fp32 value of 1 + g (1 - sigmoid(g)) cancels, so a few tiny outputs may differ more."""
    d = bf16_ulp_diff(got, want)
    w = np.abs(oracle.bf16_to_f64(want))
    bad = d > 1
    assert bad.mean() <= 1e-3
    if bad.any():
        assert np.all(w[bad] <= 1e-2 * w.max())


@pytest.mark.parametrize("N,H", [(1, 8), (64, 768), (333, 1024), (16, 14336)])
def test_swiglu_backward(q, N, H):
    gu = _mixed((N, 2 * H), N + H)
    dh = _mixed((N, H), N * 3 + H)
    d = empty_bf16(N, 2 * H)
    stats = torch.full((2,), 5.0, dtype=torch.float32, device="cuda")
    q.qffn_swiglu_backward(d, stats, dev(dh), dev(gu), N, H)
    sync()
    got = bf(d)
    want, _ = oracle.swiglu_backward(dh, gu, H)
    _check_swiglu_grad(got, want)
    st = host(stats)
    assert st[0] == np.float32(np.max(np.abs(oracle.bf16_to_f64(got))))     # its own abs-max, exactly
    assert st[1] == 5.0


@pytest.mark.parametrize("N,IC,OC,acc", [(48, 96, 64, False), (64, 256, 128, True), (256, 512, 384, False),
                                         (512, 1024, 2048, True),
                                         # accumulating with ragged tiles: IC = 160 ends inside a
                                         # 64-column box, OC = 96 inside a 128-row half tile
                                         (48, 160, 96, True), (272, 288, 352, True)])
def test_backward_qmm(q, N, IC, OC, acc):
    dout = random_bf16((N, OC), seed=N + OC, std=1e-3)
    inq, ins = oracle.quantize_tensor(random_bf16((N, IC), seed=N + IC))
    wq, ws = oracle.quantize_tensor(random_bf16((OC, IC), seed=OC + IC, std=0.02))
    old = random_bf16((OC, IC), seed=7, std=1e-2)
    amax = oracle.absmax(dout)
    stats = torch.tensor([amax, -1.0], dtype=torch.float32, device="cuda")
    sc = torch.tensor([ins, ws], dtype=torch.float32, device="cuda")
    dinp = empty_bf16(N, IC)
    dw = dev(old) if acc else empty_bf16(OC, IC)
    wsb = torch.empty(q.qffn_backward_qmm_workspace_size(N, IC, OC), dtype=torch.uint8, device="cuda")
    q.qffn_backward_qmm(dinp, dw, stats, dev(dout), dev(inq), sc[0:1], dev(wq), sc[1:2], N, IC, OC, acc, wsb)
    q.qffn_check_status()
    sync()
    rd, rw, rq, rs = oracle.backward_qmm(dout, amax, inq, ins, wq, ws, old if acc else None)
    assert host(stats)[1] == rs
    np.testing.assert_array_equal(host(wsb[:N * OC]).reshape(N, OC), rq)       # dout codes
    _check_gemm(bf(dinp), rd, rq, rs, wq.T, ws)
    _check_gemm(bf(dw), rw, rq.T, rs, inq.T, ins, old=old if acc else None)


def _ffn_backward_dev(q, dout, amax, yq, sy, hq, sh, w1q, w1s, w2q, w2s, N, C, H, acc=False,
                     dw_init=None):
    """Runs qffn_ffn_backward; returns its outputs and workspace intermediates as
    device tensors (bf16 bits as int16) plus the four stats words."""
    st = torch.tensor([amax, -1.0, -1.0, -1.0], dtype=torch.float32, device="cuda")
    sc = torch.tensor([sy, sh, w1s, w2s], dtype=torch.float32, device="cuda")
    d_ln2 = empty_bf16(N, C)
    dw1 = dev(dw_init[0]) if dw_init else empty_bf16(2 * H, C)
    dw2 = dev(dw_init[1]) if dw_init else empty_bf16(C, H)
    ws = torch.empty(q.qffn_ffn_backward_workspace_size(N, C, H), dtype=torch.uint8, device="cuda")
    q.qffn_ffn_backward(d_ln2, dw1, dw2, st[0:2], st[2:4], dev(dout), dev(yq), sc[0:1], dev(hq), sc[1:2],
                        dev(w1q), sc[2:3], dev(w2q), sc[3:4], N, C, H, acc, ws)
    q.qffn_check_status()
    sync()
    off = q.qffn_ffn_backward_workspace_offsets(N, C, H)
    # the recomputed gate|up product is not kept by the chain: the unfused GEMM makes it
    gu = empty_bf16(N, 2 * H)
    q.qffn_fp8_gemm_scaled(gu, dev(yq), sc[0:1], dev(w1q), sc[2:3], N, 2 * H, C)
    sync()
    return dict(d_ln2=d_ln2, dw1=dw1, dw2=dw2, st=host(st), gu=gu,
                dh=ws[off[0]:off[0] + N * H * 2].view(torch.int16).view(N, H),
                dgu=ws[off[1]:off[1] + N * 2 * H * 2].view(torch.int16).view(N, 2 * H))


def _ffn_backward_gpu(*a, **k):
    g = _ffn_backward_dev(*a, **k)
    return {key: (v if key == "st" else bf(v)) for key, v in g.items()}


@pytest.mark.parametrize("N,C,H", [(64, 256, 768), (1, 128, 128), (200, 384, 256), (513, 2048, 1024)])
def test_gate_up_swiglu_backward_equals_unfused(q, N, C, H):
    """The fused recompute + swiglu_backward equals the unfused GEMM into [N, 2H]
    followed by qffn_swiglu_backward, bit for bit, abs-max included."""
    yq, sy = oracle.quantize_tensor(random_bf16((N, C), seed=N + C))
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), seed=H + C, std=0.02))
    dh = random_bf16((N, H), seed=N + H, std=1e-3)
    sc = torch.tensor([sy, w1s], dtype=torch.float32, device="cuda")
    yqd, w1d, dhd = dev(yq), dev(w1q), dev(dh)
    gu = empty_bf16(N, 2 * H)
    q.qffn_fp8_gemm_scaled(gu, yqd, sc[0:1], w1d, sc[1:2], N, 2 * H, C)
    d_ref = empty_bf16(N, 2 * H)
    st_ref = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_swiglu_backward(d_ref, st_ref, dhd, gu, N, H)
    d = empty_bf16(N, 2 * H)
    st = torch.full((2,), 3.0, dtype=torch.float32, device="cuda")
    q.qffn_gate_up_swiglu_backward(d, st, dhd, yqd, sc[0:1], w1d, sc[1:2], N, C, H)
    q.qffn_check_status()
    sync()
    np.testing.assert_array_equal(bf(d), bf(d_ref))
    assert host(st)[0] == host(st_ref)[0] and host(st)[1] == 3.0
    _check_swiglu_grad(bf(d), oracle.swiglu_backward(dh, bf(gu), H)[0])


def _backward_inputs(N, C, H, seed):
    dout = random_bf16((N, C), seed=seed, std=1e-3)
    yq, sy = oracle.quantize_tensor(random_bf16((N, C), seed=seed + 1))
    h = oracle.swiglu(oracle.f64_to_bf16(np.random.default_rng(seed + 2).standard_normal((N, 2 * H))), H)[0]
    hq, sh = oracle.quantize_tensor(h)
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), seed=seed + 3, std=0.02))
    w2q, w2s = oracle.quantize_tensor(random_bf16((C, H), seed=seed + 4, std=0.02))
    return dout, yq, sy, hq, sh, w1q, w1s, w2q, w2s


@pytest.mark.parametrize("N,C,H", [(64, 256, 768), (512, 1024, 2048)])
def test_ffn_backward_stagewise_and_end_to_end(q, N, C, H):
    dout, yq, sy, hq, sh, w1q, w1s, w2q, w2s = _backward_inputs(N, C, H, N + C + H)
    amax = oracle.absmax(dout)
    g = _ffn_backward_gpu(q, dout, amax, yq, sy, hq, sh, w1q, w1s, w2q, w2s, N, C, H)
    st = g["st"]
    # down projection, fed the same dout
    rdh, rdw2, rq, rs = oracle.backward_qmm(dout, amax, hq, sh, w2q, w2s)
    assert st[1] == rs
    _check_gemm(g["dh"], rdh, rq, rs, w2q.T, w2s)
    _check_gemm(g["dw2"], rdw2, rq.T, rs, hq.T, sh)
    # recomputed up-projection output
    _check_gemm(g["gu"], oracle.fp8_gemm_scaled(yq, sy, w1q, w1s), yq, sy, w1q, w1s)
    # swiglu_backward on the GPU's own dh and gate|up
    rdgu, _ = oracle.swiglu_backward(g["dh"], g["gu"], H)
    _check_swiglu_grad(g["dgu"], rdgu)
    assert st[2] == np.float32(np.max(np.abs(oracle.bf16_to_f64(g["dgu"]))))
    # up projection, fed the GPU's own d_gate_up and its abs-max
    rdl, rdw1, rq1, rs1 = oracle.backward_qmm(g["dgu"], st[2], yq, sy, w1q, w1s)
    assert st[3] == rs1
    _check_gemm(g["d_ln2"], rdl, rq1, rs1, w1q.T, w1s)
    _check_gemm(g["dw1"], rdw1, rq1.T, rs1, yq.T, sy)
    # end to end against the oracle chain: the block-output tolerance
    ref = oracle.ffn_backward(dout, amax, yq, sy, hq, sh, w1q, w1s, w2q, w2s, H)
    for k in ("d_ln2", "dw1", "dw2"):
        assert_out_close(g[k], ref[k])


def test_ffn_backward_accumulates_weight_gradients(q):
    N, C, H = 64, 256, 256
    args = _backward_inputs(N, C, H, 17)
    dout = args[0]
    amax = oracle.absmax(dout)
    old1, old2 = random_bf16((2 * H, C), seed=41, std=1e-2), random_bf16((C, H), seed=42, std=1e-2)
    g0 = _ffn_backward_gpu(q, dout, amax, *args[1:], N, C, H)
    g1 = _ffn_backward_gpu(q, dout, amax, *args[1:], N, C, H, acc=True, dw_init=(old1, old2))
    np.testing.assert_array_equal(g1["d_ln2"], g0["d_ln2"])              # dinp is not accumulated
    yq, sy, hq, sh, w1q, w1s, w2q, w2s = args[1:]
    _, rdw2, rq, rs = oracle.backward_qmm(dout, amax, hq, sh, w2q, w2s, old2)
    _check_gemm(g1["dw2"], rdw2, rq.T, rs, hq.T, sh, old=old2)
    _, rdw1, rq1, rs1 = oracle.backward_qmm(g1["dgu"], g1["st"][2], yq, sy, w1q, w1s, old1)
    _check_gemm(g1["dw1"], rdw1, rq1.T, rs1, yq.T, sy, old=old1)


def test_ffn_backward_8b_shape_sampled(q):
    """The Llama-3-8B FFN backward (N=16384, C=4096, H=14336) in the configuration the
    benchmark times, checked on sampled outputs stage by stage: each stage is fed the
    GPU's own upstream tensors, and weight-gradient entries are sampled dot products
    over all tokens.  The forward's quantised SwiGLU output is a random code tensor."""
    N, C, H = 16384, 4096, 14336
    dout = random_bf16((N, C), seed=99, std=1e-3)
    yq, sy = oracle.quantize_tensor(random_bf16((N, C), seed=100))
    hq, sh = random_codes((N, H), seed=101), np.float32(1 / 448.0)
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), seed=102, std=0.02))
    w2q, w2s = oracle.quantize_tensor(random_bf16((C, H), seed=103, std=0.02))
    amax = oracle.absmax(dout)
    g = _ffn_backward_dev(q, dout, amax, yq, sy, hq, sh, w1q, w1s, w2q, w2s, N, C, H)
    st = g["st"]
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(N, 12, replace=False))
    ridx = torch.from_numpy(rows).cuda()
    dq, ds = oracle.quantize_with_abs_max(dout, amax)
    assert st[1] == ds
    dh_r, gu_r, dgu_r = (bf(g[k].index_select(0, ridx)) for k in ("dh", "gu", "dgu"))
    rdh = oracle.fp8_gemm_scaled(dq[rows], ds, np.ascontiguousarray(w2q.T), w2s)
    _check_gemm(dh_r, rdh, dq[rows], ds, w2q.T, w2s)
    rgu = oracle.fp8_gemm_scaled(yq[rows], sy, w1q, w1s)
    _check_gemm(gu_r, rgu, yq[rows], sy, w1q, w1s)
    _check_swiglu_grad(dgu_r, oracle.swiglu_backward(dh_r, gu_r, H)[0])
    # the recorded abs-max of d_gate_up is the max of the GPU's own tensor
    assert st[2] == float(g["dgu"].view(torch.bfloat16).abs().max().float())
    gq_r, gs = oracle.quantize_with_abs_max(dgu_r, st[2])
    assert st[3] == gs
    rdl = oracle.fp8_gemm_scaled(gq_r, gs, np.ascontiguousarray(w1q.T), w1s)
    # a 28672-term reduction of gradient products cancels heavily (|sum| ~ sum|terms| /
    # sqrt(K)), so fp32 accumulation flips the bf16 rounding of more outputs than in the
    # forward; every output still meets the error bound, and at most 1% may differ
    _check_gemm(bf(g["d_ln2"].index_select(0, ridx)), rdl, gq_r, gs, w1q.T, w1s, max_mismatch=1e-2)
    # weight gradients: 16 x 16 sampled entries each, dot products over all N tokens
    oi = np.sort(rng.choice(C, 16, replace=False))
    ii = np.sort(rng.choice(H, 16, replace=False))
    want = oracle.fp8_gemm_scaled(np.ascontiguousarray(dq[:, oi].T), ds, np.ascontiguousarray(hq[:, ii].T), sh)
    got = bf(g["dw2"])[np.ix_(oi, ii)]
    _check_gemm(got, want, dq[:, oi].T, ds, hq[:, ii].T, sh, max_mismatch=2e-2)
    oi = np.sort(rng.choice(2 * H, 16, replace=False))
    ii = np.sort(rng.choice(C, 16, replace=False))
    gq_c, _ = oracle.quantize_with_abs_max(bf(g["dgu"].index_select(1, torch.from_numpy(oi).cuda())), st[2])
    want = oracle.fp8_gemm_scaled(np.ascontiguousarray(gq_c.T), gs, np.ascontiguousarray(yq[:, ii].T), sy)
    got = bf(g["dw1"])[np.ix_(oi, ii)]
    _check_gemm(got, want, gq_c.T, gs, yq[:, ii].T, sy, max_mismatch=2e-2)


@pytest.mark.parametrize("acc", [False, True])
def test_ffn_backward_graph_capture_equals_eager(q, acc):
    """qffn_ffn_backward captured in a CUDA graph (its memsets and launches become graph
    nodes) and replayed twice gives the eager call's bits: the gradients, the stats
    words and the workspace's dh and d_gate_up."""
    N, C, H = 208, 384, 256
    dout, yq, sy, hq, sh, w1q, w1s, w2q, w2s = _backward_inputs(N, C, H, 23)
    amax = oracle.absmax(dout)
    dw_init = (random_bf16((2 * H, C), seed=31, std=1e-3), random_bf16((C, H), seed=32, std=1e-3))
    sc = torch.tensor([sy, sh, w1s, w2s], dtype=torch.float32, device="cuda")
    d_dout, d_yq, d_hq, d_w1, d_w2 = dev(dout), dev(yq), dev(hq), dev(w1q), dev(w2q)
    ws_bytes = q.qffn_ffn_backward_workspace_size(N, C, H)
    off = q.qffn_ffn_backward_workspace_offsets(N, C, H)

    def buffers():
        return dict(d_ln2=empty_bf16(N, C), dw1=dev(dw_init[0]), dw2=dev(dw_init[1]),
                    st=torch.tensor([amax, -1.0, -1.0, -1.0], dtype=torch.float32, device="cuda"),
                    ws=torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda"))

    def run(b, stream=None):
        q.qffn_ffn_backward(b["d_ln2"], b["dw1"], b["dw2"], b["st"][0:2], b["st"][2:4], d_dout, d_yq, sc[0:1],
                            d_hq, sc[1:2], d_w1, sc[2:3], d_w2, sc[3:4], N, C, H, acc, b["ws"], stream=stream)

    def snap(b):
        out = {k: host(b[k]).copy() for k in ("d_ln2", "dw1", "dw2", "st")}
        out["dh"] = host(b["ws"][off[0]:off[0] + N * H * 2]).copy()
        out["dgu"] = host(b["ws"][off[1]:off[1] + N * 2 * H * 2]).copy()
        return out

    eager = buffers()
    run(eager)
    q.qffn_check_status()
    sync()
    want = snap(eager)
    b = buffers()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run(b, stream=stream)
    for _ in range(2):
        # the accumulating form adds into dW: start each replay from the same contents
        b["dw1"].copy_(dev(dw_init[0]))
        b["dw2"].copy_(dev(dw_init[1]))
        b["st"].copy_(torch.tensor([amax, -1.0, -1.0, -1.0]))
        b["d_ln2"].fill_(-7)
        b["ws"].zero_()
        graph.replay()
        sync()
        got = snap(b)
        for k in want:
            assert np.array_equal(got[k], want[k]), k
    q.qffn_check_status()
