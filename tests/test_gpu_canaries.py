"""Guard bands around output buffers: every output is allocated inside a larger
buffer pre-filled with a canary pattern, and after the call the bytes before and
after the output must be unchanged.  Ragged shapes exercise the tails of the TMA
stores, the predicated epilogue stores and the elementwise kernels."""
import numpy as np
import pytest
import torch

import oracle
from ffn_inputs import random_bf16
from gpu_util import dev, sync

pytestmark = pytest.mark.gpu

GUARD = 4096            # bytes on each side, a multiple of 256 so alignment is kept
CANARY = 0xA5


@pytest.fixture(scope="module")
def q():
    import transformer_ffn_block_gb300 as q
    return q


class Guarded:
    """An output of `nbytes` inside a canary-filled allocation."""

    def __init__(self, nbytes):
        self.buf = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.n = nbytes

    def view(self, dtype, *shape):
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(*shape)

    def check(self, name):
        sync()
        head = self.buf[:GUARD].cpu().numpy()
        tail = self.buf[GUARD + self.n:].cpu().numpy()
        assert np.all(head == CANARY), f"{name}: bytes written before the output"
        assert np.all(tail == CANARY), f"{name}: bytes written after the output"


@pytest.mark.parametrize("N,C,H", [(1, 128, 128), (77, 256, 384), (300, 512, 256), (513, 1024, 1024)])
def test_gate_up_forms_stay_inside_their_outputs(q, N, C, H):
    yq, sy = oracle.quantize_tensor(random_bf16((N, C), seed=N + 1))
    w1q, w1s = oracle.quantize_tensor(random_bf16((2 * H, C), seed=H + 2, std=0.02))
    sc = torch.tensor([sy, w1s], dtype=torch.float32, device="cuda")
    yqd, w1d = dev(yq), dev(w1q)
    h = Guarded(N * H * 2)
    st = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_gate_up_swiglu(h.view(torch.int16, N, H), st, yqd, sc[0:1], w1d, sc[1:2], N, C, H)
    h.check("gate_up_swiglu h")
    hq = Guarded(N * H)
    q.qffn_gate_up_swiglu_quant(hq.view(torch.uint8, N, H), st, yqd, sc[0:1], w1d, sc[1:2], N, C, H)
    hq.check("gate_up_swiglu_quant hq")
    dh = dev(random_bf16((N, H), seed=5, std=1e-3))
    dgu = Guarded(N * 2 * H * 2)
    q.qffn_gate_up_swiglu_backward(dgu.view(torch.int16, N, 2 * H), st, dh, yqd, sc[0:1], w1d, sc[1:2], N, C, H)
    dgu.check("gate_up_swiglu_backward d_gate_up")


@pytest.mark.parametrize("M,N,K", [(1, 32, 16), (129, 288, 144), (300, 544, 512), (1000, 4096, 256)])
def test_gemm_and_qmm_stay_inside_their_outputs(q, M, N, K):
    a, sa = oracle.quantize_tensor(random_bf16((M, K), seed=M + K))
    w, sw = oracle.quantize_tensor(random_bf16((N, K), seed=N + K, std=0.02))
    sc = torch.tensor([sa, sw], dtype=torch.float32, device="cuda")
    out = Guarded(M * N * 2)
    q.qffn_fp8_gemm_scaled(out.view(torch.int16, M, N), dev(a), sc[0:1], dev(w), sc[1:2], M, N, K)
    out.check("fp8_gemm_scaled out")
    x = dev(random_bf16((M, K), seed=3))
    st = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_absmax(st, x, M * K)
    qb = Guarded(M * K)
    out2 = Guarded(M * N * 2)
    bias = dev(random_bf16((N,), seed=4))
    q.qffn_qmm(out2.view(torch.int16, M, N), qb.view(torch.uint8, M, K), st, x, bias, dev(w), sc[1:2], M, N, K)
    qb.check("qmm q")
    out2.check("qmm out")


@pytest.mark.parametrize("acc", [False, True])
@pytest.mark.parametrize("N,IC,OC", [(16, 32, 32), (48, 96, 64), (272, 160, 224)])
def test_backward_qmm_stays_inside_its_outputs(q, N, IC, OC, acc):
    dout = dev(random_bf16((N, OC), seed=N, std=1e-3))
    inq, ins = oracle.quantize_tensor(random_bf16((N, IC), seed=IC))
    wq, ws = oracle.quantize_tensor(random_bf16((OC, IC), seed=OC, std=0.02))
    st = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_absmax(st, dout, N * OC)
    sc = torch.tensor([ins, ws], dtype=torch.float32, device="cuda")
    dinp = Guarded(N * IC * 2)
    dw = Guarded(OC * IC * 2)
    if acc:   # the accumulating form reads the previous dW: give it finite values
        dw.view(torch.int16, OC, IC).copy_(dev(random_bf16((OC, IC), seed=5, std=1e-2)))
    wsb = torch.empty(q.qffn_backward_qmm_workspace_size(N, IC, OC), dtype=torch.uint8, device="cuda")
    q.qffn_backward_qmm(dinp.view(torch.int16, N, IC), dw.view(torch.int16, OC, IC), st, dout, dev(inq), sc[0:1],
                        dev(wq), sc[1:2], N, IC, OC, acc, wsb)
    dinp.check("backward_qmm dinp")
    dw.check("backward_qmm dw")


@pytest.mark.parametrize("N,C", [(1, 8), (37, 264), (300, 4096)])
def test_rmsnorm_and_quantize_stay_inside_their_outputs(q, N, C):
    res, x = dev(random_bf16((N, C), seed=1)), dev(random_bf16((N, C), seed=2))
    gain = dev(random_bf16((C,), seed=3))
    r, y = Guarded(N * C * 2), Guarded(N * C * 2)
    rstd = Guarded(N * 4)
    st = torch.zeros(2, dtype=torch.float32, device="cuda")
    q.qffn_rmsnorm_absmax(r.view(torch.int16, N, C), y.view(torch.int16, N, C), rstd.view(torch.float32, N), st,
                          res, x, gain, 1e-5, N, C)
    for g, name in ((r, "res_out"), (y, "y"), (rstd, "rstd")):
        g.check(name)
    n = N * C - (3 if N * C > 16 else 0)          # a length that is not a multiple of 16
    qo = Guarded(n)
    q.qffn_quantize(qo.view(torch.uint8, n), st, y.view(torch.int16, N, C).view(-1), n)
    qo.check("quantize q")


def test_decode_outputs_stay_inside(q):
    C, H = 256, 768
    x = dev(random_bf16((C,), seed=9))
    recs = []
    for rows, cols, seed in ((H, C, 10), (H, C, 11), (C, H, 12)):
        codes, scales = oracle.quantize_rows(random_bf16((rows, cols), seed=seed, std=0.02))
        recs += [dev(codes), dev(scales)]
    out = Guarded(C * 2)
    ws_bytes = q.qffn_decode_workspace_size(C, H)
    ws = Guarded(ws_bytes)                          # the workspace must stay inside its bytes too
    ws.view(torch.uint8, ws_bytes).zero_()
    q.qffn_decode_forward(out.view(torch.int16, C), x, *recs, C, H, ws.view(torch.uint8, ws_bytes))
    out.check("decode out")
    ws.check("decode workspace")
