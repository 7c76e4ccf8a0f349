"""Failure detection on the GPU without a fault: the bounded barrier wait that
every GEMM role uses is made to run out on a barrier nothing arrives on; the
host must read QFFN_ERR_TIMEOUT from the device status word, the abort flag
must release the CTA's other waiter, and the context must stay usable (a GEMM
run afterwards gives the same bits as before)."""
import time

import numpy as np
import pytest
import torch

import oracle
from ffn_inputs import random_bf16
from gpu_util import bf, dev, empty_bf16, sync

pytestmark = pytest.mark.gpu

LIMIT_NS = 50_000_000           # 50 ms


@pytest.fixture(scope="module")
def q():
    import transformer_ffn_block_gb300 as q
    return q


def _gemm(q, a, sa, w, sw):
    M, K = a.shape
    N = w.shape[0]
    sc = torch.tensor([sa, sw], dtype=torch.float32, device="cuda")
    out = empty_bf16(M, N)
    q.qffn_fp8_gemm_scaled(out, dev(a), sc[0:1], dev(w), sc[1:2], M, N, K)
    sync()
    return bf(out)


def test_waits_succeed_when_the_barriers_complete(q):
    q.qffn_check_status()
    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    q.qffn_selftest_bounded_wait(out, True, LIMIT_NS)
    q.qffn_check_status()                               # raises on QFFN_ERR_TIMEOUT
    r = out.cpu().numpy()
    assert r[0] == 1 and r[1] == 1
    assert r[2] < LIMIT_NS // 10 and r[3] < LIMIT_NS // 10


def test_wait_runs_out_reports_timeout_and_context_survives(q):
    a, sa = oracle.quantize_tensor(random_bf16((300, 256), seed=1))
    w, sw = oracle.quantize_tensor(random_bf16((512, 256), seed=2, std=0.02))
    before = _gemm(q, a, sa, w, sw)
    q.qffn_check_status()

    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    t0 = time.perf_counter()
    q.qffn_selftest_bounded_wait(out, False, LIMIT_NS)
    with pytest.raises(q.QffnError) as e:
        q.qffn_check_status()
    wall = time.perf_counter() - t0
    assert e.value.status == 5                          # QFFN_ERR_TIMEOUT
    r = out.cpu().numpy()
    assert r[0] == 0 and r[1] == 0                      # neither wait succeeded
    assert LIMIT_NS <= r[2] < LIMIT_NS + 20_000_000     # warp 0 ran out at its limit
    assert r[3] < 2 * LIMIT_NS                          # warp 1 left on the abort flag, not its 4x limit
    assert wall < 5.0

    q.qffn_check_status()                               # the status word was cleared
    after = _gemm(q, a, sa, w, sw)
    np.testing.assert_array_equal(after, before)
    q.qffn_check_status()
