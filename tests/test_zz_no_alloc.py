"""The decode entry point that needs no caller workspace (for callers that cannot
allocate device memory) against the workspace entry point, through the C ABI.

Kept in its own file, collected last, so that a run stopping at the first
failure has run every other test before this one.
"""
import numpy as np
import pytest
import torch

from ffn_inputs import DecodeConfig, decode_inputs

pytestmark = pytest.mark.gpu


def _records(q, w_bits):
    rows, cols = w_bits.shape
    wb = torch.from_numpy(np.ascontiguousarray(w_bits)).view(torch.int16).cuda()
    codes = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    q.qffn_quantize_rows(codes, scales, wb, rows, cols)
    return codes, scales


@pytest.mark.parametrize("C,H", [(4096, 14336), (256, 768),
                                 # the largest sizes the fixed scratch holds: h and u end at its
                                 # end at H = 32768, the slice partials at C = 32768
                                 (64, 32768), (32768, 64)])
def test_noalloc_decode_matches_workspace_decode_twice(C, H):
    import transformer_ffn_block_gb300 as q
    cfg = DecodeConfig("noalloc", C=C, H=H, seed=C + H)
    di = decode_inputs(cfg)
    recs = [t for k in ("w_gate", "w_up", "w_down") for t in _records(q, di[k])]
    ws = torch.zeros(q.qffn_decode_workspace_size(C, H), dtype=torch.uint8, device="cuda")
    g = torch.Generator().manual_seed(7)
    xs = [torch.from_numpy(di["x"]).view(torch.int16).cuda(),
          (torch.randn(C, generator=g)).to(torch.bfloat16).view(torch.int16).cuda()]
    for x in xs:                                   # two calls in a row, different inputs
        want = torch.empty(C, dtype=torch.int16, device="cuda")
        got = torch.full((C,), 0x7FC0, dtype=torch.int16, device="cuda")
        q.qffn_decode_forward(want, x, *recs, C, H, ws)
        stream = torch.cuda.current_stream().cuda_stream
        st = q.lib.qffn_decode_forward_noalloc(got.data_ptr(), x.data_ptr(), *[t.data_ptr() for t in recs],
                                               C, H, stream)
        assert st == 0, q.qffn_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(got, want)              # same kernels: identical bits


def test_noalloc_decode_rejects_oversized_h():
    import transformer_ffn_block_gb300 as q
    p = 1 << 20                                      # never touched: checked on the host first
    st = q.lib.qffn_decode_forward_noalloc(p, p, p, p, p, p, p, p, 4096, 32768 + 16, None)
    assert st == 2                                   # QFFN_ERR_UNSUPPORTED_SHAPE
