"""C-ABI checks that need no GPU: the library builds, loads and exports every
entry point of include/qffn.h, and the host-side argument checks return the
documented status codes before anything is enqueued."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qffn.h")


@pytest.fixture(scope="module")
def lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_qffn_build", os.path.join(ROOT, "transformer_ffn_block_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    path = b.build()
    import transformer_ffn_block_gb300 as q
    assert q.LIB_PATH == path
    return q


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qffn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("qffn_rmsnorm_absmax", "qffn_quantize", "qffn_fp8_gemm_scaled", "qffn_swiglu_quant",
              "qffn_forward", "qffn_decode_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b(qffn_[a-z0-9_]+)\b", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        assert hasattr(lib.lib, n)


def test_status_strings_and_version(lib):
    assert lib.qffn_abi_version() == 1
    for code in range(6):
        assert lib.qffn_status_string(code)
    assert lib.qffn_status_string(99) == "unknown status"


A = 1 << 20          # a fake, 16-byte-aligned address: checks fail before any use
MIS = A + 4           # misaligned
NULL = None


def _call(lib, name, *args):
    return getattr(lib.lib, name)(*args)


def test_rmsnorm_argument_checks(lib):
    f = lambda *a: _call(lib, "qffn_rmsnorm_absmax", *a)
    ok = (A, A, A, A, A, A, A, 1e-5, 4, 256, None)
    bad_null = (A, NULL, A, A, A, A, A, 1e-5, 4, 256, None)
    assert f(*bad_null) == 1
    assert f(A, A, A, A, A, A, A, -1.0, 4, 256, None) == 1            # eps < 0
    assert f(A, A, A, A, A, A, A, float("nan"), 4, 256, None) == 1
    assert f(A, A, A, A, A, A, A, 1e-5, -1, 256, None) == 1
    assert f(A, A, A, A, A, A, A, 1e-5, 4, 12, None) == 2              # C % 8
    assert f(A, A, A, A, A, A, A, 1e-5, 4, 16392, None) == 2           # C > 16384
    assert f(A, MIS, A, A, A, A, A, 1e-5, 4, 256, None) == 3
    assert f(NULL, A, A, A, A, A, A, 1e-5, 4, 256, None) == 1          # res_in given, res_out NULL
    del ok


def test_gemm_argument_checks(lib):
    f = lambda *a: _call(lib, "qffn_fp8_gemm_scaled", *a)
    assert f(A, A, A, A, NULL, 4, 32, 16, None) == 1
    assert f(A, A, A, A, A, 4, 48, 16, None) == 2     # N % 32
    assert f(A, A, A, A, A, 4, 32, 24, None) == 2     # K % 16
    assert f(A, A, A, A, A, 4, 32, 0, None) == 2
    assert f(A, MIS, A, A, A, 4, 32, 16, None) == 3
    g = lambda *a: _call(lib, "qffn_gate_up_swiglu", *a)
    assert g(A, A, A, A, A, A, 4, 256, 200, None) == 2  # H % 128
    assert g(A, A, A, A, A, A, 4, 20, 256, None) == 2   # C % 16


def test_forward_workspace_and_checks(lib):
    assert lib.qffn_forward_workspace_size(2, 32, 256, 768) > 0
    assert lib.qffn_forward_workspace_size(2, 32, 200, 768) == 0
    B, T, C, H = 8, 2048, 4096, 14336
    off = lib.qffn_forward_workspace_offsets(B, T, C, H)
    N = B * T
    assert off[0] == 0 and off[1] >= N * C * 2 and off[2] >= off[1] + N * C
    assert off[3] >= off[2] + N * H * 2
    assert lib.qffn_forward_workspace_size(B, T, C, H) >= off[3] + N * H
    assert all(o % 256 == 0 for o in off)
    f = lambda *a: _call(lib, "qffn_forward", *a)
    ws = lib.qffn_forward_workspace_size(2, 32, 256, 768)
    args = [A, A, A, A, A, A, A, A, 1e-5, A, A, A, A, 2, 32, 256, 768, A, ws, None]
    bad = list(args); bad[17] = A + 16                         # workspace not 256-aligned
    assert f(*bad) == 3
    bad = list(args); bad[18] = ws - 1                         # workspace too small
    assert f(*bad) == 1
    bad = list(args); bad[15] = 192                            # C % 128
    assert f(*bad) == 2
    bad = list(args); bad[8] = -1.0
    assert f(*bad) == 1


def test_decode_checks(lib):
    assert lib.qffn_decode_workspace_size(4096, 14336) >= 4 * 14336
    f = lambda *a: _call(lib, "qffn_decode_forward", *a)
    ws = lib.qffn_decode_workspace_size(4096, 14336)
    assert f(A, A, A, A, A, A, A, A, 4096, 14336, A, ws - 2, None) == 1
    assert f(A, A, A, A, A, A, A, A, 4100, 14336, A, ws, None) == 2
    assert f(A, MIS, A, A, A, A, A, A, 4096, 14336, A, ws, None) == 3
    assert _call(lib, "qffn_gemv", A, A, A, A, 10, 24, None) == 2
    assert _call(lib, "qffn_silu_mul", A, A, 12, None) == 2
    assert _call(lib, "qffn_gemv_silu_input", A, A, A, A, A, 10, 24, None) == 2
    assert _call(lib, "qffn_gemv_silu_input", A, A, NULL, A, A, 10, 32, None) == 1
    assert _call(lib, "qffn_gemv_silu_input", A, A, MIS, A, A, 10, 32, None) == 3
    assert _call(lib, "qffn_quantize_rows", A, A, A, 3, 8, None) == 2


def test_decode_variant_checks(lib):
    ws = lib.qffn_decode_workspace_size(4096, 14336)
    assert ws >= 2 * 2 * 14336                                      # g (then h) and u
    ex = lambda *a: _call(lib, "qffn_decode_forward_ex", *a)
    good = [A, A, A, A, A, A, A, A, 4096, 14336, A, ws]
    assert ex(*good, 2, None) == 1                                   # unknown flag bit
    assert ex(*good[:10], A, ws - 1, 1, None) == 1                  # workspace too small
    assert ex(*good[:10], A + 8, ws, 1, None) == 3                  # workspace alignment
    gu = lambda *a: _call(lib, "qffn_decode_forward_gu", *a)
    assert gu(A, A, NULL, A, A, A, 4096, 14336, A, ws, None) == 1
    assert gu(A, A, A, A, A, A, 4096, 14330, A, ws, None) == 2
    assert gu(A, A, A, A + 2, A, A, 4096, 14336, A, ws, None) == 3  # gu_row_scale


def test_python_binding_raises(lib):
    with pytest.raises(lib.QffnError) as e:
        lib.qffn_gemv(A, A, A, A, 10, 24, stream=0)
    assert e.value.status == 2


def test_recompute_form_checks(lib):
    f = lambda *a: _call(lib, "qffn_swiglu_forward_quant", *a)
    assert f(A, NULL, A, 4, 64, None) == 1
    assert f(A, A, A, 4, 12, None) == 2               # H % 8
    assert f(MIS, A, A, 4, 64, None) == 3
    g = lambda *a: _call(lib, "qffn_gate_up_swiglu_quant", *a)
    assert g(A, A, A, A, A, NULL, 4, 256, 256, None) == 1
    assert g(A, A, A, A, A, A, 4, 256, 200, None) == 2  # H % 128
    assert g(A, A, A, A, A, A, 4, 20, 256, None) == 2   # C % 16
    assert g(A, A, MIS, A, A, A, 4, 256, 256, None) == 3
    h = lambda *a: _call(lib, "qffn_forward_recompute", *a)
    ws = lib.qffn_forward_workspace_size(2, 32, 256, 768)
    args = [A, A, A, A, A, A, A, A, 1e-5, A, A, A, A, 2, 32, 256, 768, A, ws, None]
    bad = list(args); bad[4] = NULL                            # stats_h is required
    assert h(*bad) == 1
    bad = list(args); bad[18] = ws - 1
    assert h(*bad) == 1
    bad = list(args); bad[16] = 200                            # H % 128
    assert h(*bad) == 2
    bad = list(args); bad[17] = A + 16
    assert h(*bad) == 3


def test_qmm_checks(lib):
    f = lambda *a: _call(lib, "qffn_qmm", *a)
    assert f(A, NULL, A, A, NULL, A, A, 4, 32, 16, None) == 1   # q scratch required
    assert f(A, A, A, A, NULL, A, A, 4, 48, 16, None) == 2      # N % 32
    assert f(A, A, A, A, NULL, A, A, 4, 32, 24, None) == 2      # K % 16
    assert f(A, A, A, A, MIS, A, A, 4, 32, 16, None) == 3       # bias misaligned


def test_backward_checks(lib):
    assert lib.qffn_backward_qmm_workspace_size(64, 256, 128) > 0
    assert lib.qffn_backward_qmm_workspace_size(60, 256, 128) == 0          # N % 16
    assert lib.qffn_ffn_backward_workspace_size(64, 256, 768) > 0
    assert lib.qffn_ffn_backward_workspace_size(64, 256, 200) == 0          # H % 128
    off = lib.qffn_ffn_backward_workspace_offsets(64, 256, 768)
    assert off[0] == 0 and off[1] >= 64 * 768 * 2
    assert lib.qffn_ffn_backward_workspace_size(64, 256, 768) >= off[1] + 64 * 1536 * 2
    assert all(o % 256 == 0 for o in off)
    assert _call(lib, "qffn_transpose_e4m3", A, A, 24, 16, None) == 2
    assert _call(lib, "qffn_transpose_e4m3", MIS, A, 16, 16, None) == 3
    assert _call(lib, "qffn_swiglu_backward", A, A, A, A, 4, 12, None) == 2
    ws = lib.qffn_backward_qmm_workspace_size(64, 256, 128)
    f = lambda *a: _call(lib, "qffn_backward_qmm", *a)
    assert f(A, NULL, A, A, A, A, A, A, 64, 256, 128, 0, A, ws, None) == 1   # dw required
    assert f(A, A, A, A, A, A, A, A, 64, 256, 128, 0, A, ws - 1, None) == 1
    assert f(A, A, A, A, A, A, A, A, 64, 250, 128, 0, A, ws, None) == 2
    assert f(A, A, A, A, A, A, A, A, 64, 256, 128, 0, A + 16, ws, None) == 3


def test_bounded_wait_selftest_argument_checks(lib):
    f = lambda *a: _call(lib, "qffn_selftest_bounded_wait", *a)
    assert f(NULL, 0, 1000000, None) == 1
    assert f(A, 0, 99999, None) == 1                  # below 100 us
    assert f(A, 0, 2000000001, None) == 1             # above 2 s
    assert f(A + 4, 0, 1000000, None) == 3            # out not 8-byte aligned


# Every call below fails one host-side check, so nothing is ever enqueued with
# the fake addresses.

def test_absmax_argument_checks(lib):
    f = lambda *a: _call(lib, "qffn_absmax", *a)
    assert f(NULL, A, 16, None) == 1
    assert f(A, NULL, 16, None) == 1
    assert f(A, A, -1, None) == 1
    assert f(A + 2, A, 16, None) == 3                   # stats: 4-byte alignment
    assert f(A, MIS, 16, None) == 3                     # input: 16-byte alignment


def test_gemv_dual_argument_checks(lib):
    f = lambda *a: _call(lib, "qffn_gemv_dual", *a)
    good = [A, A, A, A, A, A, A, 64, 256, None]         # g, u, x, w_gate, s_gate, w_up, s_up, H, C
    for i in range(7):
        bad = list(good)
        bad[i] = NULL
        assert f(*bad) == 1, i
    assert f(A, A, A, A, A, A, A, 0, 256, None) == 1    # H >= 1
    assert f(A, A, A, A, A, A, A, 64, 24, None) == 2    # C % 16
    assert f(A, A, A, A, A, A, A, 64, 32784, None) == 2  # C > 32768
    assert f(A, A, MIS, A, A, A, A, 64, 256, None) == 3  # x
    assert f(A, A, A, MIS, A, A, A, 64, 256, None) == 3  # w_gate
    assert f(A, A, A, A, A + 2, A, A, 64, 256, None) == 3  # s_gate


def test_decode_noalloc_argument_checks(lib):
    f = lambda *a: _call(lib, "qffn_decode_forward_noalloc", *a)
    good = [A, A, A, A, A, A, A, A, 256, 768, None]     # out, x, wg, sg, wu, su, wd, sd, C, H
    for i in range(8):
        bad = list(good)
        bad[i] = NULL
        assert f(*bad) == 1, i
    assert f(A, A, A, A, A, A, A, A, 24, 768, None) == 2      # C % 16
    assert f(A, A, A, A, A, A, A, A, 256, 32784, None) == 2   # H above the library's scratch
    assert f(A, A, A, A, A, A, A, A, 32784, 256, None) == 2   # C above the library's scratch
    assert f(A, MIS, A, A, A, A, A, A, 256, 768, None) == 3   # x
    assert f(A, A, A, A + 2, A, A, A, A, 256, 768, None) == 3  # s_gate


def test_gate_up_swiglu_backward_argument_checks(lib):
    f = lambda *a: _call(lib, "qffn_gate_up_swiglu_backward", *a)
    # d_gate_up, stats, dh, yq, y_scale, w1, w1_scale, N, C, H
    assert f(NULL, A, A, A, A, A, A, 64, 256, 768, None) == 1
    assert f(A, A, NULL, A, A, A, A, 64, 256, 768, None) == 1
    assert f(A, A, A, A, A, A, A, -1, 256, 768, None) == 1
    assert f(A, A, A, A, A, A, A, 64, 24, 768, None) == 2       # C % 16
    assert f(A, A, A, A, A, A, A, 64, 256, 200, None) == 2      # H % 128
    assert f(A, A + 2, A, A, A, A, A, 64, 256, 768, None) == 3  # stats
    assert f(A, A, MIS, A, A, A, A, 64, 256, 768, None) == 3    # dh


def test_ffn_backward_argument_checks(lib):
    f = lambda *a: _call(lib, "qffn_ffn_backward", *a)
    ws = lib.qffn_ffn_backward_workspace_size(64, 256, 768)
    # 14 pointers, N, C, H, accumulate, workspace, workspace_bytes
    good = [A] * 14 + [64, 256, 768, 0, A, ws, None]

    def call(**kw):
        args = list(good)
        for i, v in kw.items():
            args[int(i[1:])] = v
        return f(*args)

    assert call(p0=NULL) == 1                           # d_ln2
    assert call(p13=NULL) == 1                          # w2_scale
    assert call(p18=NULL) == 1                          # workspace
    assert call(p14=-1) == 1                            # N
    assert call(p16=200) == 2                           # H % 128
    assert call(p14=60) == 2                            # N % 16
    assert call(p19=ws - 1) == 1                        # workspace too small
    assert call(p18=A + 16) == 3                        # workspace 256-byte alignment
    assert call(p0=MIS) == 3                            # d_ln2
    assert call(p3=A + 2) == 3                          # stats_dout
