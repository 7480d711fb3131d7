"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every function include/mxfp8.h declares, its pure size helpers agree with
the oracle's layout, and invalid arguments are rejected on the host before
any device work."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import mxfp8_block_scaled_gb300 as mx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(mx.LIB_PATH):
        from mxfp8_block_scaled_gb300 import build
        build.build()
    return mx.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mx_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_function(L):
    names = declared_functions()
    assert names == set(mx.EXPORTED), names ^ set(mx.EXPORTED)
    for n in names:
        assert hasattr(L, n), n
    out = os.popen(f"nm -D --defined-only {mx.LIB_PATH}").read()
    for n in names:
        assert re.search(rf"\bT {n}\b", out), f"{n} not exported"


def test_version_and_strings(L):
    assert mx.mx_abi_version() == 1
    for code, name in mx.STATUS_NAMES.items():
        assert mx.mx_status_string(code).startswith(name)


@pytest.mark.parametrize("rows,k", [(1, 32), (128, 128), (129, 160), (256, 512), (8192, 2048),
                                    (10944, 8192), (576, 16384), (7, 7168)])
def test_scale_bytes_matches_oracle_layout(L, rows, k):
    assert mx.mx_scale_bytes(rows, k) == oracle.mx_scale_nbytes(rows, k)


def test_scale_bytes_degenerate(L):
    assert mx.mx_scale_bytes(0, 128) == 0 and mx.mx_scale_bytes(128, 0) == 0


def test_grouped_padded_rows(L):
    offs = [0, 20, 20, 170, 171, 299]
    assert mx.mx_grouped_padded_rows(offs) == int(oracle.mx_padded_offsets(np.array(offs))[-1])
    assert mx.mx_grouped_padded_rows([0, 5, 3]) == -1
    assert mx.mx_grouped_padded_rows([1, 5]) == -1


def _op(data=0x1000, scale=0x2000, rows=128, k=256, ld=0, orient=mx.MX_ROWWISE):
    return mx.MXOperandC(data, scale, rows, k, ld, orient, 0)


def _status_of(fn, *args):
    try:
        fn(*args)
    except mx.MXError as e:
        return e.status
    return 0


INVALID, SHAPE, ALIGN = 1, 2, 3


def test_gemm_rejects_bad_arguments_on_host(L):
    c = 0x4000
    # orientation vs mode (direction table)
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(), _op(orient=mx.MX_COLWISE), c, 128, None, None) == INVALID
    assert _status_of(mx.mx_gemm, mx.MX_DGRAD, _op(), _op(), c, 128, None, None) == INVALID
    assert _status_of(mx.mx_gemm, mx.MX_WGRAD, _op(), _op(orient=mx.MX_COLWISE), c, 128, None, None) == INVALID
    assert _status_of(mx.mx_gemm, 7, _op(), _op(), c, 128, None, None) == INVALID
    # K not a multiple of 32, mismatched K
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(k=48), _op(k=48), c, 128, None, None) == SHAPE
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(k=64), _op(k=96), c, 128, None, None) == INVALID
    # alignment of data, scale, ld, output
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(data=0x1008), _op(), c, 128, None, None) == ALIGN
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(scale=0x2004), _op(), c, 128, None, None) == ALIGN
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(ld=264), _op(ld=264), c, 128, None, None) == ALIGN
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(), _op(), 0x4001, 128, None, None) == ALIGN
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(), _op(), c, 100, None, None) == INVALID  # ldc < N
    # null pointers, negative sizes, ld < k, reserved field
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(data=0), _op(), c, 128, None, None) == INVALID
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(), _op(), 0, 128, None, None) == INVALID
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(rows=-1), _op(), c, 128, None, None) == INVALID
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, _op(ld=128), _op(), c, 128, None, None) == INVALID
    bad = _op()
    bad.reserved = 1
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, bad, _op(), c, 128, None, None) == INVALID
    assert _status_of(mx.mx_gemm, mx.MX_FPROP, None, _op(), c, 128, None, None) != 0


def test_gemm_workspace_entry_points_validate_on_host(L):
    c, ws = 0x4000, 0x100000
    q = mx.mx_gemm_with_workspace
    # the operand checks are mx_gemm's
    assert _status_of(q, mx.MX_DGRAD, _op(), _op(), c, 128, ws, 1 << 20, None, None) == INVALID
    assert _status_of(q, mx.MX_FPROP, _op(k=48), _op(k=48), c, 128, ws, 1 << 20, None, None) == SHAPE
    assert _status_of(q, mx.MX_FPROP, _op(), _op(), c, 100, ws, 1 << 20, None, None) == INVALID
    # a workspace of non-zero size must be a 16-byte aligned pointer
    assert _status_of(q, mx.MX_FPROP, _op(), _op(), c, 128, None, 1 << 20, None, None) == INVALID
    assert _status_of(q, mx.MX_FPROP, _op(), _op(), c, 128, ws + 8, 1 << 20, None, None) == ALIGN
    # empty problems are no-ops with or without a workspace
    assert _status_of(q, mx.MX_FPROP, _op(rows=0), _op(), c, 128, None, 0, None, None) == 0
    w = mx.mx_gemm_workspace_bytes
    assert _status_of(w, mx.MX_FPROP, _op(), _op(orient=mx.MX_COLWISE)) == INVALID
    assert _status_of(w, mx.MX_FPROP, _op(k=48), _op(k=48)) == SHAPE
    assert w(mx.MX_FPROP, _op(rows=0), _op()) == 0
    assert L.mx_gemm_workspace_bytes(mx.MX_FPROP, _op(), _op(), None) == INVALID  # null result pointer
    # a valid query needs the device's SM count: an error status without a GPU
    assert _status_of(w, mx.MX_FPROP, _op(), _op()) in (0, 4, 7)


def _gp(mode=mx.MX_FPROP, a=None, b=None, c=0x4000, ldc=128):
    return mx.MXGemmProblemC(a or _op(), b or _op(), c, ldc, mode, 0)


def test_gemm_multi_rejects_bad_arguments_on_host(L):
    q = mx.mx_gemm_multi
    good = _gp()
    assert _status_of(q, [good, _gp(mode=mx.MX_DGRAD)], None, None) == INVALID      # orientation vs mode
    assert _status_of(q, [good, _gp(a=_op(k=48), b=_op(k=48))], None, None) == SHAPE
    assert _status_of(q, [_gp(c=0x4001)], None, None) == ALIGN
    assert _status_of(q, [_gp(ldc=100)], None, None) == INVALID
    bad = _gp()
    bad.reserved = 1
    assert _status_of(q, [good, bad], None, None) == INVALID
    assert _status_of(q, [good] * (mx.MX_MAX_GEMM_MULTI + 1), None, None) == INVALID
    assert _status_of(q, [], None, None) == 0
    assert _status_of(q, [_gp(a=_op(rows=0)), _gp(b=_op(rows=0))], None, None) == 0   # empty problems
    assert "problem 1" in (lambda: (_status_of(q, [good, _gp(ldc=100)], None, None), mx.mx_last_error())[1])()


def test_grouped_gemm_rejects_bad_arguments_on_host(L):
    c = 0x4000
    g = 0x8000
    assert _status_of(mx.mx_grouped_gemm, mx.MX_FPROP, _op(), _op(), None, 4, c, 128, None, None) == INVALID
    assert _status_of(mx.mx_grouped_gemm, mx.MX_FPROP, _op(), _op(), g, 0, c, 128, None, None) == INVALID
    # wgrad needs a capacity that is a multiple of 128
    a = _op(orient=mx.MX_COLWISE, k=160)
    assert _status_of(mx.mx_grouped_gemm, mx.MX_WGRAD, a, _op(orient=mx.MX_COLWISE, k=160), g, 2, c, 128,
                      None, None) == SHAPE


def test_group_limit_rejected_on_host(L):
    """n_groups above MX_MAX_GROUPS (512) is MX_ERR_UNSUPPORTED_SHAPE from every
    grouped call, decided on the host: the pointers here are not device memory
    and no GPU exists, so a launch or a device read could not have happened."""
    g, c, x = 0x8000, 0x4000, 0x10000
    assert mx.MX_MAX_GROUPS == 512
    for n in (513, 1024):
        assert _status_of(mx.mx_grouped_gemm, mx.MX_FPROP, _op(), _op(), g, n, c, 128, None, None) == SHAPE
        assert _status_of(mx.mx_grouped_gemm, mx.MX_WGRAD, _op(orient=mx.MX_COLWISE, k=256),
                          _op(orient=mx.MX_COLWISE, k=256), g, n, c, 128, None, None) == SHAPE
        assert _status_of(mx.mx_grouped_gemm_swiglu, _op(), _op(rows=256), g, n, c, 128, None, None) == SHAPE
        assert _status_of(mx.mx_quantize, x, 64, 64, 64, 2, None, None, 0x1000, 0x2000, g, n, 128, None,
                          None) == SHAPE
        assert "MX_MAX_GROUPS" in mx.mx_last_error()


def test_quantize_rejects_bad_arguments_on_host(L):
    x = 0x10000
    assert _status_of(mx.mx_quantize, x, 64, 64, 64, 0, 0x1000, 0x2000, None, None, None, 0, 0, None, None) == INVALID
    assert _status_of(mx.mx_quantize, x, 64, 48, 48, 1, 0x1000, 0x2000, None, None, None, 0, 0, None, None) == SHAPE
    assert _status_of(mx.mx_quantize, x, 48, 64, 64, 2, None, None, 0x1000, 0x2000, None, 0, 0, None, None) == SHAPE
    assert _status_of(mx.mx_quantize, x + 2, 64, 64, 64, 1, 0x1000, 0x2000, None, None, None, 0, 0, None,
                      None) == ALIGN
    assert _status_of(mx.mx_quantize, x, 64, 64, 68, 1, 0x1000, 0x2000, None, None, None, 0, 0, None,
                      None) == ALIGN
    assert _status_of(mx.mx_quantize, x, 64, 64, 64, 1, None, 0x2000, None, None, None, 0, 0, None,
                      None) == INVALID
    assert _status_of(mx.mx_quantize, x, 64, 64, 32, 1, 0x1000, 0x2000, None, None, None, 0, 0, None,
                      None) == INVALID
    # grouped: only for the column copy; capacity multiple of 128; n_groups >= 1
    assert _status_of(mx.mx_quantize, x, 64, 64, 64, 1, 0x1000, 0x2000, None, None, 0x9000, 2, 128, None,
                      None) == INVALID
    assert _status_of(mx.mx_quantize, x, 64, 64, 64, 2, None, None, 0x1000, 0x2000, 0x9000, 2, 100, None,
                      None) == SHAPE
    assert _status_of(mx.mx_quantize, x, 64, 64, 64, 2, None, None, 0x1000, 0x2000, 0x9000, 0, 128, None,
                      None) == INVALID
    # empty input: nothing to do, OK without touching the device
    assert _status_of(mx.mx_quantize, 0, 0, 64, 64, 1, None, None, None, None, None, 0, 0, None, None) == 0


def test_quantize_batched_rejects_bad_arguments_on_host(L):
    x = 0x10000
    q = mx.mx_quantize_batched
    assert _status_of(q, x, -1, 64, 64, 64, 4096, 3, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == INVALID
    assert _status_of(q, x, 2, 64, 64, 64, 100, 3, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == INVALID
    assert _status_of(q, x, 2, 64, 64, 64, 4100, 3, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == ALIGN
    assert _status_of(q, x, 2, 48, 64, 64, 4096, 3, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == SHAPE
    assert _status_of(q, x, 2, 64, 64, 64, 4096, 0, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == INVALID
    assert _status_of(q, x, 2, 64, 64, 64, 4096, 3, None, 0x2000, 0x3000, 0x4000, None, None) == INVALID
    assert _status_of(q, x, 0, 64, 64, 64, 4096, 3, None, None, None, None, None, None) == 0


def test_quantize_f32_rejects_bad_arguments_on_host(L):
    x = 0x10000
    q = mx.mx_quantize_f32
    assert _status_of(q, x, 1, 64, 64, 66, 0, 3, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == ALIGN  # ldx % 4
    assert _status_of(q, x + 8, 1, 64, 64, 64, 0, 3, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == ALIGN
    assert _status_of(q, x, 2, 64, 64, 64, 4098, 3, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == ALIGN
    assert _status_of(q, x, 2, 64, 64, 64, 100, 3, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == INVALID
    assert _status_of(q, x, 1, 64, 48, 48, 0, 1, 0x1000, 0x2000, None, None, None, None) == SHAPE
    assert _status_of(q, x, 1, 48, 64, 64, 0, 2, None, None, 0x3000, 0x4000, None, None) == SHAPE
    assert _status_of(q, x, 1, 64, 64, 64, 0, 3, None, 0x2000, 0x3000, 0x4000, None, None) == INVALID
    assert _status_of(q, x, 1, 64, 64, 64, 0, 9, 0x1000, 0x2000, 0x3000, 0x4000, None, None) == INVALID
    assert _status_of(q, x, 0, 64, 64, 64, 0, 3, None, None, None, None, None, None) == 0
    # a BF16-legal pitch of 66 elements is not a 16-byte FP32 pitch; 68 is
    assert _status_of(q, 0, 1, 64, 64, 68, 0, 1, 0x1000, 0x2000, None, None, None, None) == INVALID


def _qt(x=0x10000, rows=64, cols=64, ldx=None, rd=0x1000, rs=0x2000, cd=0x3000, cs=0x4000):
    return mx.MXQuantTensorC(x, rows, cols, cols if ldx is None else ldx, rd, rs, cd, cs)


def test_quantize_multi_rejects_bad_arguments_on_host(L):
    q = mx.mx_quantize_multi
    good = _qt()
    assert _status_of(q, [good, _qt(cols=48)], 3, None, None) == SHAPE          # cols % 32
    assert _status_of(q, [good, _qt(rows=48)], 3, None, None) == SHAPE          # rows % 32, column copy
    assert _status_of(q, [_qt(rows=-1)], 3, None, None) == INVALID
    assert _status_of(q, [_qt(ldx=32)], 3, None, None) == INVALID               # ldx < cols
    assert _status_of(q, [_qt(ldx=68)], 3, None, None) == ALIGN                 # ldx % 8
    assert _status_of(q, [_qt(x=0x10008)], 3, None, None) == ALIGN
    assert _status_of(q, [_qt(x=0)], 3, None, None) == INVALID
    assert _status_of(q, [good, _qt(cd=None)], 3, None, None) == INVALID        # requested output null
    assert _status_of(q, [_qt(rs=0x2008)], 1, None, None) == ALIGN
    assert _status_of(q, [good], 0, None, None) == INVALID                      # axis
    assert _status_of(q, [good] * (mx.MX_MAX_MULTI + 1), 3, None, None) == INVALID
    # rows % 32 only binds the column copy; empty matrices and n == 0 are no-ops
    assert _status_of(q, [_qt(rows=48, x=0, cd=None, cs=None, ldx=64)], 1, None, None) == INVALID  # null x
    assert _status_of(q, [_qt(rows=0, x=0, rd=None, rs=None, cd=None, cs=None)], 3, None, None) == 0
    assert _status_of(q, [], 3, None, None) == 0
    assert _status_of(q, [_qt(cols=0, x=0, rd=None, rs=None, cd=None, cs=None)], 3, None, None) == 0


def test_grouped_gemm_swiglu_rejects_bad_arguments_on_host(L):
    c, g = 0x4000, 0x8000
    q = mx.mx_grouped_gemm_swiglu
    assert _status_of(q, _op(rows=512), _op(rows=384), g, 2, c, 192, None, None) == SHAPE       # 2F % 256
    assert _status_of(q, _op(rows=512), _op(rows=512, orient=mx.MX_COLWISE), g, 2, c, 256, None, None) == INVALID
    assert _status_of(q, _op(rows=512), _op(rows=512), None, 2, c, 256, None, None) == INVALID
    assert _status_of(q, _op(rows=512), _op(rows=512), g, 0, c, 256, None, None) == INVALID
    assert _status_of(q, _op(rows=512, k=256), _op(rows=512, k=512), g, 2, c, 256, None, None) == INVALID
    assert _status_of(q, _op(rows=512), _op(rows=512), g, 2, c, 100, None, None) == INVALID   # ldc < F


def test_blockwise_rejects_bad_arguments_on_host(L):
    q = mx.mx_quantize_fp8_blockwise
    x, d, sc = 0x10000, 0x20000, 0x30000
    assert _status_of(q, x, 64, 128, 128, 2, d, sc, None, None) == INVALID          # block
    assert _status_of(q, x, 64, 96, 96, 1, d, sc, None, None) == SHAPE              # cols % 128
    assert _status_of(q, x + 8, 64, 128, 128, 1, d, sc, None, None) == ALIGN
    assert _status_of(q, x, 64, 128, 132, 1, d, sc, None, None) == ALIGN           # ldx % 8
    assert _status_of(q, x, 64, 128, 128, 1, None, sc, None, None) == INVALID
    assert _status_of(q, x, 0, 128, 128, 1, None, None, None, None) == 0
    g = mx.mx_gemm_fp8_blockwise
    c = 0x40000
    assert _status_of(g, x, sc, 64, d, sc, 64, 192, c, 64, None, None) == SHAPE    # K % 128
    assert _status_of(g, x, sc, 64, d, sc, 64, 128, c, 32, None, None) == INVALID  # ldc < N
    assert _status_of(g, x + 4, sc, 64, d, sc, 64, 128, c, 64, None, None) == ALIGN
    assert _status_of(g, x, sc + 2, 64, d, sc, 64, 128, c, 64, None, None) == ALIGN
    assert _status_of(g, None, sc, 64, d, sc, 64, 128, c, 64, None, None) == INVALID


def test_selftest_rejects_bad_arguments_on_host(L):
    assert _status_of(mx.mx_selftest_wait_timeout, 0, 0x1000, None) == INVALID
    assert _status_of(mx.mx_selftest_wait_timeout, 1000000, None, None) == INVALID
    assert _status_of(mx.mx_selftest_wait_timeout, 20 * 10 ** 9, 0x1000, None) == INVALID


def test_static_workspace_gemm_validates_on_host(L):
    c = 0x4000
    q = mx.mx_gemm_static_workspace
    assert _status_of(q, mx.MX_DGRAD, _op(), _op(), c, 128, None, None) == INVALID
    assert _status_of(q, mx.MX_FPROP, _op(k=48), _op(k=48), c, 128, None, None) == SHAPE
    assert _status_of(q, mx.MX_FPROP, _op(), _op(), c, 100, None, None) == INVALID
    assert _status_of(q, mx.MX_FPROP, _op(rows=0), _op(), c, 128, None, None) == 0   # empty: no device needed
    assert mx.MX_STATIC_WORKSPACE_BYTES == 40 * 1024 * 1024


def test_current_scaling_entry_points_validate_on_host(L):
    x, amax, scale, c = 0x10000, 0x20000, 0x30000, 0x4000
    qc = mx.mx_quantize_current
    # (x, batch, rows, cols, ldx, stride, axis, amax, fmt, row, col, scale, offs, n_groups, cap, status, stream)
    ok = (x, 1, 64, 64, 64, 0, mx.MX_BOTH, amax, 448.0, 0x1000, 0x2000, scale, None, 0, 0, None, None)

    def with_(**kw):
        names = ["x", "batch", "rows", "cols", "ldx", "stride", "axis", "amax", "fmt", "row", "col", "scale", "offs",
                 "n", "cap", "st", "s"]
        a = list(ok)
        for k, v in kw.items():
            a[names.index(k)] = v
        return a
    assert _status_of(qc, *with_(cols=48, ldx=48)) == SHAPE                 # cols % 32
    assert _status_of(qc, *with_(rows=48)) == SHAPE                         # column copy needs rows % 32
    assert _status_of(qc, *with_(axis=0)) == INVALID
    assert _status_of(qc, *with_(fmt=0.0)) == INVALID
    assert _status_of(qc, *with_(fmt=float("inf"))) == INVALID
    assert _status_of(qc, *with_(amax=None)) == INVALID
    assert _status_of(qc, *with_(scale=scale + 2)) == ALIGN
    assert _status_of(qc, *with_(x=x + 2)) == ALIGN
    assert _status_of(qc, *with_(row=None)) == INVALID
    assert _status_of(qc, *with_(col=0x2008)) == ALIGN
    assert _status_of(qc, *with_(ldx=60)) == INVALID                        # ldx < cols
    assert _status_of(qc, *with_(batch=2, stride=100)) == INVALID           # stride < rows * ldx
    # grouped: column copy of one matrix, 1 .. MX_MAX_GROUPS groups, capacity a multiple of 128
    assert _status_of(qc, *with_(offs=0x9000, n=2, cap=100)) == SHAPE
    assert _status_of(qc, *with_(offs=0x9000, n=513, cap=128)) == SHAPE
    assert _status_of(qc, *with_(offs=0x9000, n=2, cap=128, batch=2, stride=64 * 64)) == INVALID
    assert _status_of(qc, *with_(offs=0x9000, n=2, cap=128, axis=mx.MX_ROWWISE)) == INVALID
    assert _status_of(qc, *with_(batch=0)) == 0                             # nothing to do
    am = mx.mx_current_amax
    assert _status_of(am, x, 1, 64, 48, 48, 0, amax, None, None) == SHAPE
    assert _status_of(am, x, 1, 64, 64, 64, 0, None, None, None) == INVALID
    assert _status_of(am, x, 1, 64, 64, 64, 0, amax + 1, None, None) == ALIGN
    assert _status_of(am, x, 0, 64, 64, 64, 0, amax, None, None) == 0
    # GEMMs: an FP32 scale needs only 4-byte alignment; the rest is mx_gemm's checking
    g = mx.mx_gemm_current
    assert _status_of(g, mx.MX_FPROP, _op(scale=0x2004), _op(), c, 128, None, None) != ALIGN
    assert _status_of(g, mx.MX_FPROP, _op(scale=0x2002), _op(), c, 128, None, None) == ALIGN
    assert _status_of(g, mx.MX_FPROP, _op(scale=0), _op(), c, 128, None, None) == INVALID
    assert _status_of(g, mx.MX_DGRAD, _op(), _op(), c, 128, None, None) == INVALID
    assert _status_of(g, mx.MX_FPROP, _op(k=48), _op(k=48), c, 128, None, None) == SHAPE
    gg = mx.mx_grouped_gemm_current
    assert _status_of(gg, mx.MX_FPROP, _op(), _op(), None, 4, c, 128, None, None) == INVALID
    assert _status_of(gg, mx.MX_FPROP, _op(), _op(), 0x8000, 513, c, 128, None, None) == SHAPE
    assert _status_of(gg, mx.MX_WGRAD, _op(orient=mx.MX_COLWISE, k=160), _op(orient=mx.MX_COLWISE, k=160), 0x8000,
                      2, c, 128, None, None) == SHAPE


def test_current_gemm_multi_rejects_bad_arguments_on_host(L):
    """mx_gemm_current_multi: each problem checked as mx_gemm_current (FP32
    scales need only 4-byte alignment), the list as mx_gemm_multi."""
    q = mx.mx_gemm_current_multi
    good = _gp(a=_op(scale=0x2004))
    assert _status_of(q, [good, _gp(mode=mx.MX_DGRAD)], None, None) == INVALID      # orientation vs mode
    assert _status_of(q, [good, _gp(a=_op(scale=0x2002))], None, None) == ALIGN
    assert _status_of(q, [good, _gp(a=_op(scale=0))], None, None) == INVALID
    assert _status_of(q, [good, _gp(a=_op(k=48), b=_op(k=48))], None, None) == SHAPE
    bad = _gp()
    bad.reserved = 1
    assert _status_of(q, [good, bad], None, None) == INVALID
    assert _status_of(q, [good] * (mx.MX_MAX_GEMM_MULTI + 1), None, None) == INVALID
    assert _status_of(q, [], None, None) == 0
    assert _status_of(q, [_gp(a=_op(rows=0)), _gp(b=_op(rows=0))], None, None) == 0   # empty problems
    assert "problem 1" in (lambda: (_status_of(q, [good, _gp(ldc=100)], None, None), mx.mx_last_error())[1])()


def test_grouped_gemm_swiglu_quantize_rejects_bad_arguments_on_host(L):
    """The fused SwiGLU + quantisation entry: the SwiGLU checks, four non-null
    16-byte aligned outputs and a positive column capacity that is a multiple
    of 128; all decided before launch (the pointers are not device memory)."""
    q = mx.mx_grouped_gemm_swiglu_quantize
    g, rd, rs, cd, cs = 0x8000, 0x10000, 0x20000, 0x30000, 0x40000
    ok = (_op(), _op(rows=256), g, 2, rd, rs, cd, cs, 256, None, None)

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return a
    assert _status_of(q, *with_(1, _op(rows=128))) == SHAPE        # 2F not a multiple of 256
    assert _status_of(q, *with_(2, None)) == INVALID                # no group offsets
    assert _status_of(q, *with_(3, 513)) == SHAPE                   # above MX_MAX_GROUPS
    assert _status_of(q, *with_(4, None)) == INVALID
    assert _status_of(q, *with_(7, cs + 8)) == ALIGN
    assert _status_of(q, *with_(8, 100)) == SHAPE                   # capacity not a multiple of 128
    assert _status_of(q, *with_(8, 0)) == SHAPE                     # rows to place, no capacity
    assert _status_of(q, *with_(0, _op(rows=0))) == 0               # nothing to do
