"""GPU grouped GEMM (routed experts) vs the oracle: rows-ragged fprop/dgrad
and contraction-ragged wgrad, with empty, single-row and uneven groups."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import f64, u8

pytestmark = pytest.mark.gpu


def check(out_gpu, ref, S, what):
    out = f64(out_gpu)
    ok = oracle.within_tolerance(out, ref, S)
    if not ok.all():
        bad = np.argwhere(~ok)[:8]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; first "
                             f"{[(tuple(i), out[tuple(i)], ref[tuple(i)]) for i in bad]}")


def setup(counts, K, N, seed):
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    E = len(counts)
    M = int(offs[-1])
    X = workloads.normal_bf16((M, K), seed)
    W = workloads.normal_bf16((E, N, K), seed + 1, 0.02)
    dY = workloads.normal_bf16((M, N), seed + 2)
    return offs, X, W, dY


COUNTS = [[37, 0, 300, 1, 128], [0, 0, 129], [256], [5, 127, 128, 0, 0, 1000, 33, 2]]


@pytest.mark.parametrize("counts", COUNTS)
@pytest.mark.parametrize("N", [192, 320])
def test_grouped_fprop(counts, N):
    K = 256
    offs, X, W, _ = setup(counts, K, N, 10 + N + len(counts))
    o = torch.from_numpy(offs).cuda()
    xr, _ = mx.quantize(X.cuda(), mx.MX_ROWWISE)
    wr, _ = mx.quantize_stacked(W.cuda(), mx.MX_ROWWISE)
    st = mx.new_status()
    y = mx.grouped_gemm(mx.MX_FPROP, xr, wr, o, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    ac, asc = oracle.mx_quantize_rowwise(f64(X))
    wq = [oracle.mx_quantize_rowwise(f64(W[e])) for e in range(len(counts))]
    ref, S = oracle.mx_grouped_gemm_ref_mragged(ac, asc, np.stack([w[0] for w in wq]), np.stack([w[1] for w in wq]),
                                                offs)
    check(y, ref, S, f"grouped fprop {counts} N={N}")


@pytest.mark.parametrize("counts", COUNTS[:2])
def test_grouped_dgrad(counts):
    """dX = dY . W_e per group: a = dY row copy, b = stacked column copies of W."""
    K, N = 192, 256
    offs, _, W, dY = setup(counts, K, N, 50 + len(counts))
    o = torch.from_numpy(offs).cuda()
    dr, _ = mx.quantize(dY.cuda(), mx.MX_ROWWISE)
    _, wc = mx.quantize_stacked(W.cuda(), mx.MX_COLWISE)
    st = mx.new_status()
    dx = mx.grouped_gemm(mx.MX_DGRAD, dr, wc, o, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0 and dx.shape == (int(offs[-1]), K)
    ac, asc = oracle.mx_quantize_rowwise(f64(dY))
    wq = [oracle.mx_quantize_colwise(f64(W[e])) for e in range(len(counts))]
    ref, S = oracle.mx_grouped_gemm_ref_mragged(ac, asc, np.stack([w[0] for w in wq]), np.stack([w[1] for w in wq]),
                                                offs)
    check(dx, ref, S, f"grouped dgrad {counts}")


@pytest.mark.parametrize("counts", COUNTS)
def test_grouped_wgrad(counts):
    """dW_e = dY_e^T X_e over each group's tokens; empty groups give exact zeros."""
    K, N = 192, 320
    offs, X, _, dY = setup(counts, K, N, 70 + len(counts))
    o = torch.from_numpy(offs).cuda()
    cap = mx.mx_grouped_padded_rows(offs) + 128
    _, dc = mx.quantize(dY.cuda(), mx.MX_COLWISE, group_offsets=o, col_capacity=cap)
    _, xc = mx.quantize(X.cuda(), mx.MX_COLWISE, group_offsets=o, col_capacity=cap)
    st = mx.new_status()
    dw = mx.grouped_gemm(mx.MX_WGRAD, dc, xc, o, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0 and dw.shape == (len(counts), N, K)
    a, as_, _ = oracle.mx_quantize_colwise_grouped(f64(dY), offs)
    b, bs, _ = oracle.mx_quantize_colwise_grouped(f64(X), offs)
    ref, S = oracle.mx_grouped_gemm_ref_kragged(a, as_, b, bs, offs)
    check(dw, ref, S, f"grouped wgrad {counts}")
    for e, m in enumerate(counts):
        if m == 0:
            assert bool((dw[e] == 0).all())


def test_one_group_equals_dense_bitwise():
    M, K, N = 300, 256, 384
    X = workloads.normal_bf16((M, K), 90)
    W = workloads.normal_bf16((1, N, K), 91, 0.02)
    xr, _ = mx.quantize(X.cuda(), mx.MX_ROWWISE)
    wr, _ = mx.quantize_stacked(W.cuda(), mx.MX_ROWWISE)
    o = torch.tensor([0, M], dtype=torch.int64, device="cuda")
    yg = mx.grouped_gemm(mx.MX_FPROP, xr, wr, o)
    w2 = mx.MXTensor(wr.data[0], wr.scale[0], N, K, mx.MX_ROWWISE)
    yd = mx.gemm(mx.MX_FPROP, xr, w2)
    torch.cuda.synchronize()
    assert torch.equal(yg.view(torch.int16), yd.view(torch.int16))


def test_bad_offsets_reported_and_nothing_written():
    K, N = 128, 128
    offs, X, W, _ = setup([10, 20], K, N, 95)
    xr, _ = mx.quantize(X.cuda(), mx.MX_ROWWISE)
    wr, _ = mx.quantize_stacked(W.cuda(), mx.MX_ROWWISE)
    for bad in ([0, 20, 10], [0, 10, 31], [1, 10, 30]):
        o = torch.tensor(bad, dtype=torch.int64, device="cuda")
        out = torch.full((30, N), 5.0, dtype=torch.bfloat16, device="cuda")
        st = mx.new_status()
        mx.grouped_gemm(mx.MX_FPROP, xr, wr, o, out=out, status=st)
        torch.cuda.synchronize()
        assert mx.read_status(st) == 5
        assert bool((out == 5.0).all())
