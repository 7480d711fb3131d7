"""Seeded random sweep over every entry point, against the oracle: shapes
drawn across tile boundaries (ragged M, N and K, few and many tiles, both
GEMM kernels and the CTA-pair kernel), random group counts with empty and
single-row experts, random pitches and unaligned outputs. Quantisation is
checked bit for bit, GEMMs element by element within the bound."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import check_gemm_full, check_col_copy, check_row_copy, f64

pytestmark = pytest.mark.gpu


def src(g, shape, std=1.0):
    R, C = shape
    x = g.standard_normal(shape) * std
    x *= np.exp2(g.integers(-4, 5, (R, (C + 31) // 32))).repeat(32, axis=1)[:, :C]
    if R * C:
        x.reshape(-1)[g.choice(R * C, size=max(1, R * C // 1000), replace=False)] *= 300
    return workloads.to_bf16(x)


def ok_status(st):
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0


@pytest.mark.parametrize("case", range(30))
def test_random_dense_gemm(case):
    g = np.random.Generator(np.random.Philox(1000 + case))
    M = int(g.integers(1, 1400))
    N = int(g.integers(1, 1400))
    K = 32 * int(g.integers(1, 100))
    a, b = src(g, (M, K)), src(g, (N, K), 0.05)
    st = mx.new_status()
    ar, _ = mx.quantize(a.cuda(), mx.MX_ROWWISE, status=st)
    br, _ = mx.quantize(b.cuda(), mx.MX_ROWWISE, status=st)
    ldc = N + int(g.integers(0, 24))
    shift = int(g.integers(0, 2))                    # 1: output rows not 16-byte aligned
    big = torch.full((M, ldc + 1), float("nan"), dtype=torch.bfloat16, device="cuda")
    view = big[:, shift:shift + N]
    use_ws = bool(g.integers(0, 2))
    ws = mx.gemm_workspace(mx.MX_FPROP, ar, br) if use_ws else None
    mx.gemm(mx.MX_FPROP, ar, br, out=view, status=st, workspace=ws)
    ok_status(st)
    h = big.float().cpu().numpy()
    assert np.all(np.isnan(h[:, :shift])) and np.all(np.isnan(h[:, shift + N:])), f"case {case}: wrote outside C"
    check_gemm_full(view, *oracle.mx_quantize_rowwise(f64(a)), *oracle.mx_quantize_rowwise(f64(b)),
                    f"random gemm {M}x{N}x{K} ws={use_ws} shift={shift}")


@pytest.mark.parametrize("case", range(10))
def test_random_wgrad_from_column_copies(case):
    """dW = dY^T X from the column copies (tokens a multiple of 32)."""
    g = np.random.Generator(np.random.Philox(2000 + case))
    T = 32 * int(g.integers(1, 80))
    N = 32 * int(g.integers(1, 40))
    K = 32 * int(g.integers(1, 40))
    dY, X = src(g, (T, N)), src(g, (T, K))
    st = mx.new_status()
    _, dc = mx.quantize(dY.cuda(), mx.MX_COLWISE, status=st)
    _, xc = mx.quantize(X.cuda(), mx.MX_COLWISE, status=st)
    dW = mx.gemm(mx.MX_WGRAD, dc, xc, status=st)
    ok_status(st)
    check_gemm_full(dW, *oracle.mx_quantize_colwise(f64(dY)), *oracle.mx_quantize_colwise(f64(X)),
                    f"random wgrad T={T} N={N} K={K}")


@pytest.mark.parametrize("case", range(16))
def test_random_quantize(case):
    g = np.random.Generator(np.random.Philox(3000 + case))
    axis = int(g.integers(1, 4))
    R = int(g.integers(1, 700))
    if axis & mx.MX_COLWISE:
        R = 32 * ((R + 31) // 32)
    C = 32 * int(g.integers(1, 60))
    x = src(g, (R, C))
    pitch = C + 8 * int(g.integers(0, 5))
    xb = torch.zeros((R, pitch), dtype=torch.bfloat16)
    xb[:, :C] = x
    st = mx.new_status()
    row, col = mx.quantize(xb.cuda()[:, :C], axis, status=st)
    ok_status(st)
    if axis & mx.MX_ROWWISE:
        check_row_copy(x, row, f"random row {R}x{C}")
    if axis & mx.MX_COLWISE:
        check_col_copy(x, col, f"random col {R}x{C}")


@pytest.mark.parametrize("case", range(8))
def test_random_quantize_multi(case):
    g = np.random.Generator(np.random.Philox(4000 + case))
    n = int(g.integers(1, mx.MX_MAX_MULTI + 1))
    xs = [src(g, (32 * int(g.integers(0, 20)), 32 * int(g.integers(1, 20)))) for _ in range(n)]
    st = mx.new_status()
    outs = mx.quantize_multi([x.cuda() for x in xs], mx.MX_BOTH, status=st)
    ok_status(st)
    for i, (x, (row, col)) in enumerate(zip(xs, outs)):
        if x.numel():
            check_row_copy(x, row, f"multi[{i}] row")
            check_col_copy(x, col, f"multi[{i}] col")


def random_counts(g, E, total_max):
    c = g.integers(0, total_max // E + 1, E)
    c[g.integers(0, E)] = 0                          # at least one empty expert
    if E > 2:
        c[g.integers(0, E)] = 1                      # and a single-row one
    if c.sum() == 0:
        c[-1] = 100                                  # the routed input is never empty
    return c


@pytest.mark.parametrize("case", range(10))
def test_random_grouped_fprop_and_wgrad(case):
    g = np.random.Generator(np.random.Philox(5000 + case))
    E = int(g.integers(1, 12))
    counts = random_counts(g, E, 2400)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M = int(offs[-1])
    K = 32 * int(g.integers(1, 12))
    N = 32 * int(g.integers(1, 14))
    X, dY = src(g, (M, K)), src(g, (M, N))
    W = workloads.to_bf16(g.standard_normal((E, N, K)) * 0.05)
    o = torch.from_numpy(offs).cuda()
    st = mx.new_status()
    xr, _ = mx.quantize(X.cuda(), mx.MX_ROWWISE, status=st)
    wr, _ = mx.quantize_stacked(W.cuda(), mx.MX_ROWWISE, status=st)
    y = mx.grouped_gemm(mx.MX_FPROP, xr, wr, o, status=st)
    cap = mx.mx_grouped_padded_rows(offs)
    _, dc = mx.quantize(dY.cuda(), mx.MX_COLWISE, group_offsets=o, col_capacity=max(cap, 128), status=st)
    _, xc = mx.quantize(X.cuda(), mx.MX_COLWISE, group_offsets=o, col_capacity=max(cap, 128), status=st)
    dw = mx.grouped_gemm(mx.MX_WGRAD, dc, xc, o, status=st)
    ok_status(st)
    fX, fdY = f64(X), f64(dY)
    wq = [oracle.mx_quantize_rowwise(f64(W[e])) for e in range(E)]
    ref, S = oracle.mx_grouped_gemm_ref_mragged(*oracle.mx_quantize_rowwise(fX), np.stack([w[0] for w in wq]),
                                                np.stack([w[1] for w in wq]), offs)
    assert oracle.within_tolerance(f64(y), ref, S).all(), f"grouped fprop counts={list(counts)} K={K} N={N}"
    a, as_, _ = oracle.mx_quantize_colwise_grouped(fdY, offs)
    b, bs, _ = oracle.mx_quantize_colwise_grouped(fX, offs)
    ref, S = oracle.mx_grouped_gemm_ref_kragged(a, as_, b, bs, offs)
    assert oracle.within_tolerance(f64(dw), ref, S).all(), f"grouped wgrad counts={list(counts)} K={K} N={N}"


@pytest.mark.parametrize("case", range(6))
def test_random_gemm_multi(case):
    g = np.random.Generator(np.random.Philox(6000 + case))
    n = int(g.integers(2, mx.MX_MAX_GEMM_MULTI + 1))
    probs, refs = [], []
    for _ in range(n):
        M, N, K = int(g.integers(1, 3000)), int(g.integers(129, 1500)), 32 * int(g.integers(1, 40))
        a, b = src(g, (M, K)), src(g, (N, K), 0.05)
        st = mx.new_status()
        ar, _ = mx.quantize(a.cuda(), mx.MX_ROWWISE, status=st)
        br, _ = mx.quantize(b.cuda(), mx.MX_ROWWISE, status=st)
        probs.append((mx.MX_FPROP, ar, br))
        refs.append((a, b))
    st = mx.new_status()
    outs = mx.gemm_multi(probs, status=st)
    ok_status(st)
    for (a, b), o in zip(refs, outs):
        check_gemm_full(o, *oracle.mx_quantize_rowwise(f64(a)), *oracle.mx_quantize_rowwise(f64(b)),
                        f"multi {tuple(o.shape)} K={a.shape[1]}")
