"""Parity at the full workload sizes, in the launch configuration bench.py
times: quantisation bit-exact (full tensors where the oracle is quick, else
sampled rows and columns including every tile boundary) and GEMM outputs on
sampled entries (seeded random entries plus both sides of every tile
boundary), each computed by the oracle straight from the BF16 inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import (assert_bytes_equal, check_col_copy, check_gemm_sampled, check_row_copy, f64,
                            sample_entries, u8)

pytestmark = pytest.mark.gpu


def quant_both(xb_cpu):
    st = mx.new_status()
    x = xb_cpu.cuda()
    row, col = mx.quantize(x, mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return row, col


def boundary_rows(n, seed, k=256, tile=128):
    g = np.random.Generator(np.random.Philox(seed))
    b = {min(n - 1, t + d) for t in range(0, n, tile) for d in (0, tile - 1)} | {n - 1}
    return np.unique(np.concatenate([g.integers(0, n, k), np.array(sorted(b))]))


def check_rows_sampled(x_cpu, row, rows, what):
    """Selected rows of a row copy (data and logical scales) against the oracle."""
    d, s = oracle.mx_quantize_rowwise(f64(x_cpu[torch.from_numpy(rows)]))
    assert_bytes_equal(u8(row.data)[rows], d, what + " data")
    gs = oracle.mx_scale_unswizzle(u8(row.scale), row.rows, row.k // 32)[rows]
    assert_bytes_equal(gs, s, what + " scales")


def check_cols_sampled(x_cpu, col, cols, what):
    """Selected columns of the source through its column copy."""
    d, s = oracle.mx_quantize_colwise(f64(x_cpu[:, torch.from_numpy(cols)]))
    assert_bytes_equal(u8(col.data)[cols], d, what + " data")
    gs = oracle.mx_scale_unswizzle(u8(col.scale), col.rows, col.k // 32)[cols]
    assert_bytes_equal(gs, s, what + " scales")


# ---------------------------------------------------------------------------
# Dense FFN up-projection: M=8192, K=2048, N=10944
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def ffn():
    d = workloads.dense_ffn()
    q = {k: quant_both(d[k]) for k in ("X", "W", "dY")}
    return d, q


def test_ffn_quantisation(ffn):
    d, q = ffn
    for k in ("X", "W"):
        check_row_copy(d[k], q[k][0], k + " row")
        check_col_copy(d[k], q[k][1], k + " col")
    dy = d["dY"]
    check_rows_sampled(dy, q["dY"][0], boundary_rows(dy.shape[0], 1), "dY row")
    check_cols_sampled(dy, q["dY"][1], boundary_rows(dy.shape[1], 2), "dY col")


@pytest.mark.parametrize("mode", [mx.MX_FPROP, mx.MX_DGRAD, mx.MX_WGRAD])
def test_ffn_gemm(ffn, mode):
    d, q = ffn
    (xr, xc), (wr, wc), (dr, dc) = q["X"], q["W"], q["dY"]
    st = mx.new_status()
    if mode == mx.MX_FPROP:
        out = mx.gemm(mode, xr, wr, status=st)
        srcs = (d["X"], mx.MX_ROWWISE, d["W"], mx.MX_ROWWISE)
    elif mode == mx.MX_DGRAD:
        out = mx.gemm(mode, dr, wc, status=st)
        srcs = (d["dY"], mx.MX_ROWWISE, d["W"], mx.MX_COLWISE)
    else:
        out = mx.gemm(mode, dc, xc, status=st)
        srcs = (d["dY"], mx.MX_COLWISE, d["X"], mx.MX_COLWISE)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    assert bool(torch.isfinite(out.float()).all())
    ii, jj = sample_entries(out.shape[0], out.shape[1], 4096, 10 + mode, tile_n=256)
    rep = check_gemm_sampled(out, *srcs, ii, jj, what=f"ffn mode {mode}")
    assert rep["fail"] == 0


# ---------------------------------------------------------------------------
# MLA projections at M = 16384
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", [p[0] for p in workloads.MLA_PROJECTIONS])
def test_mla_projection(name):
    d = workloads.mla_projection(name)
    (xr, xc), (wr, wc), (dr, dc) = quant_both(d["X"]), quant_both(d["W"]), quant_both(d["dY"])
    check_row_copy(d["W"], wr, name + " W row")
    check_col_copy(d["W"], wc, name + " W col")
    check_rows_sampled(d["X"], xr, boundary_rows(d["X"].shape[0], 3, 128), name + " X row")
    check_cols_sampled(d["X"], xc, boundary_rows(d["X"].shape[1], 4, 128), name + " X col")
    st = mx.new_status()
    y = mx.gemm(mx.MX_FPROP, xr, wr, status=st)
    dx = mx.gemm(mx.MX_DGRAD, dr, wc, status=st)
    dw = mx.gemm(mx.MX_WGRAD, dc, xc, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    for out, srcs, tag in ((y, (d["X"], 1, d["W"], 1), "fprop"), (dx, (d["dY"], 1, d["W"], 2), "dgrad"),
                           (dw, (d["dY"], 2, d["X"], 2), "wgrad")):
        ii, jj = sample_entries(out.shape[0], out.shape[1], 1024, 20, tile_n=256)
        check_gemm_sampled(out, *srcs, ii, jj, what=f"{name} {tag}")


# ---------------------------------------------------------------------------
# Routed experts: 64 experts, 49152 rows, gate_up (N=2816, K=2048), down (N=2048, K=1408)
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def moe():
    return workloads.moe_experts()


def grouped_entry_refs(a_src, a_orient, b_stack, b_orient, offs, ii, jj):
    """Oracle values of sampled entries (i, j) of the rows-ragged grouped GEMM."""
    e_of = np.searchsorted(offs, ii, side="right") - 1
    ref = np.zeros(len(ii))
    S = np.zeros(len(ii))
    for e in np.unique(e_of):
        sel = np.flatnonzero(e_of == e)
        ac, asc = oracle.mx_quantize_rowwise(f64(a_src[torch.from_numpy(ii[sel])]))
        w = b_stack[int(e)]
        if b_orient == mx.MX_ROWWISE:
            bc, bsc = oracle.mx_quantize_rowwise(f64(w[torch.from_numpy(jj[sel])]))
        else:
            bc, bsc = oracle.mx_quantize_colwise(f64(w[:, torch.from_numpy(jj[sel])]))
        r, s = oracle.mx_gemm_ref_entries(ac, asc, bc, bsc, np.arange(len(sel)), np.arange(len(sel)))
        ref[sel] = r
        S[sel] = s
    return ref, S


def moe_samples(offs, N, seed, per_expert=24):
    g = np.random.Generator(np.random.Philox(seed))
    ii, jj = [], []
    for e in range(len(offs) - 1):
        m = offs[e + 1] - offs[e]
        if m == 0:
            continue
        rows = list(g.integers(offs[e], offs[e + 1], per_expert)) + [offs[e], offs[e + 1] - 1]
        ii += rows
        jj += list(g.integers(0, N, len(rows)))
    return np.array(ii, dtype=np.int64), np.array(jj, dtype=np.int64)


@pytest.mark.parametrize("proj", ["gate_up", "down"])
def test_moe_grouped(moe, proj):
    offs = moe["offsets"]
    o = torch.from_numpy(offs).cuda()
    A = moe["X"] if proj == "gate_up" else moe["A_down"]          # [M, K]
    W = moe["W_gate_up"] if proj == "gate_up" else moe["W_down"]  # [E, N, K]
    dY = moe["dY_gate_up"] if proj == "gate_up" else moe["dY_down"]  # [M, N]
    E, N, K = W.shape
    st = mx.new_status()
    ar, _ = mx.quantize(A.cuda(), mx.MX_ROWWISE, status=st)
    wr, wc = mx.quantize_stacked(W.cuda(), mx.MX_BOTH, status=st)
    dr, _ = mx.quantize(dY.cuda(), mx.MX_ROWWISE, status=st)
    cap = mx.mx_grouped_padded_rows(offs)
    _, dcg = mx.quantize(dY.cuda(), mx.MX_COLWISE, group_offsets=o, col_capacity=cap, status=st)
    _, acg = mx.quantize(A.cuda(), mx.MX_COLWISE, group_offsets=o, col_capacity=cap, status=st)
    y = mx.grouped_gemm(mx.MX_FPROP, ar, wr, o, status=st)
    dx = mx.grouped_gemm(mx.MX_DGRAD, dr, wc, o, status=st)
    dw = mx.grouped_gemm(mx.MX_WGRAD, dcg, acg, o, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0

    # fprop: Y[t, n] = sum_k A[t, k] W_e[n, k]
    ii, jj = moe_samples(offs, N, 31)
    ref, S = grouped_entry_refs(A, mx.MX_ROWWISE, W, mx.MX_ROWWISE, offs, ii, jj)
    out = f64(y[torch.from_numpy(ii), torch.from_numpy(jj)])
    assert oracle.within_tolerance(out, ref, S).all(), f"{proj} fprop"
    # dgrad: dX[t, k] = sum_n dY[t, n] W_e[n, k]
    ii, jj = moe_samples(offs, K, 32)
    ref, S = grouped_entry_refs(dY, mx.MX_ROWWISE, W, mx.MX_COLWISE, offs, ii, jj)
    out = f64(dx[torch.from_numpy(ii), torch.from_numpy(jj)])
    assert oracle.within_tolerance(out, ref, S).all(), f"{proj} dgrad"
    # wgrad: dW_e[n, k] = sum_{t in e} dY[t, n] A[t, k]; sampled (e, n, k)
    g = np.random.Generator(np.random.Philox(33))
    for e in range(E):
        m = int(offs[e + 1] - offs[e])
        if m == 0:
            assert bool((dw[e] == 0).all()), f"empty expert {e} not zero"
            continue
        n_idx = np.unique(np.concatenate([g.integers(0, N, 6), [0, N - 1]]))
        k_idx = np.unique(np.concatenate([g.integers(0, K, 6), [0, K - 1]]))
        seg_off = np.array([0, m])
        a, as_, _ = oracle.mx_quantize_colwise_grouped(f64(dY[offs[e]:offs[e + 1]][:, torch.from_numpy(n_idx)]),
                                                       seg_off)
        b, bs, _ = oracle.mx_quantize_colwise_grouped(f64(A[offs[e]:offs[e + 1]][:, torch.from_numpy(k_idx)]),
                                                      seg_off)
        ref, S = oracle.mx_gemm_ref(a, as_, b, bs)
        out = f64(dw[e][torch.from_numpy(n_idx)][:, torch.from_numpy(k_idx)])
        assert oracle.within_tolerance(out, ref, S).all(), f"{proj} wgrad expert {e}"


# ---------------------------------------------------------------------------
# Quantiser bandwidth sweep shapes: [M x 7168], M in {4096, 8192, 16384, 32768}
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M", list(workloads.QUANT_SWEEP_M))
def test_quant_sweep(M):
    x = workloads.quant_sweep(M)
    row, col = quant_both(x)
    if M == 4096:
        check_row_copy(x, row, f"sweep {M} row")
        check_col_copy(x, col, f"sweep {M} col")
    else:
        check_rows_sampled(x, row, boundary_rows(M, 40 + M % 97), f"sweep {M} row")
        check_cols_sampled(x, col, boundary_rows(7168, 41 + M % 89), f"sweep {M} col")
