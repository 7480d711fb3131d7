"""Parity at the full workload sizes, in the launch configuration bench.py
times.

Quantisation is checked bit for bit on every element and every scale byte
(padding included) of every tensor each workload quantises: the oracle runs
over the host cores in row or column slabs (tests.oracle_pool), straight from
the BF16 inputs. GEMM outputs are checked on sampled entries (seeded random
entries plus both sides of every tile boundary), each computed by the oracle
from the BF16 inputs, within |out - ref| <= 2^-8 |ref| + 1e-6 S."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import (check_col_copy_full, check_gemm_sampled, check_grouped_col_copy_full,
                            check_row_copy_full, check_stacked_full, check_values, f64, sample_entries)

pytestmark = pytest.mark.gpu


def quant_multi(xs_cpu):
    """Both copies of each tensor, the tensors in one launch (as the bench step does)."""
    st = mx.new_status()
    outs = mx.quantize_multi([x.cuda() for x in xs_cpu], mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return outs


def check_both_full(x_cpu, q, what):
    check_row_copy_full(x_cpu, q[0], what + " row")
    check_col_copy_full(x_cpu, q[1], what + " col")


def backward_in_one_launch(dr, wc, dc, xc):
    """dgrad and wgrad of one layer in one mx_gemm_multi launch (the bench's backward)."""
    st = mx.new_status()
    dx, dw = mx.gemm_multi([(mx.MX_DGRAD, dr, wc), (mx.MX_WGRAD, dc, xc)], status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return dx, dw


# ---------------------------------------------------------------------------
# Dense FFN up-projection: M=8192, K=2048, N=10944
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def ffn():
    d = workloads.dense_ffn()
    qx, qw = quant_multi([d["X"], d["W"]])
    (qdy,) = quant_multi([d["dY"]])
    return d, {"X": qx, "W": qw, "dY": qdy}


def test_ffn_quantisation(ffn):
    d, q = ffn
    for k in ("X", "W", "dY"):
        check_both_full(d[k], q[k], k)


@pytest.mark.parametrize("mode", [mx.MX_FPROP, mx.MX_DGRAD, mx.MX_WGRAD])
def test_ffn_gemm(ffn, mode):
    d, q = ffn
    (xr, xc), (wr, wc), (dr, dc) = q["X"], q["W"], q["dY"]
    st = mx.new_status()
    if mode == mx.MX_FPROP:
        out = mx.gemm(mode, xr, wr, status=st)
        srcs = (d["X"], mx.MX_ROWWISE, d["W"], mx.MX_ROWWISE)
    elif mode == mx.MX_DGRAD:
        out = backward_in_one_launch(dr, wc, dc, xc)[0]
        srcs = (d["dY"], mx.MX_ROWWISE, d["W"], mx.MX_COLWISE)
    else:
        out = backward_in_one_launch(dr, wc, dc, xc)[1]
        srcs = (d["dY"], mx.MX_COLWISE, d["X"], mx.MX_COLWISE)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    assert bool(torch.isfinite(out.float()).all())
    ii, jj = sample_entries(out.shape[0], out.shape[1], 4096, 10 + mode, tile_n=256)
    rep = check_gemm_sampled(out, *srcs, ii, jj, what=f"dense FFN mode {mode}")
    assert rep["fail"] == 0


# ---------------------------------------------------------------------------
# MLA projections at M = 16384
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,pages", [(p[0], False) for p in workloads.MLA_PROJECTIONS] +
                         [(p[0], True) for p in workloads.MLA_PROJECTIONS_PAGES])
def test_mla_projection(name, pages):
    d = workloads.mla_projection(name, pages=pages)
    (xr, xc), (wr, wc) = quant_multi([d["X"], d["W"]])
    ((dr, dc),) = quant_multi([d["dY"]])
    for k, q in (("X", (xr, xc)), ("W", (wr, wc)), ("dY", (dr, dc))):
        check_both_full(d[k], q, f"{name} {k}")
    # fprop with the caller workspace (it may split its last round), then
    # dgrad + wgrad in one launch, as the bench step runs them
    st = mx.new_status()
    y = mx.gemm(mx.MX_FPROP, xr, wr, status=st, workspace=mx.gemm_workspace(mx.MX_FPROP, xr, wr))
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    dx, dw = backward_in_one_launch(dr, wc, dc, xc)
    for out, srcs, tag in ((y, (d["X"], 1, d["W"], 1), "fprop"), (dx, (d["dY"], 1, d["W"], 2), "dgrad"),
                           (dw, (d["dY"], 2, d["X"], 2), "wgrad")):
        ii, jj = sample_entries(out.shape[0], out.shape[1], 1024, 20, tile_n=256)
        check_gemm_sampled(out, *srcs, ii, jj, what=f"MLA {'pages ' if pages else ''}{name} {tag}")


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
    cap = mx.mx_grouped_padded_rows(offs)
    # as the bench step: row copy + per-group padded column copy in one pass
    # for the activation and the output gradient, stacked weights both ways
    ar, acg = mx.quantize(A.cuda(), mx.MX_BOTH, group_offsets=o, col_capacity=cap, status=st)
    dr, dcg = mx.quantize(dY.cuda(), mx.MX_BOTH, group_offsets=o, col_capacity=cap, status=st)
    wr, wc = mx.quantize_stacked(W.cuda(), mx.MX_BOTH, status=st)
    y = mx.grouped_gemm(mx.MX_FPROP, ar, wr, o, status=st)
    dx = mx.grouped_gemm(mx.MX_DGRAD, dr, wc, o, status=st)
    dw = mx.grouped_gemm(mx.MX_WGRAD, dcg, acg, o, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0

    # every byte of every copy
    check_row_copy_full(A, ar, f"{proj} A row")
    check_grouped_col_copy_full(A, offs, acg, f"{proj} A grouped col")
    check_row_copy_full(dY, dr, f"{proj} dY row")
    check_grouped_col_copy_full(dY, offs, dcg, f"{proj} dY grouped col")
    check_stacked_full(W, wr, wc, f"{proj} W")

    # fprop: Y[t, n] = sum_k A[t, k] W_e[n, k]
    ii, jj = moe_samples(offs, N, 31)
    ref, S = grouped_entry_refs(A, mx.MX_ROWWISE, W, mx.MX_ROWWISE, offs, ii, jj)
    check_values(f64(y[torch.from_numpy(ii), torch.from_numpy(jj)]), ref, S, f"MoE {proj} fprop")
    # dgrad: dX[t, k] = sum_n dY[t, n] W_e[n, k]
    ii, jj = moe_samples(offs, K, 32)
    ref, S = grouped_entry_refs(dY, mx.MX_ROWWISE, W, mx.MX_COLWISE, offs, ii, jj)
    check_values(f64(dx[torch.from_numpy(ii), torch.from_numpy(jj)]), ref, S, f"MoE {proj} dgrad")
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
        check_values(f64(dw[e][torch.from_numpy(n_idx)][:, torch.from_numpy(k_idx)]), ref, S,
                     f"MoE {proj} wgrad expert {e}")


# ---------------------------------------------------------------------------
# Quantiser bandwidth sweep shapes: [M x 7168], M in {4096, 8192, 16384, 32768}
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M", list(workloads.QUANT_SWEEP_M))
def test_quant_sweep(M):
    x = workloads.quant_sweep(M)
    st = mx.new_status()
    row, col = mx.quantize(x.cuda(), mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    check_both_full(x, (row, col), f"sweep M={M}")
