"""Helpers for the GPU parity tests: move tensors between torch and the
oracle's numpy world and compare the CUDA path's outputs with the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_gb300 as mx

needs_gpu = pytest.mark.gpu

# Error reports of every GEMM parity check of the session (what, report); the
# conftest prints them at the end of the run, including the count of entries
# that would fail the bound measured against BF16(ref) (reported, not gated).
REPORTS: list = []


def _record(what: str, rep: dict) -> dict:
    REPORTS.append((what, rep))
    return rep


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> uint16 bit patterns (numpy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a BF16 tensor."""
    return oracle.bf16_bits_to_float64(bits(t))


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def first_diffs(a: np.ndarray, b: np.ndarray, n: int = 8):
    idx = np.argwhere(a != b)[:n]
    return [(tuple(i), int(a[tuple(i)]), int(b[tuple(i)])) for i in idx]


def assert_bytes_equal(gpu: np.ndarray, ref: np.ndarray, what: str):
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if not np.array_equal(gpu, ref):
        n = int(np.sum(gpu != ref))
        raise AssertionError(f"{what}: {n} of {gpu.size} bytes differ; first: {first_diffs(gpu, ref)}")


def check_row_copy(x_cpu: torch.Tensor, row: "mx.MXTensor", what: str = "row"):
    """GPU row copy == oracle 1x32 quantisation, bit for bit (data, scales, padding)."""
    d, s = oracle.mx_quantize_rowwise(f64(x_cpu))
    assert_bytes_equal(u8(row.data), d, what + " data")
    assert_bytes_equal(u8(row.scale), oracle.mx_scale_swizzle(s), what + " scales")


def check_col_copy(x_cpu: torch.Tensor, col: "mx.MXTensor", what: str = "col"):
    d, s = oracle.mx_quantize_colwise(f64(x_cpu))
    assert_bytes_equal(u8(col.data), d, what + " data")
    assert_bytes_equal(u8(col.scale), oracle.mx_scale_swizzle(s), what + " scales")


def check_gemm_full(out_gpu: torch.Tensor, a_codes, a_scale, b_codes, b_scale, what: str = "gemm"):
    """Every output element within |out - ref| <= 2**-8 |ref| + 1e-6 S."""
    ref, S = oracle.mx_gemm_ref(a_codes, a_scale, b_codes, b_scale)
    out = f64(out_gpu)
    assert out.shape == ref.shape
    ok = oracle.within_tolerance(out, ref, S)
    if not ok.all():
        bad = np.argwhere(~ok)[:8]
        rep = oracle.error_report(out, ref, S)
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; first "
                             f"{[(tuple(i), out[tuple(i)], ref[tuple(i)]) for i in bad]}; {rep}")
    return _record(what, oracle.error_report(out, ref, S))


def logical_scales(t: "mx.MXTensor") -> np.ndarray:
    return oracle.mx_scale_unswizzle(u8(t.scale), t.rows, (t.k + 31) // 32)


def sample_entries(M: int, N: int, n: int, seed: int, tile_m: int = 128, tile_n: int = 128):
    """n seeded random (i, j) plus rows/cols on both sides of every tile boundary
    and the last row/column."""
    g = np.random.Generator(np.random.Philox(seed))
    ii = list(g.integers(0, M, n))
    jj = list(g.integers(0, N, n))
    bm = sorted({min(M - 1, b) for t in range(0, M, tile_m) for b in (t, t + tile_m - 1)} | {M - 1})
    bn = sorted({min(N - 1, b) for t in range(0, N, tile_n) for b in (t, t + tile_n - 1)} | {N - 1})
    for i in bm:
        ii.append(i)
        jj.append(int(g.integers(0, N)))
    for j in bn:
        ii.append(int(g.integers(0, M)))
        jj.append(j)
    return np.array(ii, dtype=np.int64), np.array(jj, dtype=np.int64)


def check_gemm_sampled(out_gpu: torch.Tensor, a_src, a_orient: int, b_src, b_orient: int, ii, jj,
                       what: str = "gemm"):
    """Check sampled entries of C = A . B^T where A and B are the MX copies of
    the BF16 sources a_src / b_src (row copy: blocks along rows of the source;
    column copy: the source's columns). The oracle quantises only the rows /
    columns it needs, straight from the BF16 inputs."""
    ua, inv_a = np.unique(ii, return_inverse=True)
    ub, inv_b = np.unique(jj, return_inverse=True)
    if a_orient == mx.MX_ROWWISE:
        ac, asc = oracle.mx_quantize_rowwise(f64(a_src[torch.from_numpy(ua)]))
    else:
        ac, asc = oracle.mx_quantize_colwise(f64(a_src[:, torch.from_numpy(ua)]))
    if b_orient == mx.MX_ROWWISE:
        bc, bsc = oracle.mx_quantize_rowwise(f64(b_src[torch.from_numpy(ub)]))
    else:
        bc, bsc = oracle.mx_quantize_colwise(f64(b_src[:, torch.from_numpy(ub)]))
    ref, S = oracle.mx_gemm_ref_entries(ac, asc, bc, bsc, inv_a, inv_b)
    out = f64(out_gpu[torch.from_numpy(ii), torch.from_numpy(jj)])
    ok = oracle.within_tolerance(out, ref, S)
    if not ok.all():
        bad = np.flatnonzero(~ok)[:8]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} sampled entries outside tolerance; "
                             f"first {[(int(ii[b]), int(jj[b]), out[b], ref[b]) for b in bad]}")
    return _record(what, oracle.error_report(out, ref, S))


def check_values(out, ref, S, what: str) -> dict:
    """Element-wise acceptance of already computed oracle values; records the report."""
    out = np.asarray(out, dtype=np.float64)
    ok = oracle.within_tolerance(out, ref, S)
    if not ok.all():
        bad = np.flatnonzero(~ok.reshape(-1))[:8]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; first "
                             f"{[(int(b), out.reshape(-1)[b], ref.reshape(-1)[b]) for b in bad]}")
    return _record(what, oracle.error_report(out, ref, S))


# ---------------------------------------------------------------------------
# Full-tensor quantisation parity at workload sizes (oracle run over the host
# cores by tests.oracle_pool; every data byte and every scale byte, padding
# included)
# ---------------------------------------------------------------------------

def check_row_copy_full(x_cpu: torch.Tensor, row: "mx.MXTensor", what: str = "row"):
    from tests import oracle_pool
    d, s = oracle_pool.rowwise(bits(x_cpu))
    assert_bytes_equal(u8(row.data), d, what + " data")
    assert_bytes_equal(u8(row.scale), oracle.mx_scale_swizzle(s), what + " scales")


def check_col_copy_full(x_cpu: torch.Tensor, col: "mx.MXTensor", what: str = "col"):
    from tests import oracle_pool
    d, s = oracle_pool.colwise(bits(x_cpu))
    assert_bytes_equal(u8(col.data), d, what + " data")
    assert_bytes_equal(u8(col.scale), oracle.mx_scale_swizzle(s), what + " scales")


def check_grouped_col_copy_full(x_cpu: torch.Tensor, offsets, col: "mx.MXTensor", what: str = "grouped col"):
    """The per-group padded column copy [D, capacity] (capacity = padded total)."""
    from tests import oracle_pool
    d, s = oracle_pool.colwise_grouped(bits(x_cpu), offsets)
    assert col.k == d.shape[1], (what, col.k, d.shape)
    assert_bytes_equal(u8(col.data), d, what + " data")
    assert_bytes_equal(u8(col.scale), oracle.mx_scale_swizzle(s), what + " scales")


def check_stacked_full(w_cpu: torch.Tensor, row: "mx.MXStacked", col: "mx.MXStacked", what: str = "stacked"):
    """Row and column copies of every matrix of stacked weights [E, N, K]."""
    from tests import oracle_pool
    rd, rs, cd, cs = oracle_pool.stacked(bits(w_cpu))
    assert_bytes_equal(u8(row.data), rd, what + " row data")
    assert_bytes_equal(u8(col.data), cd, what + " col data")
    gr, gc = u8(row.scale), u8(col.scale)
    for e in range(rd.shape[0]):
        assert_bytes_equal(gr[e], oracle.mx_scale_swizzle(rs[e]), f"{what} row scales, expert {e}")
        assert_bytes_equal(gc[e], oracle.mx_scale_swizzle(cs[e]), f"{what} col scales, expert {e}")
