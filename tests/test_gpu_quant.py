"""GPU quantiser vs the oracle, bit for bit: data codes, scale codes and the
padding bytes of the swizzled scale tiles."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import assert_bytes_equal, check_col_copy, check_row_copy, f64, logical_scales, u8

pytestmark = pytest.mark.gpu


def run(x_cpu, axis, **kw):
    x = x_cpu.cuda()
    st = mx.new_status()
    row, col = mx.quantize(x, axis, status=st, **kw)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return row, col


def test_hand_blocks():
    """The 64 hand-built blocks (zeros, BF16 subnormals, E4M3-subnormal members,
    exact +-448, saturating members, 1e4 outliers, ties, extremes), quantised as
    1x32 row blocks and, transposed, as 32x1 column blocks."""
    hb = workloads.hand_blocks()
    row, _ = run(hb, mx.MX_ROWWISE)
    check_row_copy(hb, row, "hand blocks row")
    hbt = hb.t().contiguous()                 # [32, 64]: each column is one block
    _, col = run(hbt, mx.MX_COLWISE)
    check_col_copy(hbt, col, "hand blocks col")
    # the column copy of the transpose is the row copy of the blocks
    assert np.array_equal(u8(col.data), u8(row.data))


def exhaustive_blocks():
    """Every finite BF16 pattern under every shared exponent X in [-127, 119]
    for which it can appear below the block maximum and round to non-zero:
    block = [amax forcing X, 31 test values]."""
    pats = np.arange(1 << 16, dtype=np.uint32)
    vals = oracle.bf16_bits_to_float64(pats.astype(np.uint16))
    fin = np.isfinite(vals)
    pats, vals = pats[fin], vals[fin]
    rows = []
    for X in range(-127, 120):
        amax = (2 - 2.0 ** -7) * 2.0 ** (X + 8)
        sel = (np.abs(vals) <= amax) & (np.abs(vals) >= 2.0 ** (X - 12))
        if X == -127:
            sel |= np.abs(vals) < 2.0 ** (X - 12)   # tiny and zero members once
        v = vals[sel]
        n = (len(v) + 30) // 31
        blk = np.zeros((n, 32))
        blk[:, 0] = amax if X % 2 == 0 else -amax
        flat = np.zeros(n * 31)
        flat[: len(v)] = v
        blk[:, 1:] = flat.reshape(n, 31)
        rows.append(blk)
    b = np.concatenate(rows)
    pad = (-len(b)) % 32
    b = np.concatenate([b, np.zeros((pad, 32))])
    return workloads.to_bf16(b)


def test_exhaustive_element_codec():
    blocks = exhaustive_blocks()                     # [nblk, 32], nblk % 32 == 0
    row, _ = run(blocks, mx.MX_ROWWISE)
    check_row_copy(blocks, row, "exhaustive row")
    bt = blocks.t().contiguous()                     # [32, nblk]
    _, col = run(bt, mx.MX_COLWISE)
    check_col_copy(bt, col, "exhaustive col")


@pytest.mark.parametrize("R,C", [(32, 32), (96, 160), (128, 128), (160, 576), (256, 512), (416, 96),
                                 (1024, 2048)])
def test_dense_both(R, C):
    g = np.random.Generator(np.random.Philox(R * 1000 + C))
    x = g.standard_normal((R, C)) * np.exp2(g.integers(-6, 6, (R, 1))) * np.exp2(g.integers(-3, 3, (1, C)))
    x.reshape(-1)[g.choice(R * C, size=max(1, R * C // 500), replace=False)] *= 1000
    xb = workloads.to_bf16(x)
    row, col = run(xb, mx.MX_BOTH)
    check_row_copy(xb, row)
    check_col_copy(xb, col)
    # the single-axis kernels agree with the fused one
    r2, _ = run(xb, mx.MX_ROWWISE)
    _, c2 = run(xb, mx.MX_COLWISE)
    assert np.array_equal(u8(r2.data), u8(row.data)) and np.array_equal(u8(r2.scale), u8(row.scale))
    assert np.array_equal(u8(c2.data), u8(col.data)) and np.array_equal(u8(c2.scale), u8(col.scale))


@pytest.mark.parametrize("R", [1, 7, 77, 129, 300])
def test_rowwise_ragged_rows(R):
    xb = workloads.normal_bf16((R, 96), 700 + R)
    row, _ = run(xb, mx.MX_ROWWISE)
    check_row_copy(xb, row)


def test_input_pitch():
    wide = workloads.normal_bf16((128, 512), 801)
    xv = wide.cuda()[:, 64:320]                     # pitch 512, 256 columns
    st = mx.new_status()
    row, col = mx.quantize(xv, mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    ref = wide[:, 64:320].contiguous()
    check_row_copy(ref, row)
    check_col_copy(ref, col)


def test_single_linear_inputs():
    d = workloads.single_linear()
    for name in ("X", "W"):
        row, col = run(d[name], mx.MX_BOTH)
        check_row_copy(d[name], row, name)
        check_col_copy(d[name], col, name)


def test_nan_inf_blocks():
    x = np.ones((64, 64))
    x[0, 3] = np.nan
    x[5, 40] = -np.inf
    x[40, 7] = np.inf
    x[33, 1] = -3.0
    xb = workloads.to_bf16(x)
    row, col = run(xb, mx.MX_BOTH)
    check_row_copy(xb, row)
    check_col_copy(xb, col)
    assert logical_scales(row)[0, 0] == 0xFF and logical_scales(row)[5, 1] == 0xFF


def grouped_case(counts, D, seed, cap_extra=256, axis=mx.MX_COLWISE):
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M = int(offs[-1])
    xb = workloads.normal_bf16((M, D), seed)
    total = mx.mx_grouped_padded_rows(offs)
    cap = total + cap_extra
    x = xb.cuda()
    o = torch.from_numpy(offs).cuda()
    st = mx.new_status()
    row, col = mx.quantize(x, axis, group_offsets=o, col_capacity=cap, status=st)
    torch.cuda.synchronize()
    return xb, offs, total, cap, row, col, st


@pytest.mark.parametrize("counts", [[20, 0, 150, 1, 128], [0, 0, 5], [300], [128, 129, 127, 0, 1, 255, 256, 2]])
def test_grouped_colwise(counts):
    D = 192
    xb, offs, total, cap, row, col, st = grouped_case(counts, D, 900 + len(counts), axis=mx.MX_BOTH)
    assert mx.read_status(st) == 0
    d, s, poff = oracle.mx_quantize_colwise_grouped(f64(xb), offs)
    assert poff[-1] == total
    assert_bytes_equal(u8(col.data)[:, :total], d, "grouped col data")
    assert_bytes_equal(logical_scales(col)[:, : total // 32], s, "grouped col scales")
    check_row_copy(xb, row, "grouped row")


def test_grouped_bad_offsets_write_nothing():
    D = 64
    for offs, cap in [([0, 50, 40, 100], 512), ([0, 50, 90], 512), ([0, 50, 100], 128), ([3, 50, 100], 512)]:
        offs = np.array(offs, dtype=np.int64)
        M = 100
        x = workloads.normal_bf16((M, D), 1000).cuda()
        o = torch.from_numpy(offs).cuda()
        col_data = torch.full((D, cap), 0xAB, dtype=torch.uint8, device="cuda")
        col_scale = torch.full((mx.mx_scale_bytes(D, cap),), 0xAB, dtype=torch.uint8, device="cuda")
        st = mx.new_status()
        mx.mx_quantize(x.data_ptr(), M, D, D, mx.MX_COLWISE, None, None, col_data.data_ptr(), col_scale.data_ptr(),
                       o.data_ptr(), len(offs) - 1, cap, st.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert mx.read_status(st) == 5, offs
        assert bool((col_data == 0xAB).all()) and bool((col_scale == 0xAB).all())


def test_repeatable():
    xb = workloads.normal_bf16((512, 1024), 1100)
    r1, c1 = run(xb, mx.MX_BOTH)
    r2, c2 = run(xb, mx.MX_BOTH)
    for a, b in [(r1.data, r2.data), (r1.scale, r2.scale), (c1.data, c2.data), (c1.scale, c2.scale)]:
        assert torch.equal(a, b)


def test_batched_matches_per_matrix_oracle():
    """Stacked matrices [E, N, K] in one launch: each matrix's row and column
    copies equal the oracle's quantisation of that matrix alone."""
    E, N, K = 5, 160, 96
    w = workloads.normal_bf16((E, N, K), 1200)
    st = mx.new_status()
    row, col = mx.quantize_stacked(w.cuda(), mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    for e in range(E):
        d, s = oracle.mx_quantize_rowwise(f64(w[e]))
        assert_bytes_equal(u8(row.data[e]), d, f"batched row data {e}")
        assert_bytes_equal(u8(row.scale[e]), oracle.mx_scale_swizzle(s), f"batched row scales {e}")
        d, s = oracle.mx_quantize_colwise(f64(w[e]))
        assert_bytes_equal(u8(col.data[e]), d, f"batched col data {e}")
        assert_bytes_equal(u8(col.scale[e]), oracle.mx_scale_swizzle(s), f"batched col scales {e}")
