"""Tensors past 2^31 elements: the quantiser and the GEMM index their inputs
and outputs with 64 bits. Inputs are drawn on the device (seeded); the rows
and columns checked against the oracle include the last ones."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import check_gemm_sampled, f64, u8

pytestmark = pytest.mark.gpu


def device_normal(shape, seed, std=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * std).to(torch.bfloat16)


def test_quantize_past_2_31_elements():
    R, C = 70016, 32768                       # 2.29e9 elements
    assert R * C > 2 ** 31
    x = device_normal((R, C), 1)
    st = mx.new_status()
    row, col = mx.quantize(x, mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    rows = np.concatenate([np.arange(0, 40), np.arange(R // 2, R // 2 + 8), np.arange(R - 40, R)])
    cols = np.concatenate([np.arange(0, 8), np.arange(C - 40, C)])
    rsel = torch.from_numpy(rows).cuda()
    csel = torch.from_numpy(cols).cuda()
    # row copy: the sampled rows' codes and scales
    d, s = oracle.mx_quantize_rowwise(f64(x[rsel]))
    assert np.array_equal(u8(row.data[rsel]), d), "row codes"
    scales = oracle.mx_scale_unswizzle(u8(row.scale), R, C // 32)
    assert np.array_equal(scales[rows], s), "row scales"
    # column copy: the sampled columns (each a full 70016-element column)
    d, s = oracle.mx_quantize_colwise(f64(x[:, csel]))
    assert np.array_equal(u8(col.data[csel]), d), "column codes"
    scales = oracle.mx_scale_unswizzle(u8(col.scale), C, R // 32)
    assert np.array_equal(scales[cols], s), "column scales"


@pytest.mark.parametrize("aligned", [True, False])
def test_gemm_output_past_2_31_elements(aligned):
    M, N, K = 70000, 33000, 128               # C: 2.31e9 elements
    assert M * N > 2 ** 31
    a = device_normal((M, K), 2)
    b = device_normal((N, K), 3, 0.05)
    st = mx.new_status()
    ar, _ = mx.quantize(a, mx.MX_ROWWISE, status=st)
    br, _ = mx.quantize(b, mx.MX_ROWWISE, status=st)
    if aligned:
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    else:                                     # rows not 16-byte aligned: element stores
        out = torch.empty((M, N + 1), dtype=torch.bfloat16, device="cuda")[:, 1:]
    mx.gemm(mx.MX_FPROP, ar, br, out=out, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    g = np.random.Generator(np.random.Philox(4))
    ii = np.concatenate([g.integers(0, M, 200), [M - 1] * 20, np.arange(M - 20, M)])
    jj = np.concatenate([g.integers(0, N, 200), np.arange(N - 20, N), [N - 1] * 20])
    check_gemm_sampled(out, a, mx.MX_ROWWISE, b, mx.MX_ROWWISE, ii, jj, f"large gemm aligned={aligned}")
