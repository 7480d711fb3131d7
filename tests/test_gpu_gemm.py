"""GPU block-scaled GEMM vs the oracle: every output element within
|out - ref| <= 2**-8 |ref| + 1e-6 * sum|a*b| of the FP64 dot of the
dequantised operands. The oracle quantises the BF16 sources itself."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import check_gemm_full, f64, u8

pytestmark = pytest.mark.gpu


def src(shape, seed, spread=0, std=1.0):
    """BF16 source; `spread` > 0 gives every 32-block its own power-of-two scale."""
    g = np.random.Generator(np.random.Philox(seed))
    x = g.standard_normal(shape) * std
    if spread:
        R, C = shape
        x *= np.exp2(g.integers(-spread, spread + 1, (R, (C + 31) // 32))).repeat(32, axis=1)[:, :C]
        x *= np.exp2(g.integers(-spread, spread + 1, ((R + 31) // 32, C))).repeat(32, axis=0)[:R, :]
    return workloads.to_bf16(x)


def gpu_quant(xb, axis):
    st = mx.new_status()
    row, col = mx.quantize(xb.cuda(), axis, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return row, col


def run_gemm(mode, a, b, out=None):
    st = mx.new_status()
    c = mx.gemm(mode, a, b, out=out, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return c


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (1, 1, 32), (7, 13, 64), (129, 200, 96), (256, 256, 512),
                                   (300, 520, 160), (128, 384, 1024), (64, 96, 32), (1000, 136, 224)])
def test_fprop_shapes(M, N, K):
    x = src((M, K), M * 7 + K, spread=3)
    w = src((N, K), N * 11 + K, spread=3, std=0.02)
    xr, _ = gpu_quant(x, mx.MX_ROWWISE)
    wr, _ = gpu_quant(w, mx.MX_ROWWISE)
    y = run_gemm(mx.MX_FPROP, xr, wr)
    check_gemm_full(y, *oracle.mx_quantize_rowwise(f64(x)), *oracle.mx_quantize_rowwise(f64(w)), f"fprop {M}x{N}x{K}")


def test_block_scales_far_apart():
    """Each 32-block of both operands carries its own scale (2**-30 .. 2**30): a
    wrong scale byte, row or K step shows up as a huge error."""
    M, N, K = 256, 384, 512
    x = src((M, K), 1, spread=15)
    w = src((N, K), 2, spread=15)
    xr, _ = gpu_quant(x, mx.MX_ROWWISE)
    wr, _ = gpu_quant(w, mx.MX_ROWWISE)
    y = run_gemm(mx.MX_FPROP, xr, wr)
    check_gemm_full(y, *oracle.mx_quantize_rowwise(f64(x)), *oracle.mx_quantize_rowwise(f64(w)), "spread 15")


def test_modes_direction_table():
    """fprop Y = X W^T, dgrad dX = dY W, wgrad dW = dY^T X through the row and
    column copies (one fused quantisation per tensor)."""
    Mt, Kin, Nout = 256, 192, 320
    X = src((Mt, Kin), 3, spread=2)
    W = src((Nout, Kin), 4, spread=2, std=0.02)
    dY = src((Mt, Nout), 5, spread=2)
    xr, xc = gpu_quant(X, mx.MX_BOTH)
    wr, wc = gpu_quant(W, mx.MX_BOTH)
    dr, dc = gpu_quant(dY, mx.MX_BOTH)
    y = run_gemm(mx.MX_FPROP, xr, wr)
    dx = run_gemm(mx.MX_DGRAD, dr, wc)
    dw = run_gemm(mx.MX_WGRAD, dc, xc)
    assert y.shape == (Mt, Nout) and dx.shape == (Mt, Kin) and dw.shape == (Nout, Kin)
    fX, fW, fdY = f64(X), f64(W), f64(dY)
    check_gemm_full(y, *oracle.mx_quantize_rowwise(fX), *oracle.mx_quantize_rowwise(fW), "fprop")
    check_gemm_full(dx, *oracle.mx_quantize_rowwise(fdY), *oracle.mx_quantize_colwise(fW), "dgrad")
    check_gemm_full(dw, *oracle.mx_quantize_colwise(fdY), *oracle.mx_quantize_colwise(fX), "wgrad")


def upload(codes, scales, orient):
    rows, k = codes.shape
    return mx.MXTensor(torch.from_numpy(np.ascontiguousarray(codes)).cuda(),
                       torch.from_numpy(oracle.mx_scale_swizzle(scales)).cuda(), rows, k, orient)


def test_gemm_on_oracle_operands():
    """GEMM alone, fed with operands the oracle quantised (random codes and
    scales, every E4M3 code except NaN)."""
    g = np.random.Generator(np.random.Philox(17))
    M, N, K = 200, 264, 384
    ac = g.integers(0, 256, (M, K)).astype(np.uint8)
    bc = g.integers(0, 256, (N, K)).astype(np.uint8)
    ac[(ac & 0x7F) == 0x7F] = 0x00
    bc[(bc & 0x7F) == 0x7F] = 0x80
    asc = g.integers(100, 150, (M, K // 32)).astype(np.uint8)
    bsc = g.integers(100, 150, (N, K // 32)).astype(np.uint8)
    y = run_gemm(mx.MX_FPROP, upload(ac, asc, mx.MX_ROWWISE), upload(bc, bsc, mx.MX_ROWWISE))
    check_gemm_full(y, ac, asc, bc, bsc, "oracle operands")


def test_deterministic_bits():
    x = src((512, 1024), 21, spread=2)
    w = src((640, 1024), 22, spread=2)
    xr, _ = gpu_quant(x, mx.MX_ROWWISE)
    wr, _ = gpu_quant(w, mx.MX_ROWWISE)
    y1 = run_gemm(mx.MX_FPROP, xr, wr)
    y2 = run_gemm(mx.MX_FPROP, xr, wr)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_large_grid_bn256():
    """Enough tiles for the 128x256 tile configuration and a multi-wave
    persistent schedule."""
    M, N, K = 2048, 4096 + 192, 384
    x = src((M, K), 31)
    w = src((N, K), 32, std=0.02)
    xr, _ = gpu_quant(x, mx.MX_ROWWISE)
    wr, _ = gpu_quant(w, mx.MX_ROWWISE)
    y = run_gemm(mx.MX_FPROP, xr, wr)
    check_gemm_full(y, *oracle.mx_quantize_rowwise(f64(x)), *oracle.mx_quantize_rowwise(f64(w)), "bn256")


def test_long_k_same_sign():
    """K = 16384 with all-positive operands: the output is ~K times each term,
    so accumulation error is as large as it gets relative to the result."""
    M, N, K = 128, 256, 16384
    g = np.random.Generator(np.random.Philox(41))
    x = workloads.to_bf16(np.abs(g.standard_normal((M, K))) + 0.1)
    w = workloads.to_bf16(np.abs(g.standard_normal((N, K))) + 0.1)
    xr, _ = gpu_quant(x, mx.MX_ROWWISE)
    wr, _ = gpu_quant(w, mx.MX_ROWWISE)
    y = run_gemm(mx.MX_FPROP, xr, wr)
    check_gemm_full(y, *oracle.mx_quantize_rowwise(f64(x)), *oracle.mx_quantize_rowwise(f64(w)), "long K")


def test_output_pitch_and_untouched_columns():
    M, N, K = 256, 200, 256
    x = src((M, K), 51)
    w = src((N, K), 52)
    xr, _ = gpu_quant(x, mx.MX_ROWWISE)
    wr, _ = gpu_quant(w, mx.MX_ROWWISE)
    big = torch.full((M, 264), 7.0, dtype=torch.bfloat16, device="cuda")
    run_gemm(mx.MX_FPROP, xr, wr, out=big[:, :N])
    assert bool((big[:, N:] == 7.0).all())
    check_gemm_full(big[:, :N], *oracle.mx_quantize_rowwise(f64(x)), *oracle.mx_quantize_rowwise(f64(w)), "pitch")


def test_k_zero_writes_zeros():
    a = mx.MXTensor(torch.zeros((64, 0), dtype=torch.uint8, device="cuda"),
                    torch.zeros(16, dtype=torch.uint8, device="cuda"), 64, 0, mx.MX_ROWWISE)
    b = mx.MXTensor(torch.zeros((48, 0), dtype=torch.uint8, device="cuda"),
                    torch.zeros(16, dtype=torch.uint8, device="cuda"), 48, 0, mx.MX_ROWWISE)
    out = torch.full((64, 48), 3.0, dtype=torch.bfloat16, device="cuda")
    mx.gemm(mx.MX_FPROP, a, b, out=out)
    torch.cuda.synchronize()
    assert bool((out == 0).all())


def test_single_linear_config():
    """Single MXFP8 Linear fprop: X[256x512], W[256x512] ~ N(0,1)."""
    d = workloads.single_linear()
    xr, _ = gpu_quant(d["X"], mx.MX_ROWWISE)
    wr, _ = gpu_quant(d["W"], mx.MX_ROWWISE)
    y = run_gemm(mx.MX_FPROP, xr, wr)
    rep = check_gemm_full(y, *oracle.mx_quantize_rowwise(f64(d["X"])), *oracle.mx_quantize_rowwise(f64(d["W"])),
                          "single linear")
    assert rep["nonfinite"] == 0
