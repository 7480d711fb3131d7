"""FP32-input quantiser (weight refresh from the FP32 master) vs the oracle,
bit for bit: data codes, scale codes and the padding bytes of the swizzled
scale tiles. The oracle reads the FP32 values exactly (float64)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import assert_bytes_equal, u8

pytestmark = pytest.mark.gpu


def exact(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().double().numpy()


def check(x: torch.Tensor, row, col, what: str):
    v = exact(x)
    if row is not None:
        d, s = oracle.mx_quantize_rowwise(v)
        assert_bytes_equal(u8(row.data), d, what + " row data")
        assert_bytes_equal(u8(row.scale), oracle.mx_scale_swizzle(s), what + " row scales")
    if col is not None:
        d, s = oracle.mx_quantize_colwise(v)
        assert_bytes_equal(u8(col.data), d, what + " col data")
        assert_bytes_equal(u8(col.scale), oracle.mx_scale_swizzle(s), what + " col scales")


def run(x: torch.Tensor, axis):
    st = mx.new_status()
    row, col = mx.quantize(x.cuda(), axis, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return row, col


def hand_rows() -> torch.Tensor:
    """Rows holding the hand-worked FP32 blocks (values BF16 cannot hold, FP32
    subnormals, NaN, Inf), the rest of the matrix seeded N(0, 1)."""
    x = workloads.fp32_master((64, 64), seed=3100, std=1.0).numpy().copy()
    x[0, :4] = [256.0, 1.0625 + 2.0 ** -20, 1.0625, -(1.0625 + 2.0 ** -20)]
    x[0, 4:32] = 0.0
    x[1, :32] = 0.0
    x[1, :2] = [512.0 - 2.0 ** -15, 3.0]
    x[2, :32] = 0.0
    x[2, :4] = [448.0, 2.0 ** -10, 2.0 ** -10 + 2.0 ** -30, -(2.0 ** -10 + 2.0 ** -30)]
    x[3, :32] = np.float32(2.0 ** -140) * np.arange(-16, 16, dtype=np.float32)  # FP32 subnormals
    x[4, 5] = np.nan
    x[5, 40] = -np.inf
    x[6, 33] = np.float32(3.4e38)                      # near the FP32 maximum
    x[7, :] = 0.0
    x[7, 3] = -0.0
    return torch.from_numpy(x)


def test_f32_hand_rows_both_copies():
    x = hand_rows()
    row, col = run(x, mx.MX_BOTH)
    check(x, row, col, "hand rows")
    # the midpoint neighbour (an FP32-only value) rounds up: 0x39, not 0x38
    assert u8(row.data)[0, 1] == 0x39 and u8(row.data)[0, 2] == 0x38


@pytest.mark.parametrize("R,C", [(32, 32), (128, 64), (160, 96), (288, 224), (1024, 2048), (96, 4160)])
def test_f32_dense_both(R, C):
    x = workloads.fp32_master((R, C), seed=3200 + R + C)
    row, col = run(x, mx.MX_BOTH)
    check(x, row, col, f"f32 {R}x{C}")


@pytest.mark.parametrize("axis", [mx.MX_ROWWISE, mx.MX_COLWISE])
def test_f32_single_copy(axis):
    x = workloads.fp32_master((256, 160), seed=3300)
    row, col = run(x, axis)
    assert (row is None) == (axis == mx.MX_COLWISE) and (col is None) == (axis == mx.MX_ROWWISE)
    check(x, row, col, "f32 single copy")


def test_f32_input_pitch():
    """A view with row pitch 196 floats (784 bytes) of a wider matrix."""
    wide = workloads.fp32_master((192, 196), seed=3400)
    x = wide[:, :160]
    st = mx.new_status()
    xd = wide.cuda()[:, :160]
    row, col = mx.quantize(xd, mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    check(x, row, col, "f32 pitch")


def test_f32_stacked_with_batch_gap():
    """Stacked FP32 masters [E, N, K] whose matrices sit 64 floats apart beyond
    their own size: each matrix's copies equal the oracle's of that matrix."""
    E, N, K = 5, 160, 96
    big = workloads.fp32_master((E, N * K + 64), seed=3500)
    w_host = big[:, : N * K].reshape(E, N, K)
    dev = big.cuda()
    w = torch.as_strided(dev, (E, N, K), (N * K + 64, K, 1))
    st = mx.new_status()
    row, col = mx.quantize_stacked(w, mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    for e in range(E):
        v = exact(w_host[e])
        d, s = oracle.mx_quantize_rowwise(v)
        assert_bytes_equal(u8(row.data[e]), d, f"stacked row data {e}")
        assert_bytes_equal(u8(row.scale[e]), oracle.mx_scale_swizzle(s), f"stacked row scales {e}")
        d, s = oracle.mx_quantize_colwise(v)
        assert_bytes_equal(u8(col.data[e]), d, f"stacked col data {e}")
        assert_bytes_equal(u8(col.scale[e]), oracle.mx_scale_swizzle(s), f"stacked col scales {e}")


def test_f32_matches_bf16_path_on_bf16_values():
    """On FP32 inputs that are BF16 numbers, both input paths give the same bytes."""
    xb = workloads.normal_bf16((256, 192), 3600)
    r1, c1 = run(xb, mx.MX_BOTH)
    r2, c2 = run(xb.float(), mx.MX_BOTH)
    for a, b in [(r1.data, r2.data), (r1.scale, r2.scale), (c1.data, c2.data), (c1.scale, c2.scale)]:
        assert torch.equal(a, b)


def test_f32_full_size_expert_refresh():
    """The routed experts' gate_up master [64, 2816, 2048] in FP32, refreshed in
    one launch; experts 0, 31 and 63 checked entirely against the oracle."""
    E, N, K = 64, 2816, 2048
    w = workloads.fp32_master((E, N, K), seed=3700).cuda()
    st = mx.new_status()
    row, col = mx.quantize_stacked(w, mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    for e in (0, 31, 63):
        v = exact(w[e])
        d, s = oracle.mx_quantize_rowwise(v)
        assert_bytes_equal(u8(row.data[e]), d, f"expert {e} row data")
        assert_bytes_equal(u8(row.scale[e]), oracle.mx_scale_swizzle(s), f"expert {e} row scales")
        d, s = oracle.mx_quantize_colwise(v)
        assert_bytes_equal(u8(col.data[e]), d, f"expert {e} col data")
        assert_bytes_equal(u8(col.scale[e]), oracle.mx_scale_swizzle(s), f"expert {e} col scales")
