"""Dense GEMM with a split tail: when the last round of 256 x 256 tiles leaves
SM pairs idle, those tiles' 128-K blocks are shared out in equal runs, each
run leaves FP32 partial tiles in a workspace and a second kernel adds them in
a fixed order. Checked against the oracle element by element (small cases)
and on sampled entries (the dense FFN dgrad / wgrad contractions), plus
determinism, the caller-workspace entry point and the caller's pitch gap."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import check_gemm_full, check_gemm_sampled, f64, sample_entries

pytestmark = pytest.mark.gpu


def src(shape, seed, std=1.0):
    g = np.random.Generator(np.random.Philox(seed))
    x = g.standard_normal(shape) * std
    R, C = shape
    x *= np.exp2(g.integers(-3, 4, (R, (C + 31) // 32))).repeat(32, axis=1)[:, :C]
    return workloads.to_bf16(x)


def operands(M, N, K, seed):
    x = src((M, K), seed)
    w = src((N, K), seed + 1, std=0.02)
    xr, _ = mx.quantize(x.cuda(), mx.MX_ROWWISE)
    wr, _ = mx.quantize(w.cuda(), mx.MX_ROWWISE)
    torch.cuda.synchronize()
    return x, w, xr, wr


def gemm(xr, wr, out=None):
    """The GEMM with a workspace of the queried size (so it may split)."""
    st = mx.new_status()
    y = mx.gemm(mx.MX_FPROP, xr, wr, out=out, status=st, workspace=mx.gemm_workspace(mx.MX_FPROP, xr, wr))
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return y


def ws_bytes(xr, wr):
    return mx.mx_gemm_workspace_bytes(mx.MX_FPROP, xr.c_operand(), wr.c_operand())


# Each shape leaves a partial last round on a 152-SM GB300 and is split:
# fewer tiles than SM pairs with a long contraction (weight gradients over
# many tokens), with ragged M / N / K.
SPLIT_SHAPES = [(512, 512, 16384), (300, 520, 16000), (520, 700, 16416), (768, 256, 16384), (130, 2100, 16384)]


@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
def test_split_tail_matches_oracle(M, N, K):
    x, w, xr, wr = operands(M, N, K, M + N + K)
    assert ws_bytes(xr, wr) > 0, "shape expected to take the split tail"
    y = gemm(xr, wr)
    check_gemm_full(y, *oracle.mx_quantize_rowwise(f64(x)), *oracle.mx_quantize_rowwise(f64(w)),
                    f"split {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(576, 2048, 16384), (4096, 512, 16384), (4096, 1280, 8192)])
def test_split_tail_training_shapes_sampled(M, N, K):
    """The MLA kv_down and kv_up weight gradients (576 x 2048 and 4096 x 512,
    K = 16384 tokens) and a one-round-plus-tail grid; entries sampled across
    every tile boundary, so the whole-tile rounds and the split tail are both
    covered."""
    x, w, xr, wr = operands(M, N, K, 77 + K)
    assert ws_bytes(xr, wr) > 0
    y = gemm(xr, wr)
    ii, jj = sample_entries(M, N, 600, seed=M + N, tile_m=128, tile_n=256)
    check_gemm_sampled(y, x.cuda(), mx.MX_ROWWISE, w.cuda(), mx.MX_ROWWISE, ii, jj, f"split sampled {M}x{N}x{K}")


def test_split_tail_deterministic_and_workspace_entry_point():
    M, N, K = 520, 700, 16416
    x, w, xr, wr = operands(M, N, K, 5)
    y1 = gemm(xr, wr)
    y2 = gemm(xr, wr)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), "repeated calls differ"
    need = ws_bytes(xr, wr)
    assert need > 0 and need % 16 == 0
    # caller-owned workspace of exactly the queried size: the same split, the same bits
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y3 = torch.empty_like(y1)
    st = mx.new_status()
    mx.mx_gemm_with_workspace(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), y3.data_ptr(), y3.stride(0),
                              ws.data_ptr(), need, st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    # mx_gemm (no workspace) and too small a workspace: whole tiles only,
    # still within the bound
    y5 = mx.gemm(mx.MX_FPROP, xr, wr, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    check_gemm_full(y5, *oracle.mx_quantize_rowwise(f64(x)), *oracle.mx_quantize_rowwise(f64(w)), "mx_gemm")
    for size in (0, need - 16):
        y4 = torch.empty_like(y1)
        mx.mx_gemm_with_workspace(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), y4.data_ptr(), y4.stride(0),
                                  ws.data_ptr() if size else None, size, st.data_ptr(), None)
        torch.cuda.synchronize()
        assert mx.read_status(st) == 0
        check_gemm_full(y4, *oracle.mx_quantize_rowwise(f64(x)), *oracle.mx_quantize_rowwise(f64(w)),
                        f"whole tiles, workspace {size}")


def test_no_split_when_the_last_round_is_full():
    """76 pair tiles on 76 SM pairs: nothing to split, no workspace."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("tile count chosen for a 152-SM GB300")
    M, N, K = 256 * 19, 256 * 4, 1024
    _, _, xr, wr = operands(M, N, K, 9)
    assert ws_bytes(xr, wr) == 0


@pytest.mark.parametrize("aligned", [True, False])
def test_split_tail_pitch_gap_and_unaligned_output(aligned):
    """The reduction kernel writes BF16 rows with bounds: a ragged width inside
    a wider matrix (the columns after N stay NaN), and an output whose rows are
    not 16-byte aligned (element stores)."""
    M, N, K = 512, 300, 16384
    x, w, xr, wr = operands(M, N, K, 11)
    assert ws_bytes(xr, wr) > 0
    ldc = 320
    big = torch.full((M, ldc + 8), float("nan"), dtype=torch.bfloat16, device="cuda")
    view = big[:, :N] if aligned else big[:, 1:N + 1]
    st = mx.new_status()
    ws = mx.gemm_workspace(mx.MX_FPROP, xr, wr)
    mx.mx_gemm_with_workspace(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), view.data_ptr(), big.stride(0),
                              ws.data_ptr(), ws.numel(), st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    h = big.float().cpu().numpy()
    c0 = 0 if aligned else 1
    assert np.all(np.isnan(h[:, :c0])) and np.all(np.isnan(h[:, c0 + N:])), "wrote outside C"
    check_gemm_full(view, *oracle.mx_quantize_rowwise(f64(x)), *oracle.mx_quantize_rowwise(f64(w)),
                    f"split pitch aligned={aligned}")


def test_split_tail_captured_in_cuda_graph():
    """A split-tail GEMM (its partial tiles in the caller's workspace, then the
    reduction launch) recorded into a CUDA graph: replays give the eager call's
    bits."""
    M, N, K = 512, 512, 16384
    _, _, xr, wr = operands(M, N, K, 13)
    assert ws_bytes(xr, wr) > 0
    y_eager = gemm(xr, wr)
    out = torch.zeros_like(y_eager)
    ws = mx.gemm_workspace(mx.MX_FPROP, xr, wr)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        mx.mx_gemm_with_workspace(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), out.data_ptr(), out.stride(0),
                                  ws.data_ptr(), ws.numel(), None, stream.cuda_stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), y_eager.view(torch.int16))
