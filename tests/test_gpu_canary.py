"""Guard bytes: every output buffer sits inside a larger allocation filled with
0xA5; after the call the bytes outside the region the header says is written
must be unchanged (catches stray stores past rows, columns, pitch gaps and the
ends of scale buffers)."""
import numpy as np
import pytest
import torch

import workloads
import mxfp8_block_scaled_gb300 as mx

pytestmark = pytest.mark.gpu
G = 0xA5
PAD = 4096


def guarded(nbytes):
    buf = torch.full((nbytes + 2 * PAD,), G, dtype=torch.uint8, device="cuda")
    return buf, buf.data_ptr() + PAD


def check_guards(buf, nbytes, what):
    h = buf.cpu().numpy()
    assert np.all(h[:PAD] == G), f"{what}: bytes before the buffer written"
    assert np.all(h[PAD + nbytes:] == G), f"{what}: bytes after the buffer written"


def run_ok(fn, *args):
    st = mx.new_status()
    fn(*args[:-2], st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0


def test_quantize_dense_buffers():
    R, C = 160, 96
    x = workloads.normal_bf16((R, C), 6000).cuda()
    rd, rs, cd, cs = R * C, mx.mx_scale_bytes(R, C), C * R, mx.mx_scale_bytes(C, R)
    bufs = [guarded(n) for n in (rd, rs, cd, cs)]
    run_ok(mx.mx_quantize, x.data_ptr(), R, C, C, mx.MX_BOTH, bufs[0][1], bufs[1][1], bufs[2][1], bufs[3][1],
           None, 0, 0, None, None)
    for (b, _), n, w in zip(bufs, (rd, rs, cd, cs), ("row data", "row scale", "col data", "col scale")):
        check_guards(b, n, w)


def test_quantize_grouped_capacity_tail_untouched():
    counts = [37, 0, 100]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    o = torch.from_numpy(offs).cuda()
    R, C = int(offs[-1]), 64
    padded = mx.mx_grouped_padded_rows(offs)
    cap = padded + 256                       # columns [padded, cap) are not written
    x = workloads.normal_bf16((R, C), 6001).cuda()
    cd = torch.full((C, cap), G, dtype=torch.uint8, device="cuda")
    cs, csp = guarded(mx.mx_scale_bytes(C, cap))
    run_ok(mx.mx_quantize, x.data_ptr(), R, C, C, mx.MX_COLWISE, None, None, cd.data_ptr(), csp, o.data_ptr(), 3,
           cap, None, None)
    assert np.all(cd.cpu().numpy()[:, padded:] == G), "grouped col data beyond the padded total"
    check_guards(cs, mx.mx_scale_bytes(C, cap), "grouped col scale")


@pytest.mark.parametrize("swiglu", [False, True])
def test_grouped_outputs_pitch_gap(swiglu):
    counts = [100, 0, 156]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    o = torch.from_numpy(offs).cuda()
    M, K, N = int(offs[-1]), 256, 512
    x = workloads.normal_bf16((M, K), 6002).cuda()
    w = workloads.normal_bf16((3, N, K), 6003, 0.05).cuda()
    xr, _ = mx.quantize(x, mx.MX_ROWWISE)
    wr, _ = mx.quantize_stacked(w, mx.MX_ROWWISE)
    ncols = N // 2 if swiglu else N
    ldc = ncols + 24
    out = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = mx.new_status()
    if swiglu:
        mx.mx_grouped_gemm_swiglu(xr.c_operand(), wr.c_operand(), o.data_ptr(), 3, out.data_ptr(), ldc, st.data_ptr(),
                                  None)
    else:
        mx.mx_grouped_gemm(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), o.data_ptr(), 3, out.data_ptr(), ldc,
                           st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    h = out.float().cpu().numpy()
    assert np.all(np.isnan(h[:, ncols:])), "pitch gap written"
    assert np.all(np.isfinite(h[:, :ncols])), "output not fully written"


def test_grouped_wgrad_pitch_gap():
    counts = [100, 0, 156]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    o = torch.from_numpy(offs).cuda()
    M, N, Kout = int(offs[-1]), 192, 160
    cap = mx.mx_grouped_padded_rows(offs)
    dy = workloads.normal_bf16((M, N), 6004).cuda()
    x = workloads.normal_bf16((M, Kout), 6005).cuda()
    _, dc = mx.quantize(dy, mx.MX_COLWISE, group_offsets=o, col_capacity=cap)
    _, xc = mx.quantize(x, mx.MX_COLWISE, group_offsets=o, col_capacity=cap)
    ldc = Kout + 32
    out = torch.full((3, N, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = mx.new_status()
    mx.mx_grouped_gemm(mx.MX_WGRAD, dc.c_operand(), xc.c_operand(), o.data_ptr(), 3, out.data_ptr(), ldc,
                       st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    h = out.float().cpu().numpy()
    assert np.all(np.isnan(h[:, :, Kout:])), "wgrad pitch gap written"
    assert np.all(h[1, :, :Kout] == 0.0), "empty expert's dW must be exactly zero"


def test_f32_and_blockwise_quant_buffers():
    R, C = 160, 256
    xf = workloads.fp32_master((R, C), seed=6006).cuda()
    rd, rs, cd, cs = R * C, mx.mx_scale_bytes(R, C), C * R, mx.mx_scale_bytes(C, R)
    bufs = [guarded(n) for n in (rd, rs, cd, cs)]
    run_ok(mx.mx_quantize_f32, xf.data_ptr(), 1, R, C, C, 0, mx.MX_BOTH, bufs[0][1], bufs[1][1], bufs[2][1],
           bufs[3][1], None, None)
    for (b, _), n, w in zip(bufs, (rd, rs, cd, cs), ("f32 row data", "f32 row scale", "f32 col data", "f32 col scale")):
        check_guards(b, n, w)
    xb = workloads.normal_bf16((R, C), 6007).cuda()
    for block, sbytes in ((1, 4 * R * (C // 128)), (128, 4 * ((R + 127) // 128) * (C // 128))):
        d, dp = guarded(R * C)
        s, sp = guarded(sbytes)
        run_ok(mx.mx_quantize_fp8_blockwise, xb.data_ptr(), R, C, C, block, dp, sp, None, None)
        check_guards(d, R * C, f"blockwise {block} data")
        check_guards(s, sbytes, f"blockwise {block} scale")


def test_blockwise_gemm_pitch_gap():
    M, N, K = 200, 300, 384
    x = workloads.normal_bf16((M, K), 6008).cuda()
    w = workloads.normal_bf16((N, K), 6009, 0.02).cuda()
    qa, qb = mx.quantize_fp8_blockwise(x, 1), mx.quantize_fp8_blockwise(w, 128)
    ldc = N + 20
    out = torch.full((M + 3, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = mx.new_status()
    mx.mx_gemm_fp8_blockwise(qa.data.data_ptr(), qa.scale.data_ptr(), M, qb.data.data_ptr(), qb.scale.data_ptr(), N, K,
                             out.data_ptr(), ldc, st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    h = out.float().cpu().numpy()
    assert np.all(np.isnan(h[:M, N:])) and np.all(np.isnan(h[M:])), "blockwise GEMM wrote outside C"
    assert np.all(np.isfinite(h[:M, :N]))


@pytest.mark.parametrize("M,N,K", [(200, 300, 384), (256, 1000, 256), (640, 4100, 512)])
def test_dense_gemm_pitch_gap_ragged_width(M, N, K):
    """Output widths that are not a multiple of 8 elements, inside a wider
    matrix: the columns right after N belong to the caller."""
    x = workloads.normal_bf16((M, K), 6010 + N).cuda()
    w = workloads.normal_bf16((N, K), 6011 + N, 0.02).cuda()
    xr, _ = mx.quantize(x, mx.MX_ROWWISE)
    wr, _ = mx.quantize(w, mx.MX_ROWWISE)
    ldc = (N + 7) // 8 * 8 + 16
    big = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = mx.new_status()
    mx.mx_gemm(mx.MX_FPROP, xr.c_operand(), wr.c_operand(), big.data_ptr(), ldc, st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    h = big.float().cpu().numpy()
    assert np.all(np.isnan(h[:, N:])), "columns after N written"
    assert np.all(np.isfinite(h[:, :N]))
