"""The GEMM entry point for callers that cannot allocate device memory.

Some callers may not allocate at all: code running inside a memory
allocator's own callbacks, runtimes that reserve all their device memory at
start-up, plug-ins that only receive input and output buffers. For them
mx_gemm_static_workspace runs the dense GEMM with its split-tail scratch in a
fixed array the library declares in device memory, instead of a workspace
the caller passes to mx_gemm_with_workspace.

These tests call it through the C ABI and compare its output with the
caller-workspace entry point's on the same operands, for two calls in a row
(the array keeps the previous call's partial tiles, which must not leak into
the next result). The file is named to be collected last.
"""
import pytest
import torch

import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import check_gemm_sampled, sample_entries

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed, mode):
    """Quantised operands of one GEMM of the given mode, and their BF16 sources."""
    if mode == mx.MX_WGRAD:
        # dW[N_out, K_out] = dY^T X over M_tok tokens: a = dY col copy, b = X col copy
        dy = workloads.normal_bf16((K, M), seed)
        x = workloads.normal_bf16((K, N), seed + 1)
        _, a = mx.quantize(dy.cuda(), mx.MX_COLWISE)
        _, b = mx.quantize(x.cuda(), mx.MX_COLWISE)
        return a, b, (dy, mx.MX_COLWISE, x, mx.MX_COLWISE)
    x = workloads.normal_bf16((M, K), seed)
    w = workloads.normal_bf16((N, K), seed + 1, 0.02)
    a, _ = mx.quantize(x.cuda(), mx.MX_ROWWISE)
    b, _ = mx.quantize(w.cuda(), mx.MX_ROWWISE)
    return a, b, (x, mx.MX_ROWWISE, w, mx.MX_ROWWISE)


def _with_caller_workspace(mode, a, b):
    need = mx.mx_gemm_workspace_bytes(mode, a.c_operand(), b.c_operand())
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device="cuda")
    st = mx.new_status()
    mx.mx_gemm_with_workspace(mode, a.c_operand(), b.c_operand(), out.data_ptr(), out.stride(0), ws.data_ptr(), need,
                              st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return out, need


def _with_static_workspace(mode, a, b, out):
    st = mx.new_status()
    mx.mx_gemm_static_workspace(mode, a.c_operand(), b.c_operand(), out.data_ptr(), out.stride(0), st.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0


# (M, N, K, mode): weight gradients with a long contraction and few output
# tiles, whose last round splits (the kv_down and kv_up weight gradients of the
# MLA set), and a GEMM of whole tiles only.
CASES = [(576, 2048, 16384, mx.MX_WGRAD), (4096, 512, 16384, mx.MX_WGRAD), (1024, 1536, 2048, mx.MX_FPROP)]


def test_static_workspace_matches_caller_workspace_two_calls_in_a_row():
    prepared = []
    for i, (M, N, K, mode) in enumerate(CASES):
        a, b, srcs = _operands(M, N, K, 900 + 10 * i, mode)
        ref, need = _with_caller_workspace(mode, a, b)
        assert need <= mx.MX_STATIC_WORKSPACE_BYTES
        prepared.append((mode, a, b, srcs, ref, need))
    # the first two cases split their tail: the array is really used
    assert prepared[0][5] > 0 and prepared[1][5] > 0
    for mode, a, b, srcs, ref, _ in prepared:
        outs = []
        for call in range(2):
            out = torch.full((a.rows, b.rows), float("nan"), dtype=torch.bfloat16, device="cuda")
            _with_static_workspace(mode, a, b, out)
            outs.append(out)
            # same bits as the caller-workspace entry point (same kernels, same
            # split, same summation order) ...
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}"
        # ... and, like it, within the GEMM tolerance of the FP64 reference
        ii, jj = sample_entries(ref.shape[0], ref.shape[1], 512, 77, tile_n=256)
        rep = check_gemm_sampled(outs[1], *srcs, ii, jj, what="static workspace")
        assert rep["fail"] == 0
    # a second round over the cases in reverse order: each call starts from the
    # array as a different GEMM left it
    for mode, a, b, _, ref, _ in reversed(prepared):
        out = torch.empty((a.rows, b.rows), dtype=torch.bfloat16, device="cuda")
        _with_static_workspace(mode, a, b, out)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_static_workspace_rejects_bad_arguments_like_mx_gemm():
    a, b, _ = _operands(256, 256, 512, 950, mx.MX_FPROP)
    out = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # wrong orientation for the mode
    with pytest.raises(mx.MXError) as e:
        mx.mx_gemm_static_workspace(mx.MX_WGRAD, a.c_operand(), b.c_operand(), out.data_ptr(), out.stride(0), None, s)
    assert e.value.status == 1
    # ldc < N
    with pytest.raises(mx.MXError) as e:
        mx.mx_gemm_static_workspace(mx.MX_FPROP, a.c_operand(), b.c_operand(), out.data_ptr(), 100, None, s)
    assert e.value.status == 1
