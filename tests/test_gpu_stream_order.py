"""Stream order between back-to-back launches. Every kernel lets the next one
on the stream be scheduled early and waits (griddepcontrol.wait) before it
touches global memory, so consecutive calls must still see each other's
writes in stream order. Each chain below runs twice: issued back to back, and
with the host synchronising after every call (no overlap possible). The two
runs must agree bit for bit."""
import pytest
import torch

import workloads
import mxfp8_block_scaled_gb300 as mx

pytestmark = pytest.mark.gpu


def bits(t):
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.uint8)


def run(steps, sync):
    out = []
    for f in steps:
        out.append(f())
        if sync:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    return out


def test_read_after_write_chain():
    """quantise -> GEMM -> quantise the GEMM's output -> GEMM: each launch
    reads what the launch right before it wrote."""
    X = workloads.normal_bf16((2048, 1024), 11).cuda()
    W1 = workloads.normal_bf16((1536, 1024), 12, 0.05).cuda()
    W2 = workloads.normal_bf16((1024, 1536), 13, 0.05).cuda()

    def chain(sync):
        st = {}
        steps = [lambda: st.__setitem__("x", mx.quantize(X, mx.MX_ROWWISE)[0]),
                 lambda: st.__setitem__("w1", mx.quantize(W1, mx.MX_ROWWISE)[0]),
                 lambda: st.__setitem__("y", mx.gemm(mx.MX_FPROP, st["x"], st["w1"])),
                 lambda: st.__setitem__("yq", mx.quantize(st["y"], mx.MX_ROWWISE)[0]),
                 lambda: st.__setitem__("w2", mx.quantize(W2, mx.MX_ROWWISE)[0]),
                 lambda: st.__setitem__("z", mx.gemm(mx.MX_FPROP, st["yq"], st["w2"]))]
        run(steps, sync)
        return st

    a, b = chain(False), chain(True)
    assert torch.equal(bits(a["y"]), bits(b["y"]))
    assert torch.equal(bits(a["yq"].data), bits(b["yq"].data))
    assert torch.equal(bits(a["yq"].scale), bits(b["yq"].scale))
    assert torch.equal(bits(a["z"]), bits(b["z"]))


def test_write_after_read_overwrite():
    """A GEMM reads the quantised X; the next launch overwrites that buffer
    with another matrix's codes; a second GEMM reads the new codes. The first
    GEMM must see only the old codes."""
    M, K, N = 4096, 2048, 2048
    X1 = workloads.normal_bf16((M, K), 21).cuda()
    X2 = workloads.normal_bf16((M, K), 22).cuda()
    W = workloads.normal_bf16((N, K), 23, 0.05).cuda()
    wr, _ = mx.quantize(W, mx.MX_ROWWISE)
    x1r, _ = mx.quantize(X1, mx.MX_ROWWISE)
    x2r, _ = mx.quantize(X2, mx.MX_ROWWISE)
    torch.cuda.synchronize()
    ref1 = mx.gemm(mx.MX_FPROP, x1r, wr)
    torch.cuda.synchronize()
    ref2 = mx.gemm(mx.MX_FPROP, x2r, wr)
    torch.cuda.synchronize()

    xr, _ = mx.quantize(X1, mx.MX_ROWWISE)
    torch.cuda.synchronize()
    sp = torch.cuda.current_stream().cuda_stream
    y1 = mx.gemm(mx.MX_FPROP, xr, wr)
    mx.mx_quantize(X2.data_ptr(), M, K, K, mx.MX_ROWWISE, xr.data.data_ptr(), xr.scale.data_ptr(), None, None, None,
                   0, 0, None, sp)
    y2 = mx.gemm(mx.MX_FPROP, xr, wr)
    torch.cuda.synchronize()
    assert torch.equal(bits(y1), bits(ref1)), "the first GEMM saw codes written after it"
    assert torch.equal(bits(y2), bits(ref2)), "the second GEMM missed the new codes"


def test_split_tail_then_consumer():
    """A GEMM whose last round is split (GEMM launch, then the reduction
    launch), then a quantisation of its output right behind the reduction."""
    a = workloads.normal_bf16((512, 16384), 31).cuda()
    b = workloads.normal_bf16((512, 16384), 32, 0.05).cuda()
    ar, _ = mx.quantize(a, mx.MX_ROWWISE)
    br, _ = mx.quantize(b, mx.MX_ROWWISE)
    ws = mx.gemm_workspace(mx.MX_FPROP, ar, br)
    torch.cuda.synchronize()

    def chain(sync):
        st = {}
        steps = [lambda: st.__setitem__("y", mx.gemm(mx.MX_FPROP, ar, br, workspace=ws)),
                 lambda: st.__setitem__("yq", mx.quantize(st["y"], mx.MX_BOTH))]
        run(steps, sync)
        return st

    a1, a2 = chain(False), chain(True)
    assert torch.equal(bits(a1["y"]), bits(a2["y"]))
    for i in range(2):
        assert torch.equal(bits(a1["yq"][i].data), bits(a2["yq"][i].data))
        assert torch.equal(bits(a1["yq"][i].scale), bits(a2["yq"][i].scale))
