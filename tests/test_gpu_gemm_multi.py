"""Several independent GEMMs in one mx_gemm_multi launch (the dgrad and wgrad
of a Linear layer's backward pass, and mixed ragged shapes): every output
checked against the oracle, element by element at small sizes and on sampled
entries at the dense FFN size; determinism, K = 0, the caller's pitch gap, and
the one-launch-per-GEMM path taken when the problems do not fill the GPU."""
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
    x *= np.exp2(g.integers(-3, 4, ((R + 31) // 32, C))).repeat(32, axis=0)[:R, :]
    return workloads.to_bf16(x)


def both(x):
    r, c = mx.quantize(x.cuda(), mx.MX_BOTH)
    torch.cuda.synchronize()
    return r, c


def rowq(x):
    r, _ = mx.quantize(x.cuda(), mx.MX_ROWWISE)
    torch.cuda.synchronize()
    return r


def run_multi(problems):
    st = mx.new_status()
    outs = mx.gemm_multi(problems, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return outs


def linear_backward(M, N, K, seed):
    """X [M, K], W [N, K], dY [M, N] and their copies; the dgrad / wgrad problems."""
    X, W, dY = src((M, K), seed), src((N, K), seed + 1, 0.02), src((M, N), seed + 2)
    (xr, xc), (wr, wc), (dr, dc) = both(X), both(W), both(dY)
    return X, W, dY, [(mx.MX_DGRAD, dr, wc), (mx.MX_WGRAD, dc, xc)]


def test_dgrad_wgrad_fused_matches_oracle():
    M, N, K = 2048, 1536, 2048   # 64 + 48 pair tiles: one launch
    X, W, dY, probs = linear_backward(M, N, K, 1)
    dX, dW = run_multi(probs)
    d64, w64, x64 = f64(dY), f64(W), f64(X)
    check_gemm_full(dX, *oracle.mx_quantize_rowwise(d64), *oracle.mx_quantize_colwise(w64), "dgrad (multi)")
    check_gemm_full(dW, *oracle.mx_quantize_colwise(d64), *oracle.mx_quantize_colwise(x64), "wgrad (multi)")


def test_dense_ffn_backward_sampled():
    """dgrad 8192 x 2048 (K 10944) and wgrad 10944 x 2048 (K 8192) of the
    dense FFN up-projection in one launch."""
    M, K, N = 8192, 2048, 10944
    X, W, dY, probs = linear_backward(M, N, K, 2)
    dX, dW = run_multi(probs)
    Xc, Wc, dYc = X.cuda(), W.cuda(), dY.cuda()
    ii, jj = sample_entries(M, K, 400, seed=3, tile_m=128, tile_n=256)
    check_gemm_sampled(dX, dYc, mx.MX_ROWWISE, Wc, mx.MX_COLWISE, ii, jj, "dgrad sampled")
    ii, jj = sample_entries(N, K, 400, seed=4, tile_m=128, tile_n=256)
    check_gemm_sampled(dW, dYc, mx.MX_COLWISE, Xc, mx.MX_COLWISE, ii, jj, "wgrad sampled")


def test_ragged_mixed_problems_and_determinism():
    """Four problems of different modes and ragged sizes (fused: together they
    fill the GPU), run twice: identical bits, each within the oracle's bound."""
    shapes = [(1000, 520, 288), (300, 2100, 1024), (4096, 384, 160), (2176, 1000, 2080)]
    probs, refs = [], []
    for i, (M, N, K) in enumerate(shapes):
        a, b = src((M, K), 10 + i), src((N, K), 20 + i, 0.05)
        probs.append((mx.MX_FPROP, rowq(a), rowq(b)))
        refs.append((a, b))
    outs1 = run_multi(probs)
    outs2 = run_multi(probs)
    for (a, b), o1, o2, (M, N, K) in zip(refs, outs1, outs2, shapes):
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)), f"{M}x{N}x{K} not deterministic"
        check_gemm_full(o1, *oracle.mx_quantize_rowwise(f64(a)), *oracle.mx_quantize_rowwise(f64(b)),
                        f"multi {M}x{N}x{K}")


def test_small_problems_take_one_launch_each():
    """Problems that cannot fill the GPU together (or N <= 128) run as separate
    GEMMs; results as mx_gemm's."""
    shapes = [(256, 128, 256), (129, 200, 96)]
    probs, refs = [], []
    for i, (M, N, K) in enumerate(shapes):
        a, b = src((M, K), 30 + i), src((N, K), 40 + i, 0.05)
        probs.append((mx.MX_FPROP, rowq(a), rowq(b)))
        refs.append((a, b))
    outs = run_multi(probs)
    for (a, b), o, (M, N, K) in zip(refs, outs, shapes):
        check_gemm_full(o, *oracle.mx_quantize_rowwise(f64(a)), *oracle.mx_quantize_rowwise(f64(b)),
                        f"separate {M}x{N}x{K}")


def test_k_zero_and_pitch_gap():
    """A K = 0 problem writes zeros; outputs of ragged width inside wider NaN
    matrices keep the columns after N."""
    M, N, K = 4096, 1000, 512   # 2 x 64 pair tiles: the fused launch
    a, b = src((M, K), 50), src((N, K), 51, 0.05)
    ar, br = rowq(a), rowq(b)
    big = torch.full((M, 1016), float("nan"), dtype=torch.bfloat16, device="cuda")
    big2 = torch.full((M, 1016), float("nan"), dtype=torch.bfloat16, device="cuda")
    zero_a = mx.MXOperandC(None, None, M, 0, 0, mx.MX_ROWWISE, 0)
    zero_b = mx.MXOperandC(None, None, 8, 0, 0, mx.MX_ROWWISE, 0)
    descs = [mx.MXGemmProblemC(ar.c_operand(), br.c_operand(), big.data_ptr(), big.stride(0), mx.MX_FPROP, 0),
             mx.MXGemmProblemC(ar.c_operand(), br.c_operand(), big2.data_ptr(), big2.stride(0), mx.MX_FPROP, 0),
             # [M, 8] output in columns 1008 .. 1015 of big2: apart from the other outputs
             mx.MXGemmProblemC(zero_a, zero_b, big2[:, 1008:].data_ptr(), big2.stride(0), mx.MX_FPROP, 0)]
    st = mx.new_status()
    mx.mx_gemm_multi(descs, st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    h, h2 = big.float().cpu().numpy(), big2.float().cpu().numpy()
    assert np.all(np.isnan(h[:, N:])) and np.all(np.isnan(h2[:, N:1008])), "wrote after N"
    assert np.all(h2[:, 1008:1016] == 0), "K = 0 problem did not write zeros"
    for out in (big[:, :N], big2[:, :N]):
        check_gemm_full(out, *oracle.mx_quantize_rowwise(f64(a)), *oracle.mx_quantize_rowwise(f64(b)), "pitch gap")


def test_multi_captured_in_cuda_graph():
    """dgrad + wgrad in one launch, recorded into a CUDA graph and replayed:
    the eager call's bits."""
    X, W, dY, probs = linear_backward(2048, 1536, 2048, 60)
    dX, dW = run_multi(probs)
    gX, gW = torch.zeros_like(dX), torch.zeros_like(dW)
    descs = [mx.MXGemmProblemC(a.c_operand(), b.c_operand(), o.data_ptr(), o.stride(0), mode, 0)
             for (mode, a, b), o in zip(probs, (gX, gW))]
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        mx.mx_gemm_multi(descs, None, stream.cuda_stream)
    with torch.cuda.stream(stream):
        graph.replay()
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(gX.view(torch.int16), dX.view(torch.int16))
    assert torch.equal(gW.view(torch.int16), dW.view(torch.int16))


def test_balanced_schedule_mla_backward_matches_separate_calls():
    """MLA q_down backward: dgrad 16384 x 2048 (K 1536) and wgrad 1536 x 2048
    (K 16384 tokens) in one launch. Their tiles differ ~9x in length, so the
    launch takes the balanced (longest-first) schedule; every tile is computed
    the same way whichever cluster runs it, so the outputs equal separate
    mx_gemm calls bit for bit, and sampled entries match the oracle."""
    M, K, N = 16384, 2048, 1536
    X, W, dY, probs = linear_backward(M, N, K, 70)
    dX, dW = run_multi(probs)
    st = mx.new_status()
    sX = mx.gemm(probs[0][0], probs[0][1], probs[0][2], status=st)
    sW = mx.gemm(probs[1][0], probs[1][1], probs[1][2], status=st)
    ok = torch.cuda.synchronize() or mx.read_status(st) == 0
    assert ok
    assert torch.equal(dX.view(torch.int16), sX.view(torch.int16)), "dgrad differs from the separate call"
    assert torch.equal(dW.view(torch.int16), sW.view(torch.int16)), "wgrad differs from the separate call"
    Xc, Wc, dYc = X.cuda(), W.cuda(), dY.cuda()
    ii, jj = sample_entries(M, K, 300, seed=71, tile_m=128, tile_n=256)
    check_gemm_sampled(dX, dYc, mx.MX_ROWWISE, Wc, mx.MX_COLWISE, ii, jj, "q_down dgrad (scheduled)")
    ii, jj = sample_entries(N, K, 300, seed=72, tile_m=128, tile_n=256)
    check_gemm_sampled(dW, dYc, mx.MX_COLWISE, Xc, mx.MX_COLWISE, ii, jj, "q_down wgrad (scheduled)")
