"""GPU grouped gate_up fprop with the SwiGLU epilogue vs the oracle
(gate_up GEMM in float64, SwiGLU in float64 on the unrounded dots), within
the tolerance derived from the GEMM's FP32-accumulation bound."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import f64, logical_scales

pytestmark = pytest.mark.gpu


def run_case(counts, K, F, seed, rows=None):
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    E = len(counts)
    M = int(offs[-1])
    X = workloads.normal_bf16((M, K), seed)
    W = workloads.normal_bf16((E, 2 * F, K), seed + 1, 0.05)
    o = torch.from_numpy(offs).cuda()
    xr, _ = mx.quantize(X.cuda(), mx.MX_ROWWISE)
    wr, _ = mx.quantize_stacked(W.cuda(), mx.MX_ROWWISE)
    st = mx.new_status()
    out = mx.grouped_gemm_swiglu(xr, wr, o, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0 and out.shape == (M, F)
    ac, asc = oracle.mx_quantize_rowwise(f64(X))
    wq = [oracle.mx_quantize_rowwise(f64(W[e])) for e in range(E)]
    bc, bs = np.stack([w[0] for w in wq]), np.stack([w[1] for w in wq])
    got = f64(out)
    if rows is not None:   # sampled rows: the oracle on just those rows of each expert
        sel_offs = [0]
        sel = []
        for e in range(E):
            r = [i for i in rows if offs[e] <= i < offs[e + 1]]
            sel += r
            sel_offs.append(len(sel))
        sel = np.array(sel, dtype=np.int64)
        ref, gate, up, Sg, Su = oracle.mx_grouped_swiglu_ref(ac[sel], asc[sel], bc, bs, np.array(sel_offs))
        got = got[sel]
    else:
        ref, gate, up, Sg, Su = oracle.mx_grouped_swiglu_ref(ac, asc, bc, bs, offs)
    ok = oracle.swiglu_within_tolerance(got, ref, gate, up, Sg, Su)
    if not ok.all():
        bad = np.argwhere(~ok)[:8]
        raise AssertionError(f"swiglu {counts} F={F}: {int((~ok).sum())} of {ok.size} outside; first "
                             f"{[(tuple(i), got[tuple(i)], ref[tuple(i)]) for i in bad]}")
    return got, ref


@pytest.mark.parametrize("counts,F", [([100, 0, 156], 128), ([37, 0, 300, 1, 128], 256),
                                      ([0, 0, 129], 384), ([256], 128), ([5, 127, 128, 0, 0, 1000, 33, 2], 256)])
def test_grouped_swiglu(counts, F):
    run_case(counts, 256, F, 70 + F + len(counts))


def test_grouped_swiglu_long_k_and_signs():
    """K = 2048 and values on both sides of the SiLU knee: large negative gates
    give ~0, large positive gates pass the gate through."""
    got, ref = run_case([300, 212], 2048, 256, 90)
    assert np.isfinite(got).all()


def test_grouped_swiglu_full_size_sampled():
    """The routed experts' gate_up (K = 2048, 2F = 2816) over 49152 Zipf-routed
    rows with the fused SwiGLU; 3 rows of every expert checked against the
    oracle (first, middle, last)."""
    counts = workloads.moe_counts()
    offs = np.concatenate([[0], np.cumsum(counts)])
    rows = []
    for e in range(len(counts)):
        if counts[e]:
            rows += sorted({int(offs[e]), int(offs[e] + counts[e] // 2), int(offs[e + 1] - 1)})
    run_case(counts, 2048, 1408, 95, rows=rows)


def test_swiglu_equals_gemm_then_swiglu_of_its_bf16_is_close():
    """Cross-check against the plain grouped GEMM on the GPU: SwiGLU of its BF16
    output differs from the fused result by no more than BF16 rounding of the
    gate and up values allows (the fused path rounds once, at the end)."""
    counts = [64, 192]
    K, F = 512, 256
    offs = np.array([0, 64, 256], dtype=np.int64)
    X = workloads.normal_bf16((256, K), 97)
    W = workloads.normal_bf16((2, 2 * F, K), 98, 0.05)
    o = torch.from_numpy(offs).cuda()
    xr, _ = mx.quantize(X.cuda(), mx.MX_ROWWISE)
    wr, _ = mx.quantize_stacked(W.cuda(), mx.MX_ROWWISE)
    fused = f64(mx.grouped_gemm_swiglu(xr, wr, o))
    y = f64(mx.grouped_gemm(mx.MX_FPROP, xr, wr, o))
    unfused = oracle.swiglu(y)
    g, u = y[:, :F], y[:, F:]
    bound = 2.0 ** -8 * (1.1 * np.abs(g) * np.abs(u) + np.abs(oracle.silu(g)) * np.abs(u)) + 2.0 ** -7 * np.abs(unfused)
    assert np.all(np.abs(fused - unfused) <= bound + 1e-30)


def _fused_vs_two_step(counts, K, F, seed):
    """The fused SwiGLU + quantisation epilogue against the two-step path (the
    BF16 output of mx_grouped_gemm_swiglu, then mx_quantize of it with both
    copies and per-expert column segments): every byte of the four buffers,
    unwritten bytes included (both start as the same fill)."""
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    E = len(counts)
    M = int(offs[-1])
    X = workloads.normal_bf16((M, K), seed)
    W = workloads.normal_bf16((E, 2 * F, K), seed + 1, 0.05)
    o = torch.from_numpy(offs).cuda()
    xr, _ = mx.quantize(X.cuda(), mx.MX_ROWWISE)
    wr, _ = mx.quantize_stacked(W.cuda(), mx.MX_ROWWISE)
    cap = int(mx.mx_grouped_padded_rows(offs)) + 128   # room past the last segment, left unwritten
    st = mx.new_status()
    y = mx.grouped_gemm_swiglu(xr, wr, o, status=st)
    fills = []
    for _ in range(2):
        r0, c0 = mx.quantize(y, mx.MX_BOTH, group_offsets=o, col_capacity=cap)
        for t in (r0.data, r0.scale, c0.data, c0.scale):
            t.fill_(0xAB)
        fills.append((r0, c0))
    (r2, c2), (rf, cf) = fills
    mx.quantize(y, mx.MX_BOTH, group_offsets=o, col_capacity=cap, status=st)  # warm the path
    mx.mx_quantize(y.data_ptr(), M, F, y.stride(0), mx.MX_BOTH, r2.data.data_ptr(), r2.scale.data_ptr(),
                   c2.data.data_ptr(), c2.scale.data_ptr(), o.data_ptr(), E, cap, st.data_ptr(),
                   torch.cuda.current_stream().cuda_stream)
    mx.grouped_gemm_swiglu_quantize(xr, wr, o, cap, out=(rf, cf), status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    for name, a, b in (("row data", rf.data, r2.data), ("row scales", rf.scale, r2.scale),
                       ("col data", cf.data, c2.data), ("col scales", cf.scale, c2.scale)):
        if not torch.equal(a, b):
            bad = torch.nonzero(a != b)[:6].tolist()
            raise AssertionError(f"fused SwiGLU quantisation {counts} F={F}: {name} differs at {bad}")
    return y, offs, cap, rf, cf


@pytest.mark.parametrize("counts,F", [([100, 0, 156], 128), ([37, 0, 300, 1, 128], 256), ([0, 0, 129], 384),
                                      ([256], 128), ([5, 127, 128, 0, 0, 1000, 33, 2], 256), ([1], 128),
                                      ([31, 33, 0, 200], 128)])
def test_fused_swiglu_quantisation_equals_two_steps(counts, F):
    y, offs, cap, rf, cf = _fused_vs_two_step(counts, 256, F, 110 + F + len(counts))
    # and the codes are the oracle's quantisation of the SwiGLU output's BF16 values
    yb = f64(y)
    codes, scales = oracle.mx_quantize_rowwise(yb)
    assert np.array_equal(rf.data.cpu().numpy(), codes)
    assert np.array_equal(logical_scales(rf), scales)
    ccodes, cscales, _ = oracle.mx_quantize_colwise_grouped(yb, offs)
    kp = ccodes.shape[1]
    assert np.array_equal(cf.data.cpu().numpy()[:, :kp], ccodes)
    assert np.array_equal(logical_scales(cf)[:, :kp // 32], cscales)


def test_fused_swiglu_quantisation_full_size():
    """The routed experts' gate_up (49152 Zipf-routed rows, 64 experts, K =
    2048, 2F = 2816): the fused epilogue against the two-step path, all bytes."""
    _fused_vs_two_step(list(workloads.moe_counts()), 2048, 1408, 120)
