"""Current-scaling variant recipe (one FP32 scale per tensor or per leading
group, "DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §3.2 and §8.2, on E4M3 data)
on the GPU against the oracle: amax, both copies of the quantiser bit for bit
with their FP32 scales, and the dense and grouped GEMMs within
|out - ref| <= 2^-8 |ref| + 1e-6 S."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import assert_bytes_equal, bits, check_values, f64, u8

pytestmark = pytest.mark.gpu


def f32_bits(v) -> int:
    return int(np.float32(v).view(np.uint32))


def make_case(shape, case, seed):
    g = np.random.Generator(np.random.Philox(seed))
    x = g.standard_normal(shape).astype(np.float32)
    if case == "outliers":
        idx = g.choice(x.size, max(1, x.size // 1000), replace=False)
        x.reshape(-1)[idx] *= 1000.0
    elif case == "nan_inf":
        x.reshape(-1)[g.choice(x.size, 5, replace=False)] = np.nan
        x.reshape(-1)[g.choice(x.size, 3, replace=False)] = np.inf
        x.reshape(-1)[g.choice(x.size, 3, replace=False)] = -np.inf
        x.reshape(-1)[0] = -np.nan
    elif case == "inf":
        x.reshape(-1)[g.choice(x.size, 2, replace=False)] = -np.inf
    elif case == "zeros":
        x[:] = 0.0
        x.reshape(-1)[::7] = -0.0
    elif case == "tiny":
        x = x * np.float32(2.0 ** -128)   # BF16 subnormal range after rounding
    elif case == "negative":
        x = -np.abs(x) * 3.0
    return workloads.to_bf16(x)


def oracle_copy(xb, amax=None):
    f = f64(xb)
    a = oracle.current_amax(f) if amax is None else amax
    s = oracle.current_scale(a)
    return oracle.current_encode(f, s), s, a


CASES = ["normal", "outliers", "nan_inf", "inf", "zeros", "tiny", "negative"]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("shape", [(96, 320), (1056, 544), (128, 7168)])
def test_amax_and_both_copies(shape, case):
    xb = make_case(shape, case, 100 + 10 * CASES.index(case) + shape[0] % 7)
    st = mx.new_status()
    x = xb.cuda()
    amax = mx.current_amax(x, status=st)
    row, col = mx.quantize_current(x, mx.MX_BOTH, amax=amax, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    codes, s, a = oracle_copy(xb)
    got_a = float(amax.cpu()[0])
    assert (np.isnan(a) and np.isnan(got_a)) or f32_bits(got_a) == f32_bits(a), (got_a, a)
    assert f32_bits(float(row.scale.cpu()[0])) == f32_bits(s)
    assert_bytes_equal(u8(row.data), codes, f"{case} row")
    assert_bytes_equal(u8(col.data), np.ascontiguousarray(codes.T), f"{case} col")


def test_given_amax_sets_the_scale():
    """A larger amax (as after a maximum across ranks) sets the scale."""
    xb = workloads.normal_bf16((256, 512), 41)
    big = torch.tensor([300.0], dtype=torch.float32, device="cuda")
    row, col = mx.quantize_current(xb.cuda(), mx.MX_BOTH, amax=big)
    torch.cuda.synchronize()
    codes, s, _ = oracle_copy(xb, amax=300.0)
    assert f32_bits(float(row.scale.cpu()[0])) == f32_bits(s)
    assert_bytes_equal(u8(row.data), codes, "row")
    assert_bytes_equal(u8(col.data), np.ascontiguousarray(codes.T), "col")


def test_stacked_per_expert_scales():
    g = np.random.Generator(np.random.Philox(42))
    w = g.standard_normal((5, 160, 224)).astype(np.float32) * np.array([1, 1e3, 1e-3, 0, 7])[:, None, None].astype(np.float32)
    wb = workloads.to_bf16(w)
    row, col = mx.quantize_current(wb.cuda(), mx.MX_BOTH)
    torch.cuda.synchronize()
    codes, sc, _ = oracle.current_quantize_groups(f64(wb))
    assert [f32_bits(v) for v in row.scale.cpu().numpy()] == [f32_bits(v) for v in sc]
    assert_bytes_equal(u8(row.data), codes, "stacked rows")
    assert_bytes_equal(u8(col.data), np.ascontiguousarray(np.transpose(codes, (0, 2, 1))), "stacked cols")


@pytest.mark.parametrize("counts", [[100, 0, 156, 1, 287], [0, 0, 640], [33] * 12])
def test_grouped_column_copy(counts):
    offs = workloads.offsets_from_counts(counts)
    M = int(offs[-1])
    xb = make_case((M, 320), "outliers", 43 + len(counts))
    o = torch.from_numpy(offs).cuda()
    cap = mx.mx_grouped_padded_rows(offs)
    st = mx.new_status()
    row, col = mx.quantize_current(xb.cuda(), mx.MX_BOTH, group_offsets=o, col_capacity=cap, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    codes, s, _ = oracle_copy(xb)
    assert_bytes_equal(u8(row.data), codes, "row")
    assert_bytes_equal(u8(col.data), oracle.current_transpose_grouped(codes, offs), "grouped col")


def gemm_ref(a_codes, sa, b_codes, sb):
    return oracle.current_gemm_ref(a_codes, sa, b_codes, sb)


@pytest.mark.parametrize("M,N,K,mode", [(M, N, K, mode) for (M, N, K) in
                                        [(256, 384, 512), (992, 1088, 2048), (320, 224, 96), (2048, 2560, 1024)]
                                        for mode in (mx.MX_FPROP, mx.MX_DGRAD, mx.MX_WGRAD)] +
                         [(300, 200, 96, mx.MX_FPROP), (1000, 1100, 2048, mx.MX_FPROP)])
def test_dense_gemm(M, N, K, mode):
    """C = A . B^T for the three modes, each operand quantised with its own
    current scale from BF16 sources (fprop: X [M,K], W [N,K]; dgrad: dY [M,K'],
    W^T; wgrad: the transposed copies)."""
    g = 60 + M % 7 + N % 5
    if mode == mx.MX_FPROP:
        A, B = workloads.normal_bf16((M, K), g), workloads.normal_bf16((N, K), g + 1, 0.02)
        (ar, _), (br, _) = mx.quantize_current(A.cuda(), mx.MX_ROWWISE), mx.quantize_current(B.cuda(), mx.MX_ROWWISE)
        a, b = ar, br
        ca, sa, _ = oracle_copy(A)
        cb, sb, _ = oracle_copy(B)
    elif mode == mx.MX_DGRAD:
        # dX[M, N] = dY[M, K] . W[K, N]: b = W's transposed copy [N, K]
        A, W = workloads.normal_bf16((M, K), g), workloads.normal_bf16((K, N), g + 1, 0.02)
        a, _ = mx.quantize_current(A.cuda(), mx.MX_ROWWISE)
        _, b = mx.quantize_current(W.cuda(), mx.MX_COLWISE)
        ca, sa, _ = oracle_copy(A)
        cw, sb, _ = oracle_copy(W)
        cb = np.ascontiguousarray(cw.T)
    else:
        # dW[M, N] = dY^T . X over K tokens: both transposed copies
        dY, X = workloads.normal_bf16((K, M), g), workloads.normal_bf16((K, N), g + 1)
        _, a = mx.quantize_current(dY.cuda(), mx.MX_COLWISE)
        _, b = mx.quantize_current(X.cuda(), mx.MX_COLWISE)
        cd, sa, _ = oracle_copy(dY)
        cx, sb, _ = oracle_copy(X)
        ca, cb = np.ascontiguousarray(cd.T), np.ascontiguousarray(cx.T)
    st = mx.new_status()
    out = mx.gemm_current(mode, a, b, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    ref, S = gemm_ref(ca, sa, cb, sb)
    check_values(f64(out), ref, S, f"current {M}x{N}x{K} mode {mode}")


@pytest.mark.parametrize("counts", [[300, 0, 129, 1, 700], [64] * 8])
def test_grouped_gemms(counts):
    offs = workloads.offsets_from_counts(counts)
    E, M, H, N = len(counts), int(offs[-1]), 256, 384
    o = torch.from_numpy(offs).cuda()
    cap = mx.mx_grouped_padded_rows(offs)
    X = workloads.normal_bf16((M, H), 70)
    W = workloads.to_bf16(np.random.Generator(np.random.Philox(71)).standard_normal((E, N, H)).astype(np.float32) *
                          np.geomspace(1e-2, 10, E).astype(np.float32)[:, None, None])
    dY = workloads.normal_bf16((M, N), 72)
    st = mx.new_status()
    xr, xc = mx.quantize_current(X.cuda(), mx.MX_BOTH, group_offsets=o, col_capacity=cap, status=st)
    dr, dc = mx.quantize_current(dY.cuda(), mx.MX_BOTH, group_offsets=o, col_capacity=cap, status=st)
    wr, wc = mx.quantize_current(W.cuda(), mx.MX_BOTH, status=st)
    y = mx.grouped_gemm_current(mx.MX_FPROP, xr, wr, o, status=st)
    dx = mx.grouped_gemm_current(mx.MX_DGRAD, dr, wc, o, status=st)
    dw = mx.grouped_gemm_current(mx.MX_WGRAD, dc, xc, o, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    cx, sx, _ = oracle_copy(X)
    cd, sd, _ = oracle_copy(dY)
    cw, sw, _ = oracle.current_quantize_groups(f64(W))
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            assert bool((dw[e] == 0).all())
            continue
        ref, S = gemm_ref(cx[lo:hi], sx, cw[e], sw[e])
        check_values(f64(y[lo:hi]), ref, S, f"current grouped fprop e{e}")
        ref, S = gemm_ref(cd[lo:hi], sd, np.ascontiguousarray(cw[e].T), sw[e])
        check_values(f64(dx[lo:hi]), ref, S, f"current grouped dgrad e{e}")
        ref, S = gemm_ref(np.ascontiguousarray(cd[lo:hi].T), sd, np.ascontiguousarray(cx[lo:hi].T), sx)
        check_values(f64(dw[e]), ref, S, f"current grouped wgrad e{e}")


def test_dense_ffn_full_size():
    """The dense FFN up-projection (M=8192, K=2048, N=10944) under current
    scaling: every code of X, W and dY against the oracle (run in row slabs
    over the host cores) and sampled entries of fprop, dgrad and wgrad."""
    from tests import oracle_pool
    d = workloads.dense_ffn()
    q, ref_codes, ref_s = {}, {}, {}
    for k in ("X", "W", "dY"):
        q[k] = mx.quantize_current(d[k].cuda(), mx.MX_BOTH)
        a = oracle.current_amax(f64(d[k]))
        ref_s[k] = oracle.current_scale(a)
        ref_codes[k] = oracle_pool.current_codes(bits(d[k]), ref_s[k])
    torch.cuda.synchronize()
    for k in ("X", "W", "dY"):
        assert f32_bits(float(q[k][0].scale.cpu()[0])) == f32_bits(ref_s[k])
        assert_bytes_equal(u8(q[k][0].data), ref_codes[k], k + " row")
        assert_bytes_equal(u8(q[k][1].data), np.ascontiguousarray(ref_codes[k].T), k + " col")
    (xr, xc), (wr, wc), (dr, dc) = q["X"], q["W"], q["dY"]
    outs = {mx.MX_FPROP: mx.gemm_current(mx.MX_FPROP, xr, wr), mx.MX_DGRAD: mx.gemm_current(mx.MX_DGRAD, dr, wc),
            mx.MX_WGRAD: mx.gemm_current(mx.MX_WGRAD, dc, xc)}
    # dgrad and wgrad in one launch, as the bench step runs them: the same bits
    st = mx.new_status()
    dx, dw = mx.gemm_current_multi([(mx.MX_DGRAD, dr, wc), (mx.MX_WGRAD, dc, xc)], status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    assert torch.equal(dx.view(torch.int16), outs[mx.MX_DGRAD].view(torch.int16))
    assert torch.equal(dw.view(torch.int16), outs[mx.MX_WGRAD].view(torch.int16))
    g = np.random.Generator(np.random.Philox(80))
    cX, cW, cD = ref_codes["X"], ref_codes["W"], ref_codes["dY"]
    for mode, (A, sa, B, sb) in {mx.MX_FPROP: (cX, ref_s["X"], cW, ref_s["W"]),
                                 mx.MX_DGRAD: (cD, ref_s["dY"], cW.T, ref_s["W"]),
                                 mx.MX_WGRAD: (cD.T, ref_s["dY"], cX.T, ref_s["X"])}.items():
        out = outs[mode]
        ii = g.integers(0, out.shape[0], 2048)
        jj = g.integers(0, out.shape[1], 2048)
        Ad = oracle.current_dequantize(np.ascontiguousarray(A[ii]), sa)
        Bd = oracle.current_dequantize(np.ascontiguousarray(B[jj]), sb)
        ref, S = np.sum(Ad * Bd, axis=1), np.sum(np.abs(Ad * Bd), axis=1)
        check_values(f64(out[torch.from_numpy(ii), torch.from_numpy(jj)]), ref, S, f"current dense FFN mode {mode}")


def test_gemm_current_multi_matches_single_calls():
    """Several tensor-scaled GEMMs in one launch (mixed modes and shapes, one
    of them small enough that its tiles alone would not fill the GPU): every
    output equals the mx_gemm_current result bit for bit, and the oracle's
    within the bound."""
    cases = [(mx.MX_FPROP, 992, 1088, 2048), (mx.MX_DGRAD, 2048, 2560, 1024), (mx.MX_WGRAD, 320, 224, 96)]
    probs, refs = [], []
    for i, (mode, M, N, K) in enumerate(cases):
        A = workloads.normal_bf16((M, K) if mode != mx.MX_WGRAD else (K, M), 70 + i)
        B = workloads.normal_bf16((N, K) if mode == mx.MX_FPROP else (K, N), 80 + i, 0.02)
        ra, ca_ = mx.quantize_current(A.cuda(), mx.MX_BOTH)
        rb, cb_ = mx.quantize_current(B.cuda(), mx.MX_BOTH)
        oa, sa, _ = oracle_copy(A)
        ob, sb, _ = oracle_copy(B)
        if mode == mx.MX_FPROP:
            a, b, ra_c, rb_c = ra, rb, oa, ob
        elif mode == mx.MX_DGRAD:
            a, b, ra_c, rb_c = ra, cb_, oa, np.ascontiguousarray(ob.T)
        else:
            a, b, ra_c, rb_c = ca_, cb_, np.ascontiguousarray(oa.T), np.ascontiguousarray(ob.T)
        probs.append((mode, a, b))
        refs.append((ra_c, sa, rb_c, sb))
    st = mx.new_status()
    outs = mx.gemm_current_multi(probs, status=st)
    singles = [mx.gemm_current(mode, a, b) for mode, a, b in probs]
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    for (mode, _, _), out, one, (ca, sa, cb, sb) in zip(probs, outs, singles, refs):
        assert torch.equal(out.view(torch.int16), one.view(torch.int16))
        ref, S = gemm_ref(ca, sa, cb, sb)
        check_values(f64(out), ref, S, f"current multi mode {mode}")


def test_quotient_exhaustive_against_ieee_division():
    """Every finite BF16 x divided by the scale of every positive finite BF16
    amax: the quantiser's codes equal E4M3 of the IEEE FP32 quotient (torch's
    division on the GPU, then torch's E4M3 conversion, which the oracle pins
    check against the E4M3 rounding rule), saturated at +-448. This covers the
    reciprocal-and-correction division the kernel uses for the quotient."""
    pats = torch.arange(0, 1 << 16, dtype=torch.int32)
    finite = (pats & 0x7F80) != 0x7F80
    xbits = pats[finite].to(torch.int16)                      # 65280 finite patterns (both signs)
    assert xbits.numel() == 510 * 128
    x = xbits.view(torch.bfloat16).reshape(510, 128).cuda()
    amax_bits = torch.arange(1, 0x7F80, dtype=torch.int32)     # every positive finite BF16 amax
    amaxes = (amax_bits << 16).view(torch.float32).cuda()
    E = 480
    xs = x.unsqueeze(0).expand(E, 510, 128).contiguous()
    xf = x.float()
    for start in range(0, amaxes.numel(), E):
        am = amaxes[start:start + E]
        n = am.numel()
        row, _ = mx.quantize_current(xs[:n], mx.MX_ROWWISE, amax=am)
        # IEEE FP32 division, as the scale rule (a tensor divisor: torch turns a
        # scalar divisor into a multiplication by its reciprocal)
        s = am / torch.full_like(am, 448.0)
        assert torch.equal(row.scale.view(torch.int32), s.view(torch.int32))
        q = (xf.unsqueeze(0) / s.view(n, 1, 1)).clamp(-448.0, 448.0)
        ref = q.to(torch.float8_e4m3fn).view(torch.uint8)
        got = row.data.view(n, 510, 128)
        if not torch.equal(got, ref):
            bad = (got != ref).nonzero()[:5].tolist()
            raise AssertionError(f"amax block {start}: first mismatches {bad}")
