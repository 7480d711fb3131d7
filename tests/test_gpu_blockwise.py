"""Variant recipe on the GPU: DeepSeek-V3 blockwise FP8 (1 x 128 activation and
128 x 128 weight blocks with FP32 multipliers). Quantisers bit for bit against
the oracle (codes and FP32 multipliers); the GEMM within the acceptance bound
against the oracle's per-block promotion in float64."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import assert_bytes_equal, f64, u8

pytestmark = pytest.mark.gpu


def quant(x, block):
    st = mx.new_status()
    q = mx.quantize_fp8_blockwise(x.cuda(), block, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    return q


def check_1x128(x, q, what):
    codes, s = oracle.quantize_1x128(f64(x))
    assert_bytes_equal(u8(q.data), codes, what + " codes")
    got = q.scale.cpu().numpy()
    assert np.array_equal(got, s.T), what + " multipliers"


def check_128x128(w, q, what):
    codes, s = oracle.quantize_128x128(f64(w))
    assert_bytes_equal(u8(q.data), codes, what + " codes")
    assert np.array_equal(q.scale.cpu().numpy(), s), what + " multipliers"


@pytest.mark.parametrize("R,C", [(1, 128), (200, 384), (1024, 2048)])
def test_quant_1x128(R, C):
    x = workloads.normal_bf16((R, C), 4000 + R)
    x[0, :128] = 0.0                                     # an all-zero block
    if R > 3:
        x[3, 130] = 5000.0                               # an outlier in one block only
    check_1x128(x, quant(x, 1), f"1x128 {R}x{C}")


def test_quant_1x128_dense_ffn_activation():
    x = workloads.dense_ffn()["X"][:2048]                # 1% outlier channels x50
    check_1x128(x, quant(x, 1), "1x128 FFN activation")


@pytest.mark.parametrize("R,C", [(128, 128), (300, 256), (10944, 2048)])
def test_quant_128x128(R, C):
    w = workloads.normal_bf16((R, C), 4100 + R, 0.02)
    w[R - 1, C - 1] = 3.0                                # an outlier in the last (short) block
    check_128x128(w, quant(w, 128), f"128x128 {R}x{C}")


def test_quant_input_pitch():
    wide = workloads.normal_bf16((256, 520), 4200)
    x = wide[:, :384]
    st = mx.new_status()
    q = mx.quantize_fp8_blockwise(wide.cuda()[:, :384], 1, status=st)
    torch.cuda.synchronize()
    check_1x128(x, q, "1x128 pitch")


def gemm_case(M, N, K, seed, rows=None):
    x = workloads.normal_bf16((M, K), seed)
    w = workloads.normal_bf16((N, K), seed + 1, 0.02)
    qa, qb = quant(x, 1), quant(w, 128)
    st = mx.new_status()
    out = mx.gemm_fp8_blockwise(qa, qb, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    ac, asc = oracle.quantize_1x128(f64(x))
    bc, bsc = oracle.quantize_128x128(f64(w))
    got = f64(out)
    if rows is not None:
        ac, asc, got = ac[rows], asc[rows], got[rows]
    ref, S = oracle.gemm_blockwise_ref(ac, asc, bc, bsc)
    ok = oracle.within_tolerance(got, ref, S)
    if not ok.all():
        bad = np.argwhere(~ok)[:8]
        raise AssertionError(f"blockwise gemm {M}x{N}x{K}: {int((~ok).sum())} of {ok.size} outside; first "
                             f"{[(tuple(i), got[tuple(i)], ref[tuple(i)]) for i in bad]}")


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (200, 300, 384), (1024, 2048, 2048), (640, 384, 4096)])
def test_gemm_blockwise(M, N, K):
    gemm_case(M, N, K, 4300 + M + N)


def test_gemm_blockwise_full_size_sampled():
    """The dense FFN up-projection fprop (8192 x 10944 x 2048) with the
    blockwise recipe; 64 sampled rows checked against the oracle in full."""
    rows = np.random.Generator(np.random.Philox(4400)).choice(8192, size=64, replace=False)
    gemm_case(8192, 10944, 2048, 4400, rows=np.sort(rows))


def test_gemm_blockwise_repeatable():
    x = workloads.normal_bf16((512, 1024), 4500)
    w = workloads.normal_bf16((384, 1024), 4501, 0.02)
    qa, qb = quant(x, 1), quant(w, 128)
    assert torch.equal(mx.gemm_fp8_blockwise(qa, qb), mx.gemm_fp8_blockwise(qa, qb))
