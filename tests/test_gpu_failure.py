"""Failure reporting on the GPU without faulting it: a bounded wait on a barrier
that nothing signals gives up after its bound and reports MX_ERR_TIMEOUT
through the device status word, and the context stays usable afterwards."""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import f64

pytestmark = pytest.mark.gpu

MX_ERR_TIMEOUT = 6
assert mx.STATUS_NAMES[MX_ERR_TIMEOUT] == "MX_ERR_TIMEOUT"


def test_bounded_wait_times_out_and_reports():
    st = mx.new_status()
    t0 = time.perf_counter()
    mx.mx_selftest_wait_timeout(20_000_000, st.data_ptr(), None)   # 20 ms bound
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert mx.read_status(st) == MX_ERR_TIMEOUT
    assert 0.015 <= elapsed < 2.0, elapsed


def test_context_usable_after_timeout():
    st = mx.new_status()
    mx.mx_selftest_wait_timeout(5_000_000, st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == MX_ERR_TIMEOUT
    # a GEMM right after, checked against the oracle
    X = workloads.normal_bf16((256, 512), 5100)
    W = workloads.normal_bf16((384, 512), 5101, 0.02)
    st2 = mx.new_status()
    xr, _ = mx.quantize(X.cuda(), mx.MX_ROWWISE, status=st2)
    wr, _ = mx.quantize(W.cuda(), mx.MX_ROWWISE, status=st2)
    y = mx.gemm(mx.MX_FPROP, xr, wr, status=st2)
    torch.cuda.synchronize()
    assert mx.read_status(st2) == 0
    ref, S = oracle.mx_gemm_ref(*oracle.mx_quantize_rowwise(f64(X)), *oracle.mx_quantize_rowwise(f64(W)))
    assert oracle.within_tolerance(f64(y), ref, S).all()


def test_two_timeouts_in_one_status_word_stay_timeout():
    st = mx.new_status()
    for _ in range(2):
        mx.mx_selftest_wait_timeout(2_000_000, st.data_ptr(), None)
    torch.cuda.synchronize()
    assert mx.read_status(st) == MX_ERR_TIMEOUT


def test_selftest_rejects_bad_arguments():
    st = mx.new_status()
    with pytest.raises(mx.MXError):
        mx.mx_selftest_wait_timeout(0, st.data_ptr(), None)
    with pytest.raises(mx.MXError):
        mx.mx_selftest_wait_timeout(1_000_000, None, None)
