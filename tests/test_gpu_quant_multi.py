"""Several unrelated BF16 matrices quantised in one mx_quantize_multi launch:
every matrix's row and column copies equal the oracle's bit for bit, exactly
as a separate mx_quantize of that matrix would give."""
import numpy as np
import pytest
import torch

import workloads
import mxfp8_block_scaled_gb300 as mx
from tests.gpu_util import check_col_copy, check_row_copy

pytestmark = pytest.mark.gpu


def matrix(R, C, seed):
    g = np.random.Generator(np.random.Philox(seed))
    x = g.standard_normal((R, C)) * np.exp2(g.integers(-6, 6, (R, 1))) * np.exp2(g.integers(-3, 3, (1, C)))
    if R * C:
        x.reshape(-1)[g.choice(R * C, size=max(1, R * C // 500), replace=False)] *= 1000
    return workloads.to_bf16(x)


SETS = {
    "x_and_w": [(512, 2048), (1344, 2048)],
    "ragged_tiles": [(96, 160), (416, 96), (160, 576), (32, 32)],
    "with_empty": [(0, 64), (256, 512), (64, 0), (128, 128)],
    "eight": [(32 * (i + 1), 64 * (i % 3 + 1)) for i in range(8)],
}


@pytest.mark.parametrize("name", sorted(SETS))
@pytest.mark.parametrize("axis", [mx.MX_ROWWISE, mx.MX_COLWISE, mx.MX_BOTH])
def test_multi_matches_oracle(name, axis):
    xs = [matrix(R, C, 7000 + 31 * i + R + C) for i, (R, C) in enumerate(SETS[name])]
    st = mx.new_status()
    outs = mx.quantize_multi([x.cuda() for x in xs], axis, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    for i, (x, (row, col)) in enumerate(zip(xs, outs)):
        if x.numel() == 0:
            continue
        if axis & mx.MX_ROWWISE:
            check_row_copy(x, row, f"{name}[{i}] row")
        if axis & mx.MX_COLWISE:
            check_col_copy(x, col, f"{name}[{i}] col")


def test_multi_strided_inputs_and_single_launch_equivalence():
    """Pitched inputs (ldx > cols) and a result identical to one mx_quantize
    per matrix."""
    big = [matrix(256, 1024, 11).cuda(), matrix(384, 320, 12).cuda()]
    views = [big[0][:, :512], big[1][:, 64:320]]
    st = mx.new_status()
    outs = mx.quantize_multi(views, mx.MX_BOTH, status=st)
    torch.cuda.synchronize()
    assert mx.read_status(st) == 0
    for v, (row, col) in zip(views, outs):
        r1, c1 = mx.quantize(v, mx.MX_BOTH)
        torch.cuda.synchronize()
        assert torch.equal(row.data, r1.data) and torch.equal(row.scale, r1.scale)
        assert torch.equal(col.data, c1.data) and torch.equal(col.scale, c1.scale)
        check_row_copy(v.cpu(), row, "strided row")
        check_col_copy(v.cpu(), col, "strided col")
