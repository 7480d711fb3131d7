"""The slab-parallel oracle runs used by the full-size parity tests give
exactly the whole-tensor oracle results: slabs keep whole rows (row copy) or
whole columns (column copies), so no 1x32 or 32x1 block is cut."""
import numpy as np

import oracle
import workloads
from tests import oracle_pool
from tests.gpu_util import bits


def test_slabs_equal_whole_tensor():
    x = workloads.normal_bf16((96, 320), 5)
    b = bits(x)
    f = oracle.bf16_bits_to_float64(b)
    # tiny slabs force many pieces, including a ragged last one
    for got, want in ((oracle_pool.rowwise(b, target_elems=7 * 320), oracle.mx_quantize_rowwise(f)),
                      (oracle_pool.colwise(b, target_elems=96 * 3), oracle.mx_quantize_colwise(f))):
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
    offs = np.array([0, 5, 5, 40, 96], dtype=np.int64)
    got = oracle_pool.colwise_grouped(b, offs, target_elems=96 * 7)
    want = oracle.mx_quantize_colwise_grouped(f, offs)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
    w = workloads.normal_bf16((3, 64, 96), 6)
    rd, rs, cd, cs = oracle_pool.stacked(bits(w))
    for e in range(3):
        fe = oracle.bf16_bits_to_float64(bits(w[e]))
        d, s = oracle.mx_quantize_rowwise(fe)
        assert np.array_equal(rd[e], d) and np.array_equal(rs[e], s)
        d, s = oracle.mx_quantize_colwise(fe)
        assert np.array_equal(cd[e], d) and np.array_equal(cs[e], s)
