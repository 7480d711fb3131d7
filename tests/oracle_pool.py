"""Full-tensor oracle quantisation for the parity tests, spread over the host
cores.

The oracle is plain numpy on one core; the workload tensors reach a few
hundred million elements, so the tests cut each one into independent pieces
(row slabs for the row copy, column slabs for the column copies, experts for
stacked weights), run the unchanged oracle functions on the pieces in a
process pool and put the results back together. Blocks never straddle a
piece: row slabs keep whole rows (1x32 blocks lie along rows), column slabs
keep whole columns (32x1 blocks lie down columns). The pool uses the spawn
start method, so no worker is forked from a process that holds a CUDA
context.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

_POOL = None


def pool() -> cf.ProcessPoolExecutor:
    global _POOL
    if _POOL is None:
        n = max(1, min(16, os.cpu_count() or 1))
        _POOL = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
    return _POOL


def _rows_task(bits):
    import oracle
    return oracle.mx_quantize_rowwise(oracle.bf16_bits_to_float64(bits))


def _cols_task(bits):
    import oracle
    return oracle.mx_quantize_colwise(oracle.bf16_bits_to_float64(bits))


def _cols_grouped_task(bits, offsets):
    import oracle
    d, s, _ = oracle.mx_quantize_colwise_grouped(oracle.bf16_bits_to_float64(bits), offsets)
    return d, s


def _slabs(n: int, step: int):
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def rowwise(bits: np.ndarray, target_elems: int = 1 << 22):
    """oracle.mx_quantize_rowwise of BF16 bits [R, C]: (data [R, C], scales [R, C/32])."""
    R, C = bits.shape
    step = max(1, target_elems // max(C, 1))
    parts = list(pool().map(_rows_task, [bits[a:b] for a, b in _slabs(R, step)]))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def colwise(bits: np.ndarray, target_elems: int = 1 << 22):
    """oracle.mx_quantize_colwise of BF16 bits [R, C]: (data [C, R], scales [C, R/32])."""
    R, C = bits.shape
    step = max(1, target_elems // max(R, 1))
    parts = list(pool().map(_cols_task, [np.ascontiguousarray(bits[:, a:b]) for a, b in _slabs(C, step)]))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def colwise_grouped(bits: np.ndarray, offsets, target_elems: int = 1 << 22):
    """oracle.mx_quantize_colwise_grouped of BF16 bits [M, D] with group offsets:
    (data [D, padded], scales [D, padded/32])."""
    M, D = bits.shape
    step = max(1, target_elems // max(M, 1))
    offs = np.asarray(offsets, dtype=np.int64)
    parts = list(pool().map(_cols_grouped_task, [np.ascontiguousarray(bits[:, a:b]) for a, b in _slabs(D, step)],
                            [offs] * len(_slabs(D, step))))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def stacked(bits: np.ndarray):
    """Row and column copies of every matrix of stacked BF16 bits [E, N, K]:
    (row data [E, N, K], row scales [E, N, K/32], col data [E, K, N], col scales [E, K, N/32])."""
    E = bits.shape[0]
    rows = list(pool().map(_rows_task, [bits[e] for e in range(E)]))
    cols = list(pool().map(_cols_task, [bits[e] for e in range(E)]))
    return (np.stack([r[0] for r in rows]), np.stack([r[1] for r in rows]),
            np.stack([c[0] for c in cols]), np.stack([c[1] for c in cols]))


def _current_task(bits, scale):
    import oracle
    return oracle.current_encode(oracle.bf16_bits_to_float64(bits), scale)


def current_codes(bits: np.ndarray, scale, target_elems: int = 1 << 22):
    """oracle.current_encode of BF16 bits [R, C] with one scale (element-wise,
    so any row slab works): codes [R, C]."""
    R, C = bits.shape
    step = max(1, target_elems // max(C, 1))
    sl = _slabs(R, step)
    return np.concatenate(list(pool().map(_current_task, [bits[a:b] for a, b in sl], [scale] * len(sl))))
