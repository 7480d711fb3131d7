"""Plant plausible mistakes in a private copy of the oracle (on the CPU) and
check that at least one pin catches each of them. This shows the pins would
notice a dropped term, a wrong sign, index, rounding rule or operand order."""
import importlib.util
import os

import numpy as np
import pytest

from tests import pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "mx_oracle.py")


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("mx_oracle_mutant", ORACLE_SRC)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def m_scale_off_by_one(O):
    orig = O.mx_scale_exponent
    O.mx_scale_exponent = lambda a: np.clip(orig(a) + 1, -127, 127)


def m_scale_ceil(O):
    def f(amax):
        a = np.asarray(amax, dtype=np.float64)
        safe = np.where(np.isfinite(a) & (a > 0), a, 1.0)
        x = np.ceil(np.log2(safe)).astype(np.int64) - 8
        return np.clip(np.where(a > 0, x, -127), -127, 127)
    O.mx_scale_exponent = f


def m_zero_block_scale_one(O):
    orig = O.mx_scale_exponent
    O.mx_scale_exponent = lambda a: np.where(np.asarray(a) == 0, 0, orig(a))


def m_ties_away(O):
    vals = O._POS_VALUES
    def enc(x):
        x = np.asarray(x, dtype=np.float64)
        sign = np.signbit(x).astype(np.int64)
        a = np.minimum(np.abs(x), 448.0)
        hi = np.clip(np.searchsorted(vals, a), 0, len(vals) - 1)
        lo = np.maximum(hi - 1, 0)
        mid = (vals[lo] + vals[hi]) / 2
        idx = np.where(a >= mid, hi, lo)
        return (idx | (sign << 7)).astype(np.uint8)
    O.e4m3_encode = enc


def m_truncate(O):
    vals = O._POS_VALUES
    def enc(x):
        x = np.asarray(x, dtype=np.float64)
        sign = np.signbit(x).astype(np.int64)
        a = np.minimum(np.abs(x), 448.0)
        idx = np.searchsorted(vals, a, side="right") - 1
        return (idx | (sign << 7)).astype(np.uint8)
    O.e4m3_encode = enc


def m_no_saturation(O):
    orig = O.e4m3_encode
    def enc(x):
        c = orig(x)
        return np.where(np.abs(np.asarray(x)) > 448, 0x7F, c).astype(np.uint8)
    O.e4m3_encode = enc


def m_drop_sign(O):
    orig = O.e4m3_encode
    O.e4m3_encode = lambda x: orig(np.abs(np.asarray(x, dtype=np.float64)))


def m_decode_bias8(O):
    orig = O.e4m3_decode
    O.e4m3_decode = lambda c: orig(c) / 2.0


def m_decode_subnormal_hidden_one(O):
    def dec(codes):
        c = np.asarray(codes).astype(np.int64)
        s, e, m = (c >> 7) & 1, (c >> 3) & 0xF, c & 7
        mag = (1.0 + m / 8.0) * np.exp2(np.where(e == 0, 1, e).astype(np.float64) - 7)
        v = np.where(s == 1, -mag, mag)
        return np.where((e == 15) & (m == 7), np.nan, v)
    O.e4m3_decode = dec
    O._POS_VALUES = dec(O._POS_CODES)


def m_colwise_not_transposed(O):
    def col(x):
        x = np.asarray(x, dtype=np.float64)
        d, s = O.mx_quantize_rowwise(x.T)
        return d.T.copy().reshape(x.shape[1], x.shape[0]), s
    O.mx_quantize_colwise = col


def m_gemm_transposed(O):
    """B's K-major rows read as if B were stored [K, N] (reshape, not transpose)."""
    def g(ac, asc, bc, bsc):
        A = O.mx_dequantize(ac, asc)
        B = O.mx_dequantize(bc, bsc)
        Bw = B.reshape(B.shape[1], B.shape[0])
        return A @ Bw, np.abs(A) @ np.abs(Bw)
    O.mx_gemm_ref = g


def m_gemm_drop_b_scale(O):
    def g(ac, asc, bc, bsc):
        A = O.mx_dequantize(ac, asc)
        B = O.e4m3_decode(bc)
        return A @ B.T, np.abs(A) @ np.abs(B).T
    O.mx_gemm_ref = g


def m_dequant_scale_sign(O):
    def deq(codes, sc):
        v = O.e4m3_decode(codes)
        s = np.exp2(-(np.asarray(sc).astype(np.float64) - 127))
        return v * np.repeat(s, 32, axis=-1)[..., : v.shape[-1]]
    O.mx_dequantize = deq


def m_swizzle_swapped(O):
    def off(r, k, kbp):
        r = np.asarray(r, dtype=np.int64); k = np.asarray(k, dtype=np.int64)
        atom = (r // 128) * (kbp // 4) + k // 4
        return atom * 512 + ((r // 32) % 4) * 128 + (r % 32) * 4 + (k % 4)
    O.mx_scale_byte_offset = off


def m_group_blocks_not_restarting(O):
    def gq(x, offsets):
        x = np.asarray(x, dtype=np.float64)
        M, D = x.shape
        o = np.asarray(offsets, dtype=np.int64)
        poff = O.mx_padded_offsets(o)
        Mp = (M + 31) // 32 * 32
        xp = np.zeros((Mp, D)); xp[:M] = x
        d_all, s_all = O.mx_quantize_colwise(xp)        # blocks anchored at row 0
        Kp = int(poff[-1])
        data = np.zeros((D, Kp), np.uint8); scale = np.zeros((D, Kp // 32), np.uint8)
        for e in range(len(o) - 1):
            m = int(o[e + 1] - o[e])
            if m == 0:
                continue
            data[:, poff[e]:poff[e] + m] = d_all[:, o[e]:o[e + 1]]
            kb0 = o[e] // 32
            nb = (m + 31) // 32
            scale[:, poff[e] // 32:poff[e] // 32 + nb] = s_all[:, kb0:kb0 + nb]
        return data, scale, poff
    O.mx_quantize_colwise_grouped = gq


def m_group_pad_64(O):
    def po(offsets):
        m = O.mx_group_sizes(offsets)
        pad = (m + 63) // 64 * 64
        return np.concatenate([[0], np.cumsum(pad)]).astype(np.int64)
    O.mx_padded_offsets = po


def m_bf16_truncate(O):
    def r(x):
        x = np.asarray(x, dtype=np.float64)
        b = (x.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
        return b.astype(np.float64)
    O.bf16_round = r


def m_input_bf16_prerounding(O):
    orig = O.mx_quantize_blocks
    O.mx_quantize_blocks = lambda blocks: orig(O.bf16_round(np.asarray(blocks, dtype=np.float64)))


def m_swiglu_halves_swapped(O):
    def sw(y):
        y = np.asarray(y, dtype=np.float64)
        F = y.shape[-1] // 2
        return O.silu(y[..., F:]) * y[..., :F]
    O.swiglu = sw


def m_silu_sign(O):
    O.silu = lambda x: np.asarray(x, dtype=np.float64) / (1.0 + np.exp(np.asarray(x, dtype=np.float64)))


def m_blockwise_scale_inverted(O):
    O.blockwise_scale = lambda amax: np.where(np.asarray(amax) > 0, np.asarray(amax, dtype=np.float32) / np.float32(448.0),
                                              np.float32(1.0)).astype(np.float32)


def m_blockwise_promote_multiplies(O):
    orig = O.gemm_blockwise_ref
    O.gemm_blockwise_ref = lambda a, sa, b, sb: orig(a, 1.0 / np.asarray(sa, dtype=np.float64), b,
                                                     1.0 / np.asarray(sb, dtype=np.float64))


def m_blockwise_weight_rows(O):
    def q(w):
        c, s = O.quantize_1x128(w)
        nb = (w.shape[0] + 127) // 128
        return c, s[::128][:nb]
    O.quantize_128x128 = q


def m_current_scale_inverted(O):
    orig = O.current_scale
    O.current_scale = lambda amax, fmt=448.0: np.float32(1.0) / orig(amax, fmt)


def m_current_multiplies(O):
    O.current_encode = lambda x, s: O.e4m3_encode((np.asarray(x, dtype=np.float32) * np.float32(s)).astype(np.float64))


def m_current_exact_quotient(O):
    O.current_encode = lambda x, s: O.e4m3_encode(np.asarray(x, dtype=np.float64) / np.float64(np.float32(s)))


def m_current_no_validity(O):
    def sc(amax, fmt=448.0):
        with np.errstate(all="ignore"):
            return np.float32(np.float32(amax) / np.float32(fmt))
    O.current_scale = sc


def m_current_groups_share_amax(O):
    def q(w, fmt=448.0):
        w = np.asarray(w, dtype=np.float64)
        amax = O.current_amax(w)
        s = O.current_scale(amax, fmt)
        E = w.shape[0]
        return O.current_encode(w, s), np.full(E, s, dtype=np.float32), np.full(E, amax)
    O.current_quantize_groups = q


def m_current_transpose_unpadded(O):
    def t(codes, offsets):
        return np.ascontiguousarray(np.asarray(codes, dtype=np.uint8).T)
    O.current_transpose_grouped = t


def m_tolerance_loose(O):
    O.within_tolerance = lambda out, ref, S: np.abs(np.asarray(out) - ref) <= 2.0 ** -5 * np.abs(ref) + 1e-6 * S


MUTANTS = [m_scale_off_by_one, m_scale_ceil, m_zero_block_scale_one, m_ties_away, m_truncate,
           m_no_saturation, m_drop_sign, m_decode_bias8, m_decode_subnormal_hidden_one,
           m_colwise_not_transposed, m_gemm_transposed, m_gemm_drop_b_scale, m_dequant_scale_sign,
           m_swizzle_swapped, m_group_blocks_not_restarting, m_group_pad_64, m_bf16_truncate,
           m_tolerance_loose, m_input_bf16_prerounding, m_swiglu_halves_swapped, m_silu_sign,
           m_blockwise_scale_inverted, m_blockwise_promote_multiplies, m_blockwise_weight_rows,
           m_current_scale_inverted, m_current_multiplies, m_current_exact_quotient, m_current_no_validity,
           m_current_groups_share_amax, m_current_transpose_unpadded]


def _caught(O):
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(O)
        except (AssertionError, ValueError, IndexError):
            return pin.__name__
    return None


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_mutant_is_caught(mutant):
    O = fresh_oracle()
    mutant(O)
    assert _caught(O) is not None, f"no pin catches {mutant.__name__}"


def test_unmutated_copy_passes():
    assert _caught(fresh_oracle()) is None
