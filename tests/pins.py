"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` takes an oracle-like module ``O`` and raises AssertionError if
``O`` disagrees with a printed value, a closed form, a library routine, an
exact brute-force result or an invariant. ``test_oracle_pins`` runs them on
the real oracle; ``test_oracle_mutations`` shows that plausible mistakes
planted in a copy of the oracle fail at least one of them.
"""

from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fmt_printed_values.txt")


def read_golden():
    rows = []
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, inp, exp = line.split()[:3]
            rows.append((kind, inp, exp))
    return rows


def _close_to_printed(value: float, printed: str) -> bool:
    """True if value rounds to the printed digits (the page prints 4-5 digits)."""
    if printed == "nan":
        return math.isnan(value)
    p = float(printed)
    digits = len(printed.split("e")[0].replace(".", "").replace("-", "").lstrip("0"))
    return abs(value - p) <= 0.5 * 10 ** (math.floor(math.log10(abs(p))) - digits + 1) * 1.0001


# ---------------------------------------------------------------------------
# Formats
# ---------------------------------------------------------------------------

def pin_printed_values(O):
    """Values printed on the numerics page (golden fixture)."""
    for kind, inp, exp in read_golden():
        if kind == "e4m3_code":
            v = float(O.e4m3_decode(np.array([int(inp, 16)]))[0])
            assert _close_to_printed(v, exp), (inp, v, exp)
            if exp != "nan":
                assert v == float(exp), (inp, v, exp)
        elif kind == "bf16_code":
            v = float(O.bf16_bits_to_float64(np.array([int(inp, 16)]))[0])
            assert _close_to_printed(v, exp), (inp, v, exp)
        elif kind == "bf16_round":
            v = float(O.bf16_round(np.array([float(inp)]))[0])
            assert v == float(exp), (inp, v, exp)
        elif kind == "e4m3_table":
            vals = O.e4m3_decode(np.arange(256))
            pos = vals[np.isfinite(vals) & (vals > 0)]
            got = {"max": pos.max(), "min_normal": 2.0 ** -6, "min_sub": pos.min(),
                   "eps": float(O.e4m3_decode(np.array([0x39]))[0] - O.e4m3_decode(np.array([0x38]))[0])}
            if inp == "min_normal":
                # smallest value whose exponent field is non-zero
                codes = np.arange(1, 0x7F)
                normal = codes[((codes >> 3) & 0xF) > 0]
                got["min_normal"] = float(O.e4m3_decode(normal).min())
            assert _close_to_printed(float(got[inp]), exp), (inp, got[inp], exp)


def pin_e4m3_closed_forms(O):
    """[FMT] §二.1 closed forms with E=4, M=3 (bias 7), and the E4M3 exception
    of §二.2: the top binade is not reserved, S.1111.110 = 1.75 * 2**8."""
    E, M = 4, 3
    d = lambda c: float(O.e4m3_decode(np.array([c]))[0])
    assert d(0x08) == 2.0 ** (2 - 2 ** (E - 1))              # min normal 2**-6
    assert d(0x01) == 2.0 ** (2 - 2 ** (E - 1) - M)          # min subnormal 2**-9
    assert d(0x39) - d(0x38) == 2.0 ** -M and d(0x38) == 1.0  # eps at 1.0
    assert d(0x7E) == 1.75 * 2.0 ** 8
    assert d(0x77) == 1.875 * 2.0 ** 7                        # IEEE-style max would be 240
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    assert d(0x80) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0
    assert d(0xFE) == -448.0
    # every code: value = sign * 2**(e-7) * (1 + m/8), or 2**-6 * m/8 when e == 0
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        ref = (Fraction(m, 8) * Fraction(1, 64)) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        assert Fraction(d(c)) == (-ref if s else ref), c


def pin_e4m3_census(O):
    """256 codes - 2 NaN codes = 254 finite codes, 253 distinct values (+0 = -0);
    non-negative codes 0x00..0x7E are strictly increasing in value."""
    v = O.e4m3_decode(np.arange(256))
    fin = v[np.isfinite(v)]
    assert fin.size == 254 and np.unique(fin).size == 253
    pos = O.e4m3_decode(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)


def pin_e4m3_roundtrip_and_ties(O):
    """Every finite value encodes to its own code; every midpoint between
    neighbours goes to the even code; just off a midpoint goes to the nearer."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    vals = O.e4m3_decode(codes)
    assert np.array_equal(O.e4m3_encode(vals), codes.astype(np.uint8))
    pos = O.e4m3_decode(np.arange(0x7F))
    mids = (pos[:-1] + pos[1:]) / 2
    enc = O.e4m3_encode(mids).astype(np.int64)
    lo, hi = np.arange(0x7E), np.arange(1, 0x7F)
    assert np.array_equal(enc, np.where(lo % 2 == 0, lo, hi))
    assert np.array_equal(O.e4m3_encode(-mids).astype(np.int64), np.where(lo % 2 == 0, lo, hi) | 0x80)
    up = np.nextafter(mids, np.inf)
    dn = np.nextafter(mids, -np.inf)
    assert np.array_equal(O.e4m3_encode(up).astype(np.int64), hi)
    assert np.array_equal(O.e4m3_encode(dn).astype(np.int64), lo)


def pin_e4m3_vs_torch(O):
    """Library routine: torch's float8_e4m3fn conversion rounds to nearest even
    and saturates below 480 (above that it returns NaN, so the sweep stops
    there). Sweep every BF16 pattern with |x| < 464, plus float32 values next to
    every midpoint."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) < 464)]
    pos = O.e4m3_decode(np.arange(0x7F))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    extra = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf))])
    f = np.concatenate([f, extra, -extra, np.array([448, 455.9, 463.9], np.float32)])
    t = torch.from_numpy(f.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = O.e4m3_encode(f.astype(np.float64))
    assert np.array_equal(ours, t), np.flatnonzero(ours != t)[:10]


def pin_e4m3_saturation(O):
    """Magnitudes above 448 saturate to +-448; NaN stays NaN; sign kept on zero."""
    x = np.array([448.0, 449.0, 464.0, 480.0, 500.0, 1e9, np.inf, -500.0, -np.inf, np.nan, -0.0, 0.0, -1e-30])
    exp = [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x80, 0x00, 0x80]
    assert O.e4m3_encode(x).tolist() == exp


def pin_bf16_vs_torch(O):
    """Library routine: torch's FP32 -> BF16 conversion is round-to-nearest-even
    ([FMT] §二.2). The oracle's rounding agrees on FP32-representable inputs."""
    g = np.random.Generator(np.random.Philox(11))
    with np.errstate(over="ignore"):
        f = (g.standard_normal(200000) * np.exp2(g.integers(-140, 128, 200000))).astype(np.float32)
    f = f[np.isfinite(f)]
    t = torch.from_numpy(f).to(torch.bfloat16).float().numpy().astype(np.float64)
    ours = O.bf16_round(f.astype(np.float64))
    assert np.array_equal(ours, t)


# ---------------------------------------------------------------------------
# MX quantisation
# ---------------------------------------------------------------------------

def _block(values, fill=0.0):
    b = np.full(32, fill, dtype=np.float64)
    b[: len(values)] = values
    return b


def pin_scale_hand_blocks(O):
    """Hand-worked blocks under X = floor(log2 amax) - 8 (derivations inline)."""
    q = lambda vals: O.mx_quantize_blocks(_block(vals)[None, :])
    # amax 448 = 1.75 * 2**8 -> X = 0 -> code 127; 448 encodes as 0x7E
    s, c = q([448.0, 1.0])
    assert s[0] == 127 and c[0, 0] == 0x7E and c[0, 1] == 0x38
    # amax 1 -> X = -8 -> code 119; 1 * 2**8 = 256 = 1.0 * 2**8 -> e = 15, m = 0 -> 0x78
    s, c = q([1.0, -0.5])
    assert s[0] == 119 and c[0, 0] == 0x78 and c[0, 1] == 0xF0   # -128 = -1.0 * 2**7
    # amax 9984 (BF16 of 1e4) = 1.21875 * 2**13 -> X = 5 -> code 132; 9984 / 32 = 312
    # lies between 288 (1.125*2**8) and 320 (1.25*2**8), above the midpoint 304 -> 320 = 0x7A
    s, c = q([9984.0, 1.0])
    assert s[0] == 132 and c[0, 0] == 0x7A
    # 1.0 / 32 = 2**-5 = 1.0 * 2**-5 -> e = 2, m = 0 -> 0x10
    assert c[0, 1] == 0x10
    # amax 500 -> floor(log2 500) = 8 -> X = 0; 500 > 448 saturates to 0x7E
    s, c = q([500.0, -500.0, 3.0])
    assert s[0] == 127 and c[0, 0] == 0x7E and c[0, 1] == 0xFE and c[0, 2] == 0x44  # 3 = 1.5*2**1
    # all-zero block: X clamps to -127 -> code 0; data keeps the sign
    s, c = q([0.0, -0.0])
    assert s[0] == 0 and c[0, 0] == 0x00 and c[0, 1] == 0x80 and np.all(c[0, 2:] == 0)
    # BF16 subnormal amax 5 * 2**-133: floor(log2) = -131 -> X = -139 clamps to -127;
    # 5 * 2**-133 * 2**127 = 5 * 2**-6 = 1.25 * 2**-4 -> e = 3, m = 2 -> 0x1A;
    # 2**-133 * 2**127 = 2**-6 -> 0x08
    s, c = q([5 * 2.0 ** -133, 2.0 ** -133])
    assert s[0] == 0 and c[0, 0] == 0x1A and c[0, 1] == 0x08   # 2**-6: min normal
    # amax 2**-3 -> X = -11; sibling 2**-15 * 2**11 = 2**-4 -> 0x18 ; sibling 2**-20 * 2**11
    # = 2**-9 -> min subnormal 0x01; sibling 3 * 2**-22 * 2**11 = 1.5 * 2**-10 -> between 0
    # and 2**-9, above the midpoint 2**-10 -> 0x01; 2**-22 * 2**11 = 2**-11 -> 0
    s, c = q([2.0 ** -3, 2.0 ** -15, 2.0 ** -20, 3 * 2.0 ** -22, 2.0 ** -22, -2.0 ** -22])
    assert s[0] == 116 and c[0, :6].tolist() == [0x78, 0x18, 0x01, 0x01, 0x00, 0x80]
    # BF16 max (2 - 2**-7) * 2**127 -> X = 119 -> code 246; value / 2**119 = 255.0 * 2**0... =
    # 1.9921875 * 2**8 = 510 > 448 -> saturates
    s, c = q([(2 - 2.0 ** -7) * 2.0 ** 127])
    assert s[0] == 246 and c[0, 0] == 0x7E
    # NaN / Inf blocks: scale 0xFF, every element 0x7F with its sign
    s, c = q([np.nan, -1.0])
    assert s[0] == 0xFF and c[0, 0] == 0x7F and c[0, 1] == 0xFF and c[0, 2] == 0x7F
    s, c = q([np.inf, 1.0])
    assert s[0] == 0xFF and c[0, 0] == 0x7F


def pin_fp32_master_blocks(O):
    """Hand-worked blocks of FP32 values that BF16 cannot hold ("DeepSeek-V3 16B
    FSDP2 MXFP8/HiF8 训练设计" §8.1 and §10: weights are quantised from the
    FP32 master). Each case below would come out differently if the input were
    first rounded to BF16."""
    q = lambda vals: O.mx_quantize_blocks(_block(vals)[None, :])
    # amax 256 = 1.0 * 2**8 -> X = 0 -> code 127; 256 -> e = 15, m = 0 -> 0x78.
    # 1.0625 is the midpoint of E4M3 1.0 (0x38) and 1.125 (0x39): ties to the even
    # code 0x38. 1.0625 + 2**-20 (an FP32 value; BF16 would round it to 1.0625)
    # lies above the midpoint -> 0x39, and its negative -> 0xB9.
    s, c = q([256.0, 1.0625 + 2.0 ** -20, 1.0625, -(1.0625 + 2.0 ** -20)])
    assert s[0] == 127 and c[0, :4].tolist() == [0x78, 0x39, 0x38, 0xB9]
    # amax 512 - 2**-15 (FP32; BF16 rounds it up to 512 = 2**9): floor(log2) = 8 ->
    # X = 0 -> code 127, and the element saturates to 0x7E; 3 = 1.5 * 2**1 -> 0x44.
    s, c = q([512.0 - 2.0 ** -15, 3.0])
    assert s[0] == 127 and c[0, 0] == 0x7E and c[0, 1] == 0x44
    # amax 448 -> X = 0. 2**-10 is the midpoint of 0 and the smallest subnormal
    # 2**-9: ties to even -> 0x00; 2**-10 + 2**-30 (FP32 only) lies above it -> 0x01.
    s, c = q([448.0, 2.0 ** -10, 2.0 ** -10 + 2.0 ** -30, -(2.0 ** -10 + 2.0 ** -30)])
    assert s[0] == 127 and c[0, :4].tolist() == [0x7E, 0x00, 0x01, 0x81]
    # FP32 subnormal amax 3 * 2**-148: floor(log2) = -147 -> X clamps to -127 -> code 0;
    # 3 * 2**-148 * 2**127 = 3 * 2**-21 < 2**-10 -> 0x00, its negative -> 0x80.
    s, c = q([3 * 2.0 ** -148, -3 * 2.0 ** -148])
    assert s[0] == 0 and c[0, 0] == 0x00 and c[0, 1] == 0x80
    # The oracle takes the FP32 values as they are: float32 -> float64 is exact.
    x = np.array([1.0625 + 2.0 ** -20], dtype=np.float32)
    assert float(np.asarray(x, dtype=np.float64)[0]) == 1.0625 + 2.0 ** -20


def pin_quant_error_bound(O):
    """Invariants of MX rounding for random blocks: each dequantised element is
    within half an E4M3 spacing of the input (<= 2**-4 relative in the normal
    range, <= 2**(X-10) absolute in the subnormal range) unless it saturated;
    the block maximum lands in the top binade [256, 448] or saturates."""
    g = np.random.Generator(np.random.Philox(5))
    x = g.standard_normal((4000, 32)) * np.exp2(g.integers(-30, 30, (4000, 1)))
    x = O.bf16_bits_to_float64((x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))
    s, c = O.mx_quantize_blocks(x)
    X = s.astype(np.float64) - 127
    deq = O.e4m3_decode(c) * np.exp2(X)[:, None]
    scaled = np.abs(x) * np.exp2(-X)[:, None]
    sat = scaled > 448
    normal = (scaled >= 2.0 ** -6) & ~sat
    sub = scaled < 2.0 ** -6
    err = np.abs(deq - x)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]))
    assert np.all(err[sub] <= np.broadcast_to(np.exp2(X - 10)[:, None], x.shape)[sub])
    assert np.all(np.abs(deq[sat]) == 448 * np.broadcast_to(np.exp2(X)[:, None], x.shape)[sat])
    amax_idx = np.argmax(np.abs(x), axis=1)
    top = c[np.arange(len(c)), amax_idx] & 0x7F
    assert np.all((top >> 3) == 0xF) and np.all(top != 0x7F)


def _loop_quantize_cols(O, x):
    """Explicit loops: for each column c and each 32-row block, quantise."""
    R, C = x.shape
    data = np.zeros((C, R), np.uint8)
    sc = np.zeros((C, R // 32), np.uint8)
    for c in range(C):
        for rb in range(R // 32):
            s, codes = O.mx_quantize_blocks(x[rb * 32:(rb + 1) * 32, c][None, :])
            sc[c, rb] = s[0]
            data[c, rb * 32:(rb + 1) * 32] = codes[0]
    return data, sc


def _loop_quantize_rows(O, x):
    R, C = x.shape
    data = np.zeros((R, C), np.uint8)
    sc = np.zeros((R, C // 32), np.uint8)
    for r in range(R):
        for kb in range(C // 32):
            s, codes = O.mx_quantize_blocks(x[r, kb * 32:(kb + 1) * 32][None, :])
            sc[r, kb] = s[0]
            data[r, kb * 32:(kb + 1) * 32] = codes[0]
    return data, sc


def _rand_bf16(shape, seed, spread=8):
    g = np.random.Generator(np.random.Philox(seed))
    x = g.standard_normal(shape) * np.exp2(g.integers(-spread, spread, shape))
    return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def pin_row_col_blocking(O):
    """Row copy = 1x32 blocks along rows; col copy = 32x1 blocks down columns,
    stored transposed. Checked against explicit loops on a non-square input."""
    x = O.bf16_bits_to_float64(_rand_bf16((64, 96), 3))
    d, s = O.mx_quantize_rowwise(x)
    ld, ls = _loop_quantize_rows(O, x)
    assert np.array_equal(d, ld) and np.array_equal(s, ls)
    d, s = O.mx_quantize_colwise(x)
    ld, ls = _loop_quantize_cols(O, x)
    assert d.shape == (96, 64) and np.array_equal(d, ld) and np.array_equal(s, ls)


def pin_scale_layout(O):
    """Scale-tile layout: explicit byte positions and a round trip."""
    off = lambda r, k, kbp: int(O.mx_scale_byte_offset(r, k, kbp))
    assert off(0, 0, 4) == 0 and off(1, 0, 4) == 16 and off(31, 0, 4) == 496
    assert off(32, 0, 4) == 4 and off(64, 0, 4) == 8 and off(96, 3, 4) == 15
    assert off(0, 1, 4) == 1 and off(0, 4, 8) == 512 and off(128, 0, 8) == 1024
    assert off(129, 5, 8) == 1024 + 512 + 16 + 1
    g = np.random.Generator(np.random.Philox(9))
    for rows, kb in [(1, 1), (200, 13), (128, 4), (300, 64)]:
        s = g.integers(0, 255, (rows, kb)).astype(np.uint8)
        buf = O.mx_scale_swizzle(s)
        assert buf.size == O.mx_scale_nbytes(rows, kb * 32)
        assert np.array_equal(O.mx_scale_unswizzle(buf, rows, kb), s)
        pad = np.ones(buf.size, bool)
        r, k = np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij")
        pad[O.mx_scale_byte_offset(r, k, ((kb + 3) // 4) * 4)] = False
        assert np.all(buf[pad] == 0)
        assert np.unique(O.mx_scale_byte_offset(r, k, ((kb + 3) // 4) * 4)).size == rows * kb


def pin_grouped_quant(O):
    """Grouped 32x1 blocks restart at each group's first row; segments are
    zero-padded to multiples of 128 and stored transposed; empty groups take
    no columns."""
    counts = [20, 0, 150, 1, 128]
    offs = np.concatenate([[0], np.cumsum(counts)])
    x = O.bf16_bits_to_float64(_rand_bf16((int(offs[-1]), 64), 4))
    d, s, poff = O.mx_quantize_colwise_grouped(x, offs)
    assert poff.tolist() == [0, 128, 128, 384, 512, 640]
    assert d.shape == (64, 640) and s.shape == (64, 20)
    for e in range(len(counts)):
        m = counts[e]
        seg = np.zeros((int(poff[e + 1] - poff[e]), 64))
        seg[:m] = x[offs[e]:offs[e] + m]
        ld, ls = _loop_quantize_cols(O, seg)
        assert np.array_equal(d[:, poff[e]:poff[e + 1]], ld)
        assert np.array_equal(s[:, poff[e] // 32:poff[e + 1] // 32], ls)
    # the 20-row group's block holds rows 0..19 only: its scale follows their amax
    amax = np.max(np.abs(x[0:20]), axis=0)
    assert np.array_equal(s[:, 0], O.mx_scale_exponent(amax) + 127)


# ---------------------------------------------------------------------------
# GEMM
# ---------------------------------------------------------------------------

def _rand_operand(O, rows, k, seed):
    g = np.random.Generator(np.random.Philox(seed))
    codes = g.integers(0, 256, (rows, k)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C
    scale = g.integers(120, 134, (rows, k // 32)).astype(np.uint8)
    return codes, scale


def _exact_value(code: int, scode: int) -> Fraction:
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    v *= Fraction(2) ** (scode - 127)
    return -v if s else v


def pin_gemm_bruteforce(O):
    """Exact rational dot products of dequantised operands (non-square so that
    a transposed operand fails)."""
    M, N, K = 3, 5, 96
    ac, asc = _rand_operand(O, M, K, 1)
    bc, bsc = _rand_operand(O, N, K, 2)
    ref, S = O.mx_gemm_ref(ac, asc, bc, bsc)
    assert ref.shape == (M, N)
    for i in range(M):
        for j in range(N):
            terms = [_exact_value(int(ac[i, k]), int(asc[i, k // 32])) *
                     _exact_value(int(bc[j, k]), int(bsc[j, k // 32])) for k in range(K)]
            assert Fraction(ref[i, j]) == sum(terms), (i, j)
            assert Fraction(S[i, j]) == sum(abs(t) for t in terms), (i, j)
    r2, s2 = O.mx_gemm_ref_entries(ac, asc, bc, bsc, [0, 2, 1], [4, 0, 3])
    assert np.array_equal(r2, ref[[0, 2, 1], [4, 0, 3]]) and np.array_equal(s2, S[[0, 2, 1], [4, 0, 3]])


def pin_gemm_single_block(O):
    """K = 32, one element pair non-zero: the result is the textbook product
    q_a * q_b * 2**(Xa + Xb)."""
    a = np.zeros((1, 32), np.uint8)
    b = np.zeros((1, 32), np.uint8)
    a[0, 7] = 0x7A      # 320 (1.25 * 2**8)
    b[0, 7] = 0xB3      # -(1 + 3/8) * 2**-1 = -0.6875
    ref, S = O.mx_gemm_ref(a, np.array([[130]], np.uint8), b, np.array([[120]], np.uint8))
    assert ref[0, 0] == 320 * -0.6875 * 2.0 ** (3 - 7) and S[0, 0] == -ref[0, 0]


def pin_gemm_modes(O):
    """fprop / dgrad / wgrad through the row and column copies equal the plain
    products of the dequantised tensors they were made from: X W^T, dY W, dY^T X
    ([DSV3] §8 direction table)."""
    g = np.random.Generator(np.random.Philox(21))
    M, K, N = 64, 96, 32
    X = O.bf16_bits_to_float64(_rand_bf16((M, K), 22, 2))
    W = O.bf16_bits_to_float64(_rand_bf16((N, K), 23, 2))
    dY = O.bf16_bits_to_float64(_rand_bf16((M, N), 24, 2))
    xr, xrs = O.mx_quantize_rowwise(X)
    wr, wrs = O.mx_quantize_rowwise(W)
    y, _ = O.mx_gemm_ref(xr, xrs, wr, wrs)
    assert np.allclose(y, O.mx_dequantize(xr, xrs) @ O.mx_dequantize(wr, wrs).T, rtol=0, atol=0)
    # dgrad dX[M, K] = dY[M, N] W[N, K]: A = dY row copy, B = W column copy ([K, N])
    dr, drs = O.mx_quantize_rowwise(dY)
    wc, wcs = O.mx_quantize_colwise(W)
    dx, _ = O.mx_gemm_ref(dr, drs, wc, wcs)
    assert dx.shape == (M, K)
    Wq_col = O.mx_dequantize(wc, wcs).T       # W as seen through its column copy, [N, K]
    assert np.allclose(dx, O.mx_dequantize(dr, drs) @ Wq_col, rtol=1e-12, atol=0)
    assert np.max(np.abs(Wq_col - W)) <= 2.0 ** -4 * np.max(np.abs(W))
    # wgrad dW[N, K] = dY^T X: A = dY column copy [N, M], B = X column copy [K, M]
    dc, dcs = O.mx_quantize_colwise(dY)
    xc, xcs = O.mx_quantize_colwise(X)
    dw, _ = O.mx_gemm_ref(dc, dcs, xc, xcs)
    assert dw.shape == (N, K)
    assert np.allclose(dw, O.mx_dequantize(dc, dcs) @ O.mx_dequantize(xc, xcs).T, rtol=1e-12, atol=0)
    assert np.allclose(dw, dY.T @ X, rtol=0.1, atol=0.2 * np.sqrt(M))


def pin_grouped_gemm(O):
    """One group equals the dense GEMM; empty groups give no rows (M-ragged) and
    exact zeros (K-ragged); permuting experts permutes the results."""
    K, N, Kout = 64, 48, 32
    counts = [37, 0, 91, 5]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    Mt = int(offs[-1])
    X = O.bf16_bits_to_float64(_rand_bf16((Mt, K), 31, 2))
    W = np.stack([O.bf16_bits_to_float64(_rand_bf16((N, K), 40 + e, 2)) for e in range(4)])
    xr, xrs = O.mx_quantize_rowwise(X)
    wq = [O.mx_quantize_rowwise(W[e]) for e in range(4)]
    wc = np.stack([w[0] for w in wq])
    ws = np.stack([w[1] for w in wq])
    ref, S = O.mx_grouped_gemm_ref_mragged(xr, xrs, wc, ws, offs)
    for e in range(4):
        r, s = O.mx_gemm_ref(xr[offs[e]:offs[e + 1]], xrs[offs[e]:offs[e + 1]], wc[e], ws[e])
        assert np.array_equal(ref[offs[e]:offs[e + 1]], r)
    one, _ = O.mx_grouped_gemm_ref_mragged(xr, xrs, wc[:1], ws[:1], np.array([0, Mt]))
    dense, _ = O.mx_gemm_ref(xr, xrs, wc[0], ws[0])
    assert np.array_equal(one, dense)
    # K-ragged wgrad
    dY = O.bf16_bits_to_float64(_rand_bf16((Mt, N), 50, 2))
    a, as_, _ = O.mx_quantize_colwise_grouped(dY, offs)
    b, bs, _ = O.mx_quantize_colwise_grouped(X, offs)
    dw, _ = O.mx_grouped_gemm_ref_kragged(a, as_, b, bs, offs)
    assert dw.shape == (4, N, K)
    assert np.all(dw[1] == 0)
    for e in [0, 2, 3]:
        seg = slice(offs[e], offs[e + 1])
        pad = ((counts[e] + 127) // 128) * 128
        dpad = np.zeros((pad, N)); dpad[:counts[e]] = dY[seg]
        xpad = np.zeros((pad, K)); xpad[:counts[e]] = X[seg]
        ac_, acs = O.mx_quantize_colwise(dpad)
        bc_, bcs = O.mx_quantize_colwise(xpad)
        r, _ = O.mx_gemm_ref(ac_, acs, bc_, bcs)
        assert np.array_equal(dw[e], r)
    # permutation of experts
    perm = [2, 0, 3, 1]
    counts_p = [counts[p] for p in perm]
    offs_p = np.concatenate([[0], np.cumsum(counts_p)]).astype(np.int64)
    Xp = np.concatenate([X[offs[p]:offs[p + 1]] for p in perm])
    dYp = np.concatenate([dY[offs[p]:offs[p + 1]] for p in perm])
    a2, as2, _ = O.mx_quantize_colwise_grouped(dYp, offs_p)
    b2, bs2, _ = O.mx_quantize_colwise_grouped(Xp, offs_p)
    dw2, _ = O.mx_grouped_gemm_ref_kragged(a2, as2, b2, bs2, offs_p)
    for i, p in enumerate(perm):
        assert np.array_equal(dw2[i], dw[p])


def pin_blockwise_fp8(O):
    """DeepSeek-V3 blockwise FP8 as the numerics page states it (§七.2-§七.3:
    s = 448 / amax, x~ = fl_E4M3(s * x); 1x128 activation and 128x128 weight
    blocks; each 128-K partial sum promoted with s_a and s_w). Hand-worked
    blocks, block structure by explicit loops, and exact GEMM values."""
    row = lambda vals: O.quantize_1x128(np.array([list(vals) + [0.0] * (128 - len(vals))]))
    # amax 1 -> s = 448: 1 -> 448 = 0x7E, 0.5 -> 224 = 1.75 * 2**7 -> 0x76, -1 -> 0xFE
    c, sc = row([1.0, 0.5, -1.0])
    assert sc[0, 0] == 448.0 and c[0, :3].tolist() == [0x7E, 0x76, 0xFE]
    # amax 3 -> s = fl32(448/3): 448/3 * 2**16 = 9786709.33 -> s = 9786709 * 2**-16
    # = 149.33332824707031 (FP32 spacing 2**-16 on [128, 256)). x = 1: s lies in [144, 160)
    # (E4M3 step 16 at 2**7), below the midpoint 152 -> 144 = 1.125 * 2**7 -> 0x71.
    # x = 3: 3 s = 29360127 * 2**-16 = 448 - 2**-16, the FP32 midpoint of 448 - 2**-15 and
    # 448 (spacing 2**-15 on [256, 512)); ties to even -> 448.0 -> 0x7E.
    c, sc = row([1.0, 3.0])
    assert float(sc[0, 0]) == 9786709 * 2.0 ** -16 and c[0, 0] == 0x71 and c[0, 1] == 0x7E
    # amax 448 -> s = 1: the codes are the plain E4M3 codes (2.0 -> 0x40, -0.25 -> 0xA8)
    c, sc = row([448.0, 2.0, -0.25])
    assert sc[0, 0] == 1.0 and c[0, :3].tolist() == [0x7E, 0x40, 0xA8]
    # all-zero block: s = 1 and the data keeps the sign
    c, sc = O.quantize_1x128(np.concatenate([np.zeros((1, 128)), -np.zeros((1, 128))]))
    assert np.all(sc == 1.0) and np.all(c[0] == 0x00) and np.all(c[1] == 0x80)
    # block structure: 1x128 blocks per row; 128x128 blocks share one amax
    g = np.random.Generator(np.random.Philox(21))
    x = g.standard_normal((3, 256)) * np.array([1.0, 10.0, 0.01])[:, None]
    c, sc = O.quantize_1x128(x)
    for i in range(3):
        for kb in range(2):
            assert sc[i, kb] == np.float32(448.0) / np.float32(np.abs(x[i, kb * 128:(kb + 1) * 128]).max())
    w = g.standard_normal((200, 256))
    w[5, 3] = 1000.0          # one outlier: only block (0, 0) sees it
    cw, sw = O.quantize_128x128(w)
    assert sw.shape == (2, 2)
    assert sw[0, 0] == np.float32(448.0) / np.float32(1000.0)
    assert sw[1, 0] == np.float32(448.0) / np.float32(np.abs(w[128:, :128]).max())
    assert sw[0, 1] == np.float32(448.0) / np.float32(np.abs(w[:128, 128:]).max())
    # GEMM, one-hot: A row i = 1.0 (0x38) at k_i with s_a = 2, B = codes with s_b = 4:
    # each output is (1/2) * b / 4
    a = np.zeros((2, 256), dtype=np.uint8)
    a[0, 5] = 0x38
    a[1, 130] = 0x38
    a_s = np.full((2, 2), 2.0, dtype=np.float32)
    b = g.integers(0, 0x7E, size=(3, 256)).astype(np.uint8)
    b_s = np.full((1, 2), 4.0, dtype=np.float32)
    ref, S = O.gemm_blockwise_ref(a, a_s, b, b_s)
    bv = O.e4m3_decode(b)
    assert np.array_equal(ref[0], bv[:, 5] / 8.0) and np.array_equal(ref[1], bv[:, 130] / 8.0)
    # two K blocks with different scales add: exact rational sum against brute force
    a_s2 = np.array([[2.0, 0.5]], dtype=np.float32)
    b_s2 = np.array([[4.0, 0.25]], dtype=np.float32)
    a2 = g.integers(0, 0x7E, size=(1, 256)).astype(np.uint8)
    b2 = g.integers(0, 0x7E, size=(1, 256)).astype(np.uint8)
    r2, _ = O.gemm_blockwise_ref(a2, a_s2, b2, b_s2)
    av, bv2 = O.e4m3_decode(a2)[0], O.e4m3_decode(b2)[0]
    exact = sum(Fraction(av[k]) * Fraction(bv2[k]) / (Fraction(float(a_s2[0, k // 128])) * Fraction(float(b_s2[0, k // 128])))
                for k in range(256))
    assert abs(Fraction(r2[0, 0]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)


def _fp32_rn(q: Fraction) -> Fraction:
    """The FP32 number nearest to the rational q (ties to even), by exact
    arithmetic: 24 significant bits, subnormal spacing 2**-149."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                      # binade [2**e, 2**(e+1)), or the subnormal range
    ulp = Fraction(2) ** (e - 23)
    m = a / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def pin_current_scaling(O):
    """Current scaling with one FP32 scale per tensor or per leading group
    ("DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §3.2: scale = valid(amax) ?
    amax / format_max : 1.0 in FP32; dense per tensor, 3-D grouped weights per
    leading group), on E4M3 data: closed forms, the FP32 rounding of the scale
    and of the quotient, validity, per-group independence, exact GEMM values."""
    # the page's own format maxima: amax 30 with 15 -> 2, amax 448 with 224 -> 2
    assert O.current_scale(30.0, 15.0) == 2.0 and O.current_scale(448.0, 224.0) == 2.0
    assert O.current_scale(7.5, 15.0) == 0.5
    # E4M3: 448 -> 1, 224 -> 0.5, 896 -> 2 (exact), and amax 1 -> the FP32 nearest 1/448
    assert O.current_scale(448.0) == 1.0 and O.current_scale(224.0) == 0.5 and O.current_scale(896.0) == 2.0
    assert Fraction(float(O.current_scale(1.0))) == _fp32_rn(Fraction(1, 448))
    # invalid amax (zero, infinite, NaN) -> 1.0
    for a in (0.0, float("inf"), float("nan")):
        assert O.current_scale(a) == 1.0
    # the scale is the FP32 rounding of amax / 448 over BF16 amax values,
    # subnormal FP32 scales included (BF16 subnormal amax)
    g = np.random.Generator(np.random.Philox(31))
    pats = np.concatenate([g.integers(0x0001, 0x7F80, 400), [0x0001, 0x007F, 0x0080, 0x7F7F]]).astype(np.uint32)
    for b in pats:
        a = float((b << 16).astype(np.uint32).view(np.float32))
        assert Fraction(float(O.current_scale(a))) == _fp32_rn(Fraction(a) / 448), hex(int(b))
    # one element: amax 3 -> s = fl32(3/448); x = 1 -> fl32(1/s) = 149.33... lies in
    # [144, 160) below the midpoint 152 -> 144 = 1.125 * 2**7 -> 0x71; x = -3 -> -448 -> 0xFE
    s3 = O.current_scale(3.0)
    assert Fraction(float(s3)) == _fp32_rn(Fraction(3, 448))
    assert O.current_encode(np.array([1.0, -3.0, 0.0, -0.0]), s3).tolist() == [0x71, 0xFE, 0x00, 0x80]
    # the quotient is rounded to FP32 before E4M3: amax 0.6875 -> s = fl32(11/7168);
    # x = 33/512 gives x/s = 42.0000009..., whose FP32 rounding is exactly 42, the
    # midpoint of 40 (0x62, even mantissa) and 44 (0x63): ties to even -> 0x62 (the
    # exact quotient would round up to 0x63)
    s = O.current_scale(0.6875)
    assert Fraction(float(s)) == _fp32_rn(Fraction(11, 7168))
    q = Fraction(33, 512) / Fraction(float(s))
    assert q > 42 and _fp32_rn(q) == 42
    assert O.current_encode(np.array([0.064453125]), s)[0] == 0x62
    # every element against exact arithmetic on a random tensor with an outlier;
    # the amax element lands on +-448 (the quotient is within an FP32 rounding of 448)
    x = g.standard_normal((8, 40)).astype(np.float32).astype(np.float64)
    x[3, 7] = -57.25
    codes, sc, amax = O.current_quantize(x)
    assert amax == 57.25 and Fraction(float(sc)) == _fp32_rn(Fraction(57.25) / 448)
    assert codes[3, 7] == 0xFE
    for i in range(0, 8, 3):
        for j in range(0, 40, 7):
            qv = _fp32_rn(Fraction(x[i, j]) / Fraction(float(sc)))
            assert codes[i, j] == O.e4m3_encode(np.array([float(qv)]))[0]
    # scale 1 (amax exactly 448): the codes are the plain E4M3 codes
    y = np.array([[448.0, 2.0, -0.25, 3.3]])
    cy, sy, _ = O.current_quantize(y)
    assert sy == 1.0 and np.array_equal(cy, O.e4m3_encode(y))
    # per leading group: each group's scale from its own amax only
    w = g.standard_normal((3, 16, 32)) * np.array([1.0, 100.0, 0.001])[:, None, None]
    cw, sw, aw = O.current_quantize_groups(w)
    for e in range(3):
        assert sw[e] == O.current_scale(np.abs(w[e]).max()) and aw[e] == np.abs(w[e]).max()
    cw2, sw2, _ = O.current_quantize_groups(w[::-1])
    assert np.array_equal(sw2, sw[::-1]) and np.array_equal(cw2, cw[::-1])
    # GEMM: exact rational sum of (qa * s_a) * (qb * s_b)
    a = g.integers(0, 0x7E, size=(3, 64)).astype(np.uint8) | (g.integers(0, 2, size=(3, 64)) << 7).astype(np.uint8)
    b = g.integers(0, 0x7E, size=(2, 64)).astype(np.uint8)
    sa, sb = np.float32(0.3), np.float32(1.7)
    ref, S = O.current_gemm_ref(a, sa, b, sb)
    av, bv = O.e4m3_decode(a), O.e4m3_decode(b)
    for i in range(3):
        for j in range(2):
            exact = sum(Fraction(av[i, k]) * Fraction(bv[j, k]) for k in range(64)) * Fraction(float(sa)) * \
                Fraction(float(sb))
            assert abs(Fraction(ref[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 80)
            assert S[i, j] >= abs(ref[i, j])
    # grouped operand layout: rows of group e transposed into its padded segment
    c = g.integers(1, 255, size=(200, 5)).astype(np.uint8)
    offs = np.array([0, 0, 130, 131, 200])
    t = O.current_transpose_grouped(c, offs)
    assert t.shape == (5, 0 + 256 + 128 + 128)
    for col in range(5):
        assert np.array_equal(t[col, 0:130], c[0:130, col]) and np.all(t[col, 130:256] == 0)
        assert t[col, 256] == c[130, col] and np.all(t[col, 257:384] == 0)
        assert np.array_equal(t[col, 384:453], c[131:200, col]) and np.all(t[col, 453:] == 0)


def pin_swiglu(O):
    """SiLU by its closed forms, SwiGLU's gate/up halves by explicit loops, and
    the grouped SwiGLU reference on one-hot operands whose dots are single
    E4M3 values ("DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §5: gate_up_proj
    [E, 2F, H], gate rows first)."""
    ln3 = math.log(3.0)
    # sigmoid(ln 3) = 1 / (1 + 1/3) = 3/4, sigmoid(-ln 3) = 1/4
    v = O.silu(np.array([0.0, ln3, -ln3, 40.0, -40.0]))
    assert v[0] == 0.0
    assert abs(v[1] - 0.75 * ln3) <= 1e-15 and abs(v[2] + 0.25 * ln3) <= 1e-15
    assert abs(v[3] - 40.0 / (1.0 + math.exp(-40.0))) <= 1e-13
    assert abs(v[4] + 40.0 * math.exp(-40.0) / (1.0 + math.exp(-40.0))) <= 1e-30
    x = np.random.Generator(np.random.Philox(11)).standard_normal(1000) * 8
    assert np.allclose(O.silu(x) - O.silu(-x), x, rtol=0, atol=1e-12)       # x*s(x) + x*s(-x) = x
    # the slope bound used by the tolerance: max |silu'| = 1.0998 at x ~ 2.40
    t = np.linspace(-20, 20, 400001)
    d = np.abs(np.gradient(O.silu(t), t))
    assert 1.09 < d.max() <= O.SILU_MAX_SLOPE
    # halves: out[:, f] = silu(y[:, f]) * y[:, F + f]
    y = np.random.Generator(np.random.Philox(12)).standard_normal((5, 6))
    out = O.swiglu(y)
    for i in range(5):
        for f in range(3):
            g, u = y[i, f], y[i, 3 + f]
            assert abs(out[i, f] - g / (1.0 + math.exp(-g)) * u) <= 1e-15 * (1 + abs(u))
    # one-hot grouped case: E = 2, F = 2 (N = 4), K = 32; row i of A is 1.0 at
    # column k_i (code 0x38, scale 2**0), so dot(i, n) = B_e[n, k_i]
    offs = np.array([0, 2, 3])
    ks = [3, 17, 30]
    a = np.zeros((3, 32), dtype=np.uint8)
    for i, k in enumerate(ks):
        a[i, k] = 0x38
    a_s = np.full((3, 1), 127, dtype=np.uint8)
    g = np.random.Generator(np.random.Philox(13))
    b = g.integers(0, 0x7E, size=(2, 4, 32)).astype(np.uint8) | (g.integers(0, 2, size=(2, 4, 32)) << 7).astype(np.uint8)
    b_s = np.full((2, 4, 1), 127, dtype=np.uint8)
    res, gate, up, _, _ = O.mx_grouped_swiglu_ref(a, a_s, b, b_s, offs)
    for i, k in enumerate(ks):
        e = 0 if i < 2 else 1
        for f in range(2):
            gv = float(O.e4m3_decode(np.array([b[e, f, k]]))[0])
            uv = float(O.e4m3_decode(np.array([b[e, 2 + f, k]]))[0])
            assert gate[i, f] == gv and up[i, f] == uv
            assert abs(res[i, f] - gv / (1.0 + math.exp(-gv)) * uv) <= 1e-12 * (1 + abs(uv * gv))
    # the acceptance bound: exact passes, BF16-sized rounding passes, 2**-6 fails
    r = np.array([1.0, -3.0, 100.0])
    z = np.zeros(3)
    assert np.all(O.swiglu_within_tolerance(r, r, r, r, z, z))
    assert np.all(O.swiglu_within_tolerance(r * (1 + 2.0 ** -9), r, r, r, z, z))
    assert not np.any(O.swiglu_within_tolerance(r * (1 + 2.0 ** -6), r, r, r, z, z))


def pin_tolerance(O):
    """Acceptance bound: BF16 rounding of the exact value passes; an error of
    2**-6 relative fails; a 1e-6*S-sized absolute error passes."""
    g = np.random.Generator(np.random.Philox(77))
    ref = g.standard_normal(10000) * 100
    S = np.abs(ref) * 30
    assert np.all(O.within_tolerance(O.bf16_round(ref), ref, S))
    assert not np.any(O.within_tolerance(ref * (1 + 2.0 ** -6) + 1e-3, ref, np.zeros_like(S)))
    assert np.all(O.within_tolerance(ref + 0.9e-6 * S, ref, S))
    assert not np.any(O.within_tolerance(ref + 2.0 ** -7 * np.abs(ref) + 2e-6 * S, ref, S))


ALL_PINS = [
    pin_printed_values, pin_e4m3_closed_forms, pin_e4m3_census, pin_e4m3_roundtrip_and_ties,
    pin_e4m3_vs_torch, pin_e4m3_saturation, pin_bf16_vs_torch, pin_scale_hand_blocks,
    pin_fp32_master_blocks, pin_quant_error_bound, pin_row_col_blocking, pin_scale_layout, pin_grouped_quant,
    pin_gemm_bruteforce, pin_gemm_single_block, pin_gemm_modes, pin_grouped_gemm, pin_blockwise_fp8, pin_swiglu,
    pin_current_scaling, pin_tolerance,
]
