"""Plain CPU oracle for MXFP8 block-scaled quantisation, GEMM and grouped GEMM.

THIS IS TEST INFRASTRUCTURE. Only the tests, the smoke check in
``__graft_entry__`` and the CPU-baseline / reference legs of ``bench.py`` may
import it. The CUDA library never calls it, links it or shares code with it;
the product path fails when its extension is missing instead of falling back
to anything here.

Everything is float64 numpy, written for a reader to check by eye against the
pages. No blocking, fusion or reordering beyond what the definitions state.
The pages cited (by title and section):

[FMT]  "浮点格式、数值稳定性与混合精度" (arganzheng.life):
       §二.1 三段位与四类编码 (value formula, subnormals, special encodings);
       §二.2 八种格式的位布局 (format table; E4M3 and BF16 notes);
       §五.1 (FP32 accumulation, BF16 output); §八.3 (judging kernel-vs-reference
       differences against an FP64 reference); §九.1 (printed bit patterns).
[DSV3] "DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" (hyper-parallel issue #329):
       §3 table and §3.1 (E4M3 data, E8M0 scale, 1x32 / 32x1 blocks, separate
       row and col copies); §7.4 QuantizedOperand; §8 direction table
       (fprop / dgrad / wgrad); §13.3-13.4 quantize / matmul / grouped_matmul.
[TT]   "低精度训练特性（MXFP8 / HiFloat8）" (torchtitan-npu):
       实现原理 / 线性层低精度 (block size 32: every 32 elements share one
       scale); MoE 专家层低精度 (grouped GEMM, per-group quantisation for wgrad).

Readings taken where the pages are silent (each is also pinned by a test):

* Scale rule: X = floor(log2(amax)) - 8 and the block scale is 2**X (the OCP
  MX rule; 8 is the exponent of E4M3's largest binade, 448 = 1.75 * 2**8).
  X is clamped to [-127, 127]; the E8M0 code is X + 127.
* Element rounding: round to nearest, ties to even, magnitudes above 448
  saturate to 448 ([FMT] §二.2 leaves saturate-or-NaN to the conversion mode).
* All-zero block (amax = 0): X clamps to -127, scale code 0x00, data codes
  keep the sign (+0 -> 0x00, -0 -> 0x80).
* A block holding NaN or Inf: scale code 0xFF (E8M0 NaN) and every data code
  0x7F with the element's sign bit. Parity unpinned by the pages: documented
  behaviour only.
* Column (32x1) copies are stored transposed: the 32x1 blocks of T[R, C]
  become 1x32 blocks of the [C, R] result, so every GEMM operand is K-major.
* Grouped column quantisation: 32x1 blocks restart at each group's first row;
  each group's segment is zero-padded to a multiple of 128 rows.
* GEMM reference: the FP64 dot of the dequantised operands, kept unrounded,
  together with S = sum |a*b|; see ``within_tolerance`` for why.
* Blockwise variant recipe (1x128 / 128x128 with FP32 multipliers): the
  multiplier s = fl32(448 / amax) and the product fl32(s * x) are FP32
  steps, then RNE to E4M3; an all-zero block takes s = 1.
* Current-scaling variant (one FP32 scale per tensor or per leading group):
  scale = fl32(amax / 448) for a finite amax above zero, else 1.0; element =
  E4M3(fl32(x / scale)). 448 stands in for the HiF8 format maxima the page
  gives, since the data format here is E4M3.
* SwiGLU after the grouped gate_up GEMM: gate = the first F output columns,
  up = the last F ([DSV3] §5 lays gate_up_proj out as [E, 2F, H]), computed in
  float64 on the unrounded dots; see ``swiglu_within_tolerance``.
"""

from __future__ import annotations

import math

import numpy as np

# ----------------------------------------------------------------------------
# Format constants
# ----------------------------------------------------------------------------

E4M3_EXP_BITS = 4
E4M3_MAN_BITS = 3
E4M3_BIAS = 7            # [FMT] §二.2 table: E4M3 1/4/3, bias 7
E4M3_MAX = 448.0         # [FMT] §二.2 E4M3 note: S.1111.110 = 1.75 * 2**8
E4M3_EMAX = 8            # exponent of the largest E4M3 binade (448 = 1.75 * 2**8)
E8M0_BIAS = 127
E8M0_NAN = 0xFF
MX_BLOCK = 32            # [TT] 线性层低精度: every 32 elements share one scale
GROUP_PAD = 128          # grouped column segments start on multiples of 128 rows

# Scale-tile layout (not on the pages: it is the layout the block-scaled tensor
# core instruction reads, fixed by the library's C header). A logical scale
# matrix [rows, kb] is padded to [ceil(rows/128)*128, ceil(kb/4)*4] with zero
# bytes and cut into 512-byte atoms of 128 rows x 4 scale columns. Atoms are
# ordered with the scale-column atom index fastest. Inside an atom, the byte
# for (r, k) sits at (r % 32) * 16 + ((r // 32) % 4) * 4 + (k % 4).
SCALE_ATOM_ROWS = 128
SCALE_ATOM_COLS = 4
SCALE_ATOM_BYTES = 512


def _ceil_to(x: int, m: int) -> int:
    return ((x + m - 1) // m) * m


# ----------------------------------------------------------------------------
# BF16 ([FMT] §二.2: BF16 is the upper 16 bits of FP32; FP32 -> BF16 is
# round-to-nearest-even on the low 16 bits)
# ----------------------------------------------------------------------------

def bf16_bits_to_float64(bits) -> np.ndarray:
    """Exact value of BF16 bit patterns: place them as the top half of an FP32."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest BF16 value, ties to even.

    BF16 keeps 8 significant bits (7 stored + hidden) with FP32's exponent
    range ([FMT] §二.2 table). In the binade [2**e, 2**(e+1)) the spacing is
    2**(e-7); below the smallest normal 2**-126 the spacing stays 2**-133.
    Results beyond the largest finite BF16 value become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    _, e2 = np.frexp(np.abs(x[fin]))          # |x| = m * 2**e2, m in [0.5, 1)
    e = np.maximum(e2 - 1, -126)              # floor(log2|x|), subnormal floor
    ulp = np.exp2((e - 7).astype(np.float64))
    r = np.rint(x[fin] / ulp) * ulp           # np.rint rounds half to even
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > bf16_max, np.copysign(np.inf, r), r)
    out[fin] = r
    return out


# ----------------------------------------------------------------------------
# E4M3 ([FMT] §二.1 value formula with E=4, M=3, bias 7; §二.2 E4M3 note:
# no infinities, only S.1111.111 is NaN, maximum 448)
# ----------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """E4M3 byte codes -> float64 values.

    normal    (e in 1..15): (-1)**s * (1 + m/8) * 2**(e - 7)
    subnormal (e == 0):     (-1)**s * (m/8) * 2**(1 - 7)
    NaN: exponent field 1111 with mantissa 111 (0x7F, 0xFF) only.
    """
    c = np.asarray(codes).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2((e - E4M3_BIAS).astype(np.float64))
    subnormal = (m / 8.0) * 2.0 ** (1 - E4M3_BIAS)
    mag = np.where(e == 0, subnormal, normal)
    val = np.where(s == 1, -mag, mag)
    return np.where((e == 0xF) & (m == 0x7), np.nan, val)


# Non-negative finite codes 0x00..0x7E decode to strictly increasing values
# 0 .. 448 (checked by a test); this table is the set the encoder rounds onto.
_POS_CODES = np.arange(0x00, 0x7F, dtype=np.int64)
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(x) -> np.ndarray:
    """float64 -> E4M3 code by the definition of round-to-nearest-even.

    The result is the finite E4M3 value nearest to x; at an exact midpoint the
    code with an even mantissa (code & 1 == 0) wins. Magnitudes above 448
    saturate to 448 (including +-inf). The sign is kept, so -0 and negative
    values that round to zero give 0x80. NaN gives 0x7F with the sign bit.

    Midpoints (lo + hi) / 2 of neighbouring E4M3 values are dyadic numbers with
    few bits, exact in float64, so the comparisons below are exact.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, a)
    hi = np.searchsorted(_POS_VALUES, a, side="left")     # first value >= a
    hi = np.clip(hi, 0, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    v_hi = _POS_VALUES[hi]
    v_lo = _POS_VALUES[lo]
    mid = (v_lo + v_hi) / 2.0
    take_hi = (a == v_hi) | (a > mid) | ((a == mid) & (_POS_CODES[hi] % 2 == 0))
    idx = np.where(take_hi, hi, lo)
    code = _POS_CODES[idx] | (sign << 7)
    code = np.where(nan, 0x7F | (sign << 7), code)
    return code.astype(np.uint8)


# ----------------------------------------------------------------------------
# E8M0 scale ([DSV3] §3 table: scale dtype E8M0; exponent-only, bias 127)
# ----------------------------------------------------------------------------

def e8m0_decode(codes) -> np.ndarray:
    """E8M0 code k -> 2**(k - 127); 0xFF is NaN."""
    k = np.asarray(codes).astype(np.int64)
    v = np.exp2((k - E8M0_BIAS).astype(np.float64))
    return np.where(k == E8M0_NAN, np.nan, v)


def mx_scale_exponent(amax) -> np.ndarray:
    """Shared exponent X = floor(log2(amax)) - 8, clamped to [-127, 127].

    floor(log2(a)) is read exactly from frexp (a = m * 2**e, m in [0.5, 1)
    gives floor(log2(a)) = e - 1), also for subnormal inputs. amax = 0 gives
    the clamp value -127. Non-finite amax is handled by the caller.
    """
    a = np.asarray(amax, dtype=np.float64)
    safe = np.where(np.isfinite(a) & (a > 0), a, 1.0)
    _, e = np.frexp(safe)
    x = (e.astype(np.int64) - 1) - E4M3_EMAX
    x = np.where(a > 0, x, -E8M0_BIAS)
    return np.clip(x, -127, 127)


# ----------------------------------------------------------------------------
# MX block quantisation ([DSV3] §3, §3.1, §8.1; [TT] 线性层低精度)
# ----------------------------------------------------------------------------

def mx_quantize_blocks(blocks) -> tuple[np.ndarray, np.ndarray]:
    """Quantise blocks of 32 values (last axis) to (E8M0 code, E4M3 codes).

    amax = max |x| over the block; X = floor(log2 amax) - 8 (clamped);
    element code = RNE-saturating E4M3 of x * 2**-X. Power-of-two scaling is
    exact in float64 for every BF16 or FP32 input, so only the E4M3 rounding rounds.
    """
    b = np.asarray(blocks, dtype=np.float64)
    assert b.shape[-1] == MX_BLOCK
    with np.errstate(invalid="ignore"):
        amax = np.max(np.abs(b), axis=-1)          # NaN propagates
    finite = np.isfinite(amax)
    X = mx_scale_exponent(amax)
    scale_code = np.where(finite, X + E8M0_BIAS, E8M0_NAN).astype(np.uint8)
    y = b * np.exp2(-X.astype(np.float64))[..., None]
    codes = e4m3_encode(y)
    nan_codes = (0x7F | (np.signbit(b).astype(np.int64) << 7)).astype(np.uint8)
    codes = np.where(finite[..., None], codes, nan_codes)
    return scale_code, codes


def mx_quantize_rowwise(x) -> tuple[np.ndarray, np.ndarray]:
    """1x32 blocks along the last dim of x[R, C] ([DSV3] §3 row copy).

    Returns data [R, C] (E4M3 codes) and logical scales [R, C/32] (E8M0).
    """
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape
    assert C % MX_BLOCK == 0
    sc, codes = mx_quantize_blocks(x.reshape(R, C // MX_BLOCK, MX_BLOCK))
    return codes.reshape(R, C), sc


def mx_quantize_colwise(x) -> tuple[np.ndarray, np.ndarray]:
    """32x1 blocks down each column of x[R, C] ([DSV3] §3 col copy).

    A 32x1 block of x is a 1x32 block of its transpose, so the copy is stored
    transposed: data [C, R] and logical scales [C, R/32].
    """
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape
    assert R % MX_BLOCK == 0
    return mx_quantize_rowwise(x.T)


def mx_group_sizes(offsets) -> np.ndarray:
    """Rows per group from offsets[E+1] (offsets[0] = 0, non-decreasing)."""
    o = np.asarray(offsets, dtype=np.int64)
    assert o[0] == 0 and np.all(np.diff(o) >= 0)
    return np.diff(o)


def mx_padded_offsets(offsets) -> np.ndarray:
    """Start of each group's zero-padded column segment (multiples of 128)."""
    m = mx_group_sizes(offsets)
    pad = (m + GROUP_PAD - 1) // GROUP_PAD * GROUP_PAD
    return np.concatenate([[0], np.cumsum(pad)]).astype(np.int64)


def mx_quantize_colwise_grouped(x, offsets) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Per-group 32x1 quantisation for the grouped wgrad ([TT] MoE 专家层低精度:
    per-group dynamic MX quantisation; [DSV3] §13.3 group_list argument).

    Rows [offsets[e], offsets[e+1]) of x[M, D] form group e. Its rows are
    zero-padded to a multiple of 128 and quantised in 32x1 blocks that start
    at the group's first row, then stored transposed at columns
    [poff[e], poff[e+1]) of data [D, poff[E]] and scales [D, poff[E]/32].
    """
    x = np.asarray(x, dtype=np.float64)
    M, D = x.shape
    o = np.asarray(offsets, dtype=np.int64)
    assert o[-1] == M
    poff = mx_padded_offsets(o)
    Kp = int(poff[-1])
    data = np.zeros((D, Kp), dtype=np.uint8)
    scale = np.zeros((D, Kp // MX_BLOCK), dtype=np.uint8)
    for e in range(len(o) - 1):
        m = int(o[e + 1] - o[e])
        if m == 0:
            continue
        seg = np.zeros((int(poff[e + 1] - poff[e]), D), dtype=np.float64)
        seg[:m] = x[o[e]:o[e + 1]]
        d, s = mx_quantize_colwise(seg)
        data[:, poff[e]:poff[e + 1]] = d
        scale[:, poff[e] // MX_BLOCK:poff[e + 1] // MX_BLOCK] = s
    return data, scale, poff


def mx_dequantize(codes, scale_codes) -> np.ndarray:
    """Value of each element: E4M3 value times its block's 2**X ([DSV3] §3.1)."""
    v = e4m3_decode(codes)
    s = e8m0_decode(scale_codes)
    return v * np.repeat(s, MX_BLOCK, axis=-1)[..., : v.shape[-1]]


# ----------------------------------------------------------------------------
# Scale-tile layout (library ABI; see the layout note with the constants)
# ----------------------------------------------------------------------------

def mx_scale_padded_shape(rows: int, kb: int) -> tuple[int, int]:
    return _ceil_to(rows, SCALE_ATOM_ROWS), _ceil_to(kb, SCALE_ATOM_COLS)


def mx_scale_nbytes(rows: int, k: int) -> int:
    """Bytes of the swizzled scale buffer of an operand [rows, k]."""
    pr, pk = mx_scale_padded_shape(rows, (k + MX_BLOCK - 1) // MX_BLOCK)
    return pr * pk


def mx_scale_byte_offset(r, k, kb_padded: int):
    """Byte position of logical scale (r, k) in the swizzled buffer."""
    r = np.asarray(r, dtype=np.int64)
    k = np.asarray(k, dtype=np.int64)
    atom = (r // SCALE_ATOM_ROWS) * (kb_padded // SCALE_ATOM_COLS) + k // SCALE_ATOM_COLS
    return atom * SCALE_ATOM_BYTES + (r % 32) * 16 + ((r // 32) % 4) * 4 + (k % 4)


def mx_scale_swizzle(logical) -> np.ndarray:
    """Logical scales [rows, kb] -> swizzled byte buffer (padding bytes are 0)."""
    s = np.asarray(logical, dtype=np.uint8)
    rows, kb = s.shape
    pr, pk = mx_scale_padded_shape(rows, kb)
    out = np.zeros(pr * pk, dtype=np.uint8)
    r, k = np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij")
    out[mx_scale_byte_offset(r, k, pk)] = s
    return out


def mx_scale_unswizzle(buf, rows: int, kb: int) -> np.ndarray:
    """Swizzled byte buffer -> logical scales [rows, kb]."""
    b = np.asarray(buf, dtype=np.uint8).reshape(-1)
    _, pk = mx_scale_padded_shape(rows, kb)
    r, k = np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij")
    return b[mx_scale_byte_offset(r, k, pk)]


# ----------------------------------------------------------------------------
# GEMM references ([DSV3] §8 direction table and §13.4 matmul interfaces;
# [FMT] §五.1 FP32 accumulation with BF16 output, §八.3 FP64 reference)
# ----------------------------------------------------------------------------

def mx_gemm_ref(a_codes, a_scale, b_codes, b_scale) -> tuple[np.ndarray, np.ndarray]:
    """C[M, N] = A[M, K] . B[N, K]^T on the dequantised operands, in float64.

    Every GEMM mode reduces to this form once column copies are stored
    transposed: fprop Y = X_row . W_row^T, dgrad dX = dY_row . (W_col^T)^T,
    wgrad dW = dY_col^T . (X_col^T)^T. Returns (ref, S) with S = sum |a*b|.
    """
    A = mx_dequantize(a_codes, a_scale)
    B = mx_dequantize(b_codes, b_scale)
    return A @ B.T, np.abs(A) @ np.abs(B).T


def mx_gemm_ref_entries(a_codes, a_scale, b_codes, b_scale, rows, cols):
    """(ref, S) for selected output entries (i, j) only: one dot per entry."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    A = mx_dequantize(a_codes[rows], a_scale[rows])
    B = mx_dequantize(b_codes[cols], b_scale[cols])
    return np.sum(A * B, axis=1), np.sum(np.abs(A * B), axis=1)


def mx_grouped_gemm_ref_mragged(a_codes, a_scale, b_codes, b_scale, offsets):
    """Grouped fprop/dgrad: rows [off[e], off[e+1]) of A times expert e's B.

    a: [M, K] (row copy), b: [E, N, K] stacked per expert. Returns
    (ref [M, N], S [M, N]); rows of an empty group do not exist.
    ([DSV3] §5.2 routed experts, §13.4 grouped_matmul with group_list.)
    """
    o = np.asarray(offsets, dtype=np.int64)
    E = len(o) - 1
    M = int(o[-1])
    N = b_codes.shape[1]
    ref = np.zeros((M, N))
    S = np.zeros((M, N))
    for e in range(E):
        if o[e + 1] == o[e]:
            continue
        r, s = mx_gemm_ref(a_codes[o[e]:o[e + 1]], a_scale[o[e]:o[e + 1]],
                           b_codes[e], b_scale[e])
        ref[o[e]:o[e + 1]] = r
        S[o[e]:o[e + 1]] = s
    return ref, S


def mx_grouped_gemm_ref_kragged(a_codes, a_scale, b_codes, b_scale, offsets):
    """Grouped wgrad: dW_e = dY_e^T . X_e over group e's token segment.

    a: [N, Kp] = grouped column copy of dY, b: [Kout, Kp] = grouped column copy
    of X, both with the padded segments of ``mx_padded_offsets(offsets)``.
    Returns (ref [E, N, Kout], S). An empty group gives dW_e = 0 exactly (the
    empty sum).
    """
    o = np.asarray(offsets, dtype=np.int64)
    poff = mx_padded_offsets(o)
    E = len(o) - 1
    N, Kout = a_codes.shape[0], b_codes.shape[0]
    ref = np.zeros((E, N, Kout))
    S = np.zeros((E, N, Kout))
    for e in range(E):
        if o[e + 1] == o[e]:
            continue
        k0, k1 = int(poff[e]), int(poff[e + 1])
        r, s = mx_gemm_ref(a_codes[:, k0:k1], a_scale[:, k0 // 32:k1 // 32],
                           b_codes[:, k0:k1], b_scale[:, k0 // 32:k1 // 32])
        ref[e] = r
        S[e] = s
    return ref, S


# ----------------------------------------------------------------------------
# Acceptance
# ----------------------------------------------------------------------------

TOL_REL = 2.0 ** -8
TOL_ABS_S = 1e-6


# ----------------------------------------------------------------------------
# Variant recipe: DeepSeek-V3 blockwise FP8 (1x128 activations, 128x128 weights)
# ----------------------------------------------------------------------------

FP8_BLOCK = 128


def blockwise_scale(amax) -> np.ndarray:
    """Per-block multiplier s = 448 / amax in FP32 ("浮点格式、数值稳定性与混合精度"
    §七.2-§七.3: s = 448 / amax, x~ = fl_E4M3(s * x)); an all-zero block takes
    s = 1 (the page leaves amax = 0 open)."""
    a = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore"):
        s = np.float32(E4M3_MAX) / a
    return np.where(a > 0, s, np.float32(1.0)).astype(np.float32)


def blockwise_encode(x, s) -> np.ndarray:
    """E4M3 codes of fl32(s * x): the product rounded once to FP32, then RNE
    to E4M3 (both sides of the comparison take the decision in FP32)."""
    y = (np.asarray(x, dtype=np.float32) * np.asarray(s, dtype=np.float32)).astype(np.float32)
    return e4m3_encode(y.astype(np.float64))


def quantize_1x128(x) -> tuple[np.ndarray, np.ndarray]:
    """Activation blocks of 1 x 128 along the last dim of x[R, C] (C % 128 == 0).
    Returns codes [R, C] and the FP32 multipliers s [R, C/128]."""
    x = np.asarray(x, dtype=np.float64)
    R, C = x.shape
    assert C % FP8_BLOCK == 0
    b = x.reshape(R, C // FP8_BLOCK, FP8_BLOCK)
    s = blockwise_scale(np.max(np.abs(b), axis=-1))
    codes = blockwise_encode(b, s[..., None])
    return codes.reshape(R, C), s


def quantize_128x128(w) -> tuple[np.ndarray, np.ndarray]:
    """Weight blocks of 128 x 128 over w[N, K] (K % 128 == 0; the last row block
    may be short). Returns codes [N, K] and s [ceil(N/128), K/128]."""
    w = np.asarray(w, dtype=np.float64)
    N, K = w.shape
    assert K % FP8_BLOCK == 0
    nb = (N + FP8_BLOCK - 1) // FP8_BLOCK
    amax = np.zeros((nb, K // FP8_BLOCK))
    for i in range(nb):
        blk = np.abs(w[i * FP8_BLOCK:(i + 1) * FP8_BLOCK]).reshape(-1, K // FP8_BLOCK, FP8_BLOCK)
        amax[i] = blk.max(axis=(0, 2))
    s = blockwise_scale(amax)
    s_rows = np.repeat(s, FP8_BLOCK, axis=0)[:N]
    codes = blockwise_encode(w.reshape(N, K // FP8_BLOCK, FP8_BLOCK), s_rows[..., None]).reshape(N, K)
    return codes, s


def gemm_blockwise_ref(a_codes, a_s, b_codes, b_s) -> tuple[np.ndarray, np.ndarray]:
    """C = sum over 128-K blocks kb of (A_kb . B_kb^T) / (s_a[:, kb] s_b[nb, kb]),
    the promotion of each block's partial sum with its two scales (same page,
    §七.3), in float64. Returns (ref, S) with S = sum |a * b| of the dequantised
    operands."""
    a_codes, b_codes = np.asarray(a_codes), np.asarray(b_codes)
    M, K = a_codes.shape
    N = b_codes.shape[0]
    A = e4m3_decode(a_codes)
    B = e4m3_decode(b_codes)
    sb_rows = np.repeat(np.asarray(b_s, dtype=np.float64), FP8_BLOCK, axis=0)[:N]
    ref = np.zeros((M, N))
    S = np.zeros((M, N))
    for kb in range(K // FP8_BLOCK):
        sl = slice(kb * FP8_BLOCK, (kb + 1) * FP8_BLOCK)
        Ad = A[:, sl] / np.asarray(a_s, dtype=np.float64)[:, kb:kb + 1]
        Bd = B[:, sl] / sb_rows[:, kb:kb + 1]
        ref += Ad @ Bd.T
        S += np.abs(Ad) @ np.abs(Bd).T
    return ref, S


# ----------------------------------------------------------------------------
# Variant recipe: current scaling with one FP32 scale per tensor or per group
# ("DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §3: the FP32 scale of HiF8
# current scaling is a scalar for a dense tensor and one per leading group for
# a grouped tensor, taken from the current tensor's amax; §3.2: scale =
# valid(amax) ? amax / format_max : 1.0 in FP32, dense tensors per tensor, 3-D
# grouped weights per leading group; §8.2: activations and gradients take
# amax and scale at every quantisation, weights after the optimizer step.)
# Here the data format is E4M3, so format_max is E4M3's largest value 448;
# the page's 15 and 224 belong to the HiF8 format, which is not built.
# ----------------------------------------------------------------------------

CURRENT_FORMAT_MAX = E4M3_MAX


def current_amax(x) -> float:
    """amax = max |x| over the whole tensor (NaN propagates)."""
    with np.errstate(invalid="ignore"):
        return float(np.max(np.abs(np.asarray(x, dtype=np.float64))))


def current_scale(amax, format_max: float = CURRENT_FORMAT_MAX) -> np.float32:
    """scale = amax / format_max as an FP32 division when amax is valid
    (finite and above zero), else 1.0."""
    a = np.float32(amax)
    if not (np.isfinite(a) and a > 0):
        return np.float32(1.0)
    return np.float32(a) / np.float32(format_max)


def current_encode(x, scale) -> np.ndarray:
    """E4M3 codes of fl32(x / scale): the quotient rounded once to FP32, then
    to E4M3 (nearest, ties to even, saturating; NaN keeps its sign bit)."""
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        q = (np.asarray(x, dtype=np.float32) / np.float32(scale)).astype(np.float32)
    return e4m3_encode(q.astype(np.float64))


def current_quantize(x, format_max: float = CURRENT_FORMAT_MAX):
    """One tensor (any shape) with its own scale: (codes, scale, amax)."""
    amax = current_amax(x)
    s = current_scale(amax, format_max)
    return current_encode(x, s), s, amax


def current_quantize_groups(w, format_max: float = CURRENT_FORMAT_MAX):
    """Stacked w[E, ...]: each leading group with its own amax and scale.
    Returns (codes [E, ...], scales FP32 [E], amax [E])."""
    w = np.asarray(w, dtype=np.float64)
    out = [current_quantize(w[e], format_max) for e in range(w.shape[0])]
    return (np.stack([o[0] for o in out]), np.array([o[1] for o in out], dtype=np.float32),
            np.array([o[2] for o in out]))


def current_dequantize(codes, scale) -> np.ndarray:
    """Value of each element: its E4M3 value times the FP32 scale."""
    return e4m3_decode(codes) * np.float64(np.float32(scale))


def current_transpose_grouped(codes, offsets) -> np.ndarray:
    """The layout of a grouped column operand: codes [M, D] of rows grouped by
    offsets, transposed to [D, padded] with each group's segment starting at
    the same 128-multiple column as the MX grouped column copy and zero codes
    in the padding (the scale is one per tensor, so only the layout changes)."""
    c = np.asarray(codes, dtype=np.uint8)
    o = np.asarray(offsets, dtype=np.int64)
    poff = mx_padded_offsets(o)
    out = np.zeros((c.shape[1], int(poff[-1])), dtype=np.uint8)
    for e in range(len(o) - 1):
        m = int(o[e + 1] - o[e])
        out[:, poff[e]:poff[e] + m] = c[o[e]:o[e + 1]].T
    return out


def current_gemm_ref(a_codes, a_scale, b_codes, b_scale) -> tuple[np.ndarray, np.ndarray]:
    """C = A . B^T on the dequantised operands in float64, with S = sum |a*b|."""
    A = current_dequantize(a_codes, a_scale)
    B = current_dequantize(b_codes, b_scale)
    return A @ B.T, np.abs(A) @ np.abs(B).T


# ----------------------------------------------------------------------------
# Grouped SwiGLU between gate_up and down (kept in high precision)
# ----------------------------------------------------------------------------

SILU_MAX_SLOPE = 1.1     # max |d/dx x*sigmoid(x)| = 1.0998... (at x ~ 2.40)


def silu(x) -> np.ndarray:
    """x * sigmoid(x) = x / (1 + exp(-x)) in float64 (for x -> -inf the value
    tends to -0, for x -> +inf to x)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        e = np.exp(-x)
    return np.where(np.isinf(e), -0.0 * np.abs(x), x / (1.0 + e))


def swiglu(y) -> np.ndarray:
    """SwiGLU of a gate_up output y[..., 2F]: gate = y[..., :F], up = y[..., F:]
    ("DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §5: gate_up_proj [E, 2F, H],
    gate rows first; the grouped SwiGLU sits between gate_up and down and is not
    a low-precision operator, §1)."""
    y = np.asarray(y, dtype=np.float64)
    F = y.shape[-1] // 2
    assert y.shape[-1] == 2 * F
    return silu(y[..., :F]) * y[..., F:]


def mx_grouped_swiglu_ref(a_codes, a_scale, b_codes, b_scale, offsets):
    """Grouped gate_up fprop followed by SwiGLU, all in float64.

    Returns (out [M, F], gate [M, F], up [M, F], S_gate, S_up): the unrounded
    SwiGLU output, the unrounded gate and up dots and their sum|a*b| terms."""
    ref, S = mx_grouped_gemm_ref_mragged(a_codes, a_scale, b_codes, b_scale, offsets)
    F = ref.shape[1] // 2
    gate, up = ref[:, :F], ref[:, F:]
    return swiglu(ref), gate, up, S[:, :F], S[:, F:]


def swiglu_within_tolerance(out, ref, gate, up, S_gate, S_up) -> np.ndarray:
    """Acceptance for a SwiGLU computed in FP32 from FP32 accumulations and
    rounded once to BF16: each accumulation is within 1e-6 * S of its dot (the
    GEMM bound), so silu(g) * u moves by at most
    SILU_MAX_SLOPE * dg * (|u| + du) + |silu(g)| * du; FP32 evaluation adds
    <= 1e-5 * |out| and the BF16 rounding <= 2**-8 * |out|."""
    out = np.asarray(out, dtype=np.float64)
    dg = TOL_ABS_S * S_gate
    du = TOL_ABS_S * S_up
    bound = (TOL_REL + 1e-5) * np.abs(ref) + SILU_MAX_SLOPE * dg * (np.abs(up) + du) + np.abs(silu(gate)) * du
    return np.abs(out - ref) <= bound


def within_tolerance(out, ref, S) -> np.ndarray:
    """Per-element acceptance |out - ref| <= 2**-8 * |ref| + 1e-6 * S.

    ref is the unrounded float64 dot. Rounding the true value to BF16 moves it
    by at most half a BF16 spacing, which is <= 2**-8 * |ref| (8 significant
    bits), and FP32 accumulation error is covered by the 1e-6 * S term.
    Measuring against an FP64 reference follows [FMT] §八.3. Checking against
    a BF16-rounded ref instead would reject correct results whose exact value
    sits within accumulation error of a BF16 rounding midpoint (those may round
    either way, a one-spacing = up to 2**-7 relative difference).
    """
    out = np.asarray(out, dtype=np.float64)
    return np.abs(out - ref) <= TOL_REL * np.abs(ref) + TOL_ABS_S * S


def within_tolerance_literal(out, ref, S) -> np.ndarray:
    """The same bound measured against BF16(ref); reported, not gated."""
    rb = bf16_round(ref)
    out = np.asarray(out, dtype=np.float64)
    return np.abs(out - rb) <= TOL_REL * np.abs(rb) + TOL_ABS_S * S


def error_report(out, ref, S) -> dict:
    """Layered numeric metrics ([DSV3] §17.3.2: max abs, MSE, NRMSE, cosine,
    non-finite count) next to the acceptance counts."""
    out = np.asarray(out, dtype=np.float64)
    d = out - ref
    nrm = float(np.sqrt(np.mean(ref ** 2))) or 1.0
    denom = float(np.linalg.norm(out) * np.linalg.norm(ref)) or 1.0
    return {
        "n": int(out.size),
        "max_abs": float(np.max(np.abs(d))) if d.size else 0.0,
        "mse": float(np.mean(d ** 2)) if d.size else 0.0,
        "nrmse": float(np.sqrt(np.mean(d ** 2)) / nrm) if d.size else 0.0,
        "cosine": float(np.sum(out * ref) / denom) if d.size else 1.0,
        "nonfinite": int(np.sum(~np.isfinite(out))),
        "fail": int(np.sum(~within_tolerance(out, ref, S))),
        "fail_literal_bf16_ref": int(np.sum(~within_tolerance_literal(out, ref, S))),
    }
