"""Seeded synthetic inputs for the MXFP8 path.

Shared by the tests, ``bench.py`` and the smoke check. This module holds only
random-number generation, shapes and value distributions: none of the
method's arithmetic. Every generator takes an explicit seed and draws from a
counter-based Philox stream (numpy ``Generator(Philox(seed))``); values are
produced in float32 and rounded once to BF16 by torch's CPU conversion.

Shapes stand in for the DeepSeek-V3 16B layers described in
"DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计" §1.1 and §4.1 (dense FFN, MLA
projections, 64 routed experts with top-6 routing); no dataset is involved.
"""

from __future__ import annotations

import numpy as np
import torch

SEED_BASE = 2026  # the design page's ST fixes seed 2026; config i uses 2026 + i


def philox(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed))


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32/float64 array -> contiguous CPU BF16 tensor (RNE by torch)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal_bf16(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    g = philox(seed)
    return to_bf16(g.standard_normal(shape, dtype=np.float32) * np.float32(std))


# ---------------------------------------------------------------------------
# Config 1: single Linear 256x512 plus 64 hand-built blocks
# ---------------------------------------------------------------------------

def hand_blocks() -> torch.Tensor:
    """64 blocks of 32 BF16 values ([64, 32]; row i is block i), eight of each kind:

    0-7   all-zero blocks (+0, -0 and mixed signs)
    8-15  blocks of BF16 subnormals (k * 2**-133)
    16-23 blocks whose small members land in E4M3's subnormal range after scaling
    24-31 blocks holding exact +-448 and other exact E4M3 values
    32-39 blocks whose amax lies in (448, 512), i.e. saturating members
    40-47 N(0,1) blocks with one 1e4 outlier (BF16 1e4 = 9984)
    48-55 blocks of exact rounding midpoints (ties) after scaling
    56-63 extremes: BF16 max, min normal, wide dynamic range, negative amax
    Every value is exactly representable in BF16.
    """
    g = philox(SEED_BASE + 100)
    b = np.zeros((64, 32), dtype=np.float64)
    # 0-7 zeros
    b[1, :] = -0.0
    b[2, ::2] = -0.0
    b[3, 5] = -0.0
    # 8-15 BF16 subnormals: k * 2**-133, k in 1..127
    for i in range(8, 16):
        k = g.integers(1, 128, size=32)
        s = g.choice([-1.0, 1.0], size=32)
        b[i] = s * k * 2.0 ** -133
        if i == 8:
            b[i, :] = 2.0 ** -133        # every member the smallest subnormal
    # 16-23 amax = 2**-3 (or a random normal) with tiny siblings
    for i in range(16, 24):
        amax = 2.0 ** -3 if i < 20 else float(g.uniform(1, 2)) * 2.0 ** int(g.integers(-20, 20))
        b[i] = amax * 2.0 ** -g.integers(9, 19, size=32) * g.choice([-1.0, 1.0], size=32)
        b[i, int(g.integers(0, 32))] = amax
    # 24-31 exact E4M3 values with +-448
    e4 = np.array([(1 + m / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8)])
    e4 = e4[e4 <= 448]
    for i in range(24, 32):
        b[i] = g.choice(e4, size=32) * g.choice([-1.0, 1.0], size=32)
        b[i, 0] = 448.0
        b[i, 1] = -448.0
    # 32-39 amax in (448, 512): BF16 spacing there is 2
    for i in range(32, 40):
        b[i] = np.floor(g.uniform(-448, 448, size=32) / 2) * 2
        b[i, 3] = 450.0 + 8 * (i - 32)              # 450 .. 506
        b[i, 7] = -(452.0 + 2 * (i - 32))
    # 40-47 N(0,1) with one 1e4 outlier
    for i in range(40, 48):
        b[i] = g.standard_normal(32)
        b[i, int(g.integers(0, 32))] = 1e4 if i % 2 == 0 else -1e4
    # 48-55 ties: amax 256 gives scale 1; members at midpoints of E4M3 spacings
    mids = np.array([1.0625, 1.1875, 2.125, 3.75 + 0.125, 0.5 + 1 / 32, 3 * 2.0 ** -10,
                     5 * 2.0 ** -10, 2.0 ** -10, 272.0, 304.0, 336.0, 17.0, 19.0, 0.03125 + 2.0 ** -9])
    for i in range(48, 56):
        b[i] = g.choice(mids, size=32) * g.choice([-1.0, 1.0], size=32)
        b[i, 31] = 256.0 if i % 2 == 0 else -256.0
    # 56-63 extremes
    bf16_max = (2 - 2.0 ** -7) * 2.0 ** 127
    b[56] = g.standard_normal(32)
    b[56, 0] = bf16_max
    b[57] = 2.0 ** -126 * g.choice([-1.0, 1.0], size=32)
    b[58] = g.choice([-1.0, 1.0], size=32) * 2.0 ** g.integers(-60, 60, size=32).astype(np.float64)
    b[59] = -np.abs(g.standard_normal(32))
    b[59, 9] = -300.0
    b[60] = g.standard_normal(32) * 1e-30
    b[61] = g.standard_normal(32) * 1e30
    b[62] = g.choice([-1.0, 1.0], size=32) * 2.0 ** g.integers(-133, 127, size=32).astype(np.float64)
    b[63] = np.arange(32) - 16.0
    t = to_bf16(b)
    return t


def single_linear(seed: int = SEED_BASE + 1, M: int = 256, N: int = 256, K: int = 512):
    """X[M, K], W[N, K] ~ N(0, 1) in BF16 (single MXFP8 Linear fprop)."""
    return {"X": normal_bf16((M, K), seed), "W": normal_bf16((N, K), seed + 7)}


# ---------------------------------------------------------------------------
# Config 2: dense FFN up-projection, fprop + dgrad + wgrad
# ---------------------------------------------------------------------------

def dense_ffn(seed: int = SEED_BASE + 2, M: int = 8192, K: int = 2048, N: int = 10944,
              outlier_channel_frac: float = 0.01, outlier_scale: float = 50.0,
              w_std: float = 0.02):
    """X[M, K] ~ N(0,1) with 1% of channels scaled x50, W[N, K] ~ N(0, 0.02),
    dY[M, N] ~ N(0, 1)."""
    g = philox(seed)
    x = g.standard_normal((M, K), dtype=np.float32)
    n_out = max(1, int(round(outlier_channel_frac * K)))
    ch = g.choice(K, size=n_out, replace=False)
    x[:, ch] *= np.float32(outlier_scale)
    w = g.standard_normal((N, K), dtype=np.float32) * np.float32(w_std)
    dy = g.standard_normal((M, N), dtype=np.float32)
    return {"X": to_bf16(x), "W": to_bf16(w), "dY": to_bf16(dy), "outlier_channels": np.sort(ch)}


# ---------------------------------------------------------------------------
# Config 3: MLA projection set at M = 16384 tokens
# ---------------------------------------------------------------------------

MLA_PROJECTIONS = (("q_down", 2048, 1536), ("kv_down", 2048, 576),
                   ("kv_up", 512, 4096), ("o_proj", 2048, 2048))

# The attention projections of the frozen 16B model configuration itself
# ("DeepSeek-V3 16B FSDP2 MXFP8/HiF8 训练设计", frozen 16B spec: hidden 2048,
# 16 heads, q_lora_rank null, kv_lora_rank 3072, qk_nope / qk_rope head dims
# 64 / 64, v_head_dim 128), with the DeepSeek-V3 attention's projection widths:
# q_proj 2048 -> 16 * (64 + 64), kv_a_proj_with_mqa 2048 -> 3072 + 64,
# kv_b_proj 3072 -> 16 * (64 + 128), o_proj 16 * 128 -> 2048.
MLA_PROJECTIONS_PAGES = (("q_proj", 2048, 2048), ("kv_a_proj_with_mqa", 2048, 3136),
                         ("kv_b_proj", 3072, 3072), ("o_proj", 2048, 2048))


def mla_projection(name: str, seed: int = SEED_BASE + 3, M: int = 16384, pages: bool = False):
    """X[M, K_in] ~ N(0,1), W[N_out, K_in] ~ N(0, 0.02), dY[M, N_out] ~ N(0,1).
    pages: a projection of MLA_PROJECTIONS_PAGES (seeds of their own)."""
    table = MLA_PROJECTIONS_PAGES if pages else MLA_PROJECTIONS
    idx = [p[0] for p in table].index(name)
    _, k_in, n_out = table[idx]
    s = seed * 16 + idx + (8 if pages else 0)
    return {"X": normal_bf16((M, k_in), s), "W": normal_bf16((n_out, k_in), s + 1, 0.02),
            "dY": normal_bf16((M, n_out), s + 2)}


# ---------------------------------------------------------------------------
# Config 4: 64 routed experts, 8192 tokens x top-6 = 49152 rows
# ---------------------------------------------------------------------------

def moe_counts(E: int = 64, total: int = 49152, alpha: float = 1.1, n_zero: int = 4,
               cap: int = 8192, seed: int = SEED_BASE + 4) -> np.ndarray:
    """Rows per expert: p_r ~ r**-alpha over ranks r = 1..E with the n_zero
    lowest ranks emptied, largest-remainder rounding to ``total``, each expert
    capped at ``cap`` (excess moved down the ranks in proportion), then a
    seeded permutation from rank to expert id."""
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** -alpha
    p[E - n_zero:] = 0.0
    p /= p.sum()
    raw = p * total
    c = np.floor(raw).astype(np.int64)
    rem = total - c.sum()
    order = np.argsort(-(raw - c), kind="stable")
    c[order[:rem]] += 1
    for _ in range(E):
        over = c > cap
        if not over.any():
            break
        excess = int((c[over] - cap).sum())
        c[over] = cap
        free = (~over) & (p > 0) & (c < cap)
        w = p * free
        add = np.floor(excess * w / w.sum()).astype(np.int64)
        left = excess - add.sum()
        idx = np.flatnonzero(free)
        add[idx[:left]] += 1
        c += add
    assert c.sum() == total and c.max() <= cap
    perm = philox(seed).permutation(E)
    counts = np.zeros(E, dtype=np.int64)
    counts[perm] = c
    return counts


def offsets_from_counts(counts) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(counts, dtype=np.int64))]).astype(np.int64)


def moe_experts(seed: int = SEED_BASE + 4, E: int = 64, H: int = 2048, F: int = 1408,
                tokens: int = 8192, topk: int = 6, counts=None):
    """Grouped-GEMM inputs for the routed experts (gate_up: N = 2F, K = H;
    down: N = H, K = F). Rows are grouped contiguously by expert."""
    if counts is None:
        counts = moe_counts(E=E, total=tokens * topk, seed=seed)
    M = int(np.sum(counts))
    s = seed * 16
    return {
        "counts": np.asarray(counts, dtype=np.int64),
        "offsets": offsets_from_counts(counts),
        "X": normal_bf16((M, H), s),                       # input to gate_up
        "W_gate_up": normal_bf16((E, 2 * F, H), s + 1, 0.02),
        "dY_gate_up": normal_bf16((M, 2 * F), s + 2),
        "A_down": normal_bf16((M, F), s + 3),              # input to down
        "W_down": normal_bf16((E, H, F), s + 4, 0.02),
        "dY_down": normal_bf16((M, H), s + 5),
    }


# ---------------------------------------------------------------------------
# Config 5: quantiser bandwidth sweep
# ---------------------------------------------------------------------------

QUANT_SWEEP_M = (4096, 8192, 16384, 32768)


def quant_sweep(M: int, C: int = 7168, seed: int = SEED_BASE + 5, frac: float = 0.001,
                scale: float = 1000.0) -> torch.Tensor:
    """[M, C] ~ N(0,1) with 0.1% of entries (seeded positions) scaled x1000."""
    g = philox(seed * 100003 + M)
    x = g.standard_normal((M, C), dtype=np.float32)
    n = int(round(frac * M * C))
    pos = g.choice(M * C, size=n, replace=False)
    x.reshape(-1)[pos] *= np.float32(scale)
    return to_bf16(x)


# ---------------------------------------------------------------------------
# Weight refresh: FP32 master weights (stacked experts or one matrix)
# ---------------------------------------------------------------------------

def fp32_master(shape, seed: int = SEED_BASE + 6, std: float = 0.02, spread: int = 6) -> torch.Tensor:
    """FP32 master weights: N(0, std) with a per-row power-of-two factor in
    [2**-spread, 2**spread] (seeded), kept in FP32 (24-bit mantissas, so most
    values are not BF16 numbers)."""
    g = philox(seed)
    x = g.standard_normal(shape, dtype=np.float32) * np.float32(std)
    rows = int(np.prod(shape[:-1]))
    f = np.exp2(g.integers(-spread, spread + 1, size=rows)).astype(np.float32)
    x = (x.reshape(rows, shape[-1]) * f[:, None]).reshape(shape)
    return torch.from_numpy(np.ascontiguousarray(x))
