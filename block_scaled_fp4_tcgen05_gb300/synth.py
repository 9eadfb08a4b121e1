"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method (no scale, rounding or GEMM
step): it only draws numbers from a seed and stores them as fp32 or as bf16
bit patterns.  Both the CUDA path and the CPU oracle are fed from here.

Workloads follow the GEMM shapes the pages measure (Llama-3-8B layers in the
"quadbit" README, sections "Headline result" and the bf16 speed-up table:
prefill attention 4096^3, ffn-up N=14336, ffn-down K=14336, decode M=128,
square 8192) and the MoE up-projection of the DeepGEMM pull request
("Packed MXFP4 & NVFP4 GEMM + mega-MoE"), with synthetic values:
  activations  N(0, 1) with 1% of entries multiplied by 20 (outliers)
  weights      N(0, 0.02)
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202
MXFP4 = 0
NVFP4 = 1


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal_f32(gen: np.random.Generator, shape, sigma: float = 1.0,
               outlier_p: float = 0.0, outlier_mul: float = 20.0) -> np.ndarray:
    """fp32 N(0, sigma); each entry independently x outlier_mul with prob. outlier_p."""
    x = gen.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma)
    if outlier_p > 0.0:
        mask = gen.random(size=shape, dtype=np.float32) < np.float32(outlier_p)
        x = np.where(mask, x * np.float32(outlier_mul), x).astype(np.float32)
    return np.ascontiguousarray(x, dtype=np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Store fp32 values as bf16 (round to nearest even on the bit pattern).
    Inputs are finite; this is how the synthetic activations are typed."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations_bf16(seed: int, rows: int, cols: int) -> np.ndarray:
    """Activation-like bf16 matrix: N(0,1) with 1% x20 outliers."""
    return f32_to_bf16_bits(normal_f32(rng(seed), (rows, cols), 1.0, 0.01, 20.0))


def weights_bf16(seed: int, rows: int, cols: int) -> np.ndarray:
    """Weight-like bf16 matrix: N(0, 0.02)."""
    return f32_to_bf16_bits(normal_f32(rng(seed), (rows, cols), 0.02))


def norm_weight_bf16(seed: int, cols: int) -> np.ndarray:
    """An RMSNorm weight vector gamma [cols] as bf16: N(1, 0.1)."""
    return f32_to_bf16_bits(normal_f32(rng(seed), (cols,), 0.1) + np.float32(1.0))


def moe_counts(seed: int, tokens: int = 4096, experts: int = 8, topk: int = 2,
               alpha: float = 0.5) -> np.ndarray:
    """Per-expert routed-row counts: p ~ Dirichlet(alpha), counts ~
    Multinomial(tokens * topk, p), redrawn while any expert gets more rows than
    there are tokens (a token reaches one expert at most once)."""
    gen = rng(seed)
    while True:
        p = gen.dirichlet(np.full(experts, alpha))
        counts = gen.multinomial(tokens * topk, p)
        if counts.max() <= tokens:
            return counts.astype(np.int64)


@dataclass(frozen=True)
class GemmCase:
    name: str
    fmt: int
    M: int
    N: int
    K: int
    seed: int
    note: str = ""


@dataclass(frozen=True)
class GroupedCase:
    name: str
    fmt: int
    tokens: int
    experts: int
    topk: int
    N: int
    K: int
    seed: int
    counts: tuple = field(default=())


# The five workloads (index 0 is the small case the oracle finishes at once).
SMALL_MX = GemmCase("mxfp4_gemm_nt_128x256x256", MXFP4, 128, 256, 256, SEED_BASE + 0,
                    "fp32 N(0,1) operands quantized by the oracle")
PREFILL_NV = GemmCase("nvfp4_gemm_nt_4096x4096x4096", NVFP4, 4096, 4096, 4096, SEED_BASE + 1,
                      "prefill attention projection")
DECODE_UP = GemmCase("nvfp4_gemm_nt_128x14336x4096", NVFP4, 128, 14336, 4096, SEED_BASE + 2,
                     "decode ffn-up")
DECODE_ATTN = GemmCase("nvfp4_gemm_nt_128x4096x4096", NVFP4, 128, 4096, 4096, SEED_BASE + 2,
                       "decode attention projection")
QUANT_ROWS, QUANT_COLS, QUANT_SEED = 16384, 4096, SEED_BASE + 2
COMPUTE_SWEEP = tuple(
    GemmCase(f"{'mx' if f == MXFP4 else 'nv'}fp4_gemm_nt_{M}x{N}x{K}", f, M, N, K, SEED_BASE + 3)
    for f in (MXFP4, NVFP4)
    for (M, N, K) in ((4096, 14336, 4096), (4096, 4096, 14336), (8192, 8192, 8192))
)
MOE_UP = GroupedCase("nvfp4_grouped_up_4096tok_top2_8exp", NVFP4, 4096, 8, 2, 14336, 4096,
                     SEED_BASE + 4)
# the square NVFP4 GEMM of the compute sweep (quadbit README, "Headline result": square 8192)
SQUARE_NV = next(c for c in COMPUTE_SWEEP if c.fmt == NVFP4 and c.M == c.N == c.K == 8192)
