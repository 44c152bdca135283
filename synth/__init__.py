"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and rounds them to bf16; it holds none of
the quantization or GEMM arithmetic, so that the oracle and the CUDA library
consume identical inputs without sharing any method code.

Recipe (stated once, used everywhere): numpy ``default_rng(seed)`` draws fp64
samples, which are cast to fp32 and then rounded to bf16 with round-to-nearest
-even (torch's cast). Outliers are planted on exact counts of distinct positions
drawn without replacement. The distributions follow the LLM-layer workloads the
method is evaluated on: activations Student-t (heavy tails), weights N(0, 0.02),
gradients Laplace(0, 1e-3).
"""
from __future__ import annotations

import numpy as np
import torch

# Data seeds are 1000 + workload index; random-sign masks come from seed + 7.
DATA_SEED_BASE = 1000


def bf16_from_f64(a: np.ndarray) -> torch.Tensor:
    """fp64 -> fp32 -> bf16 (round to nearest even), as a CPU torch tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (a view of the same bytes)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def normal(rows: int, cols: int, std: float, seed: int) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return bf16_from_f64(rng.normal(0.0, std, size=(rows, cols)))


def student_t(rows: int, cols: int, df: float, seed: int) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return bf16_from_f64(rng.standard_t(df, size=(rows, cols)))


def laplace(rows: int, cols: int, b: float, seed: int, outlier_frac: float = 0.0,
            outlier_mult: float = 100.0) -> torch.Tensor:
    """Laplace(0, b); optionally round(outlier_frac * n) distinct entries x outlier_mult."""
    rng = np.random.default_rng(seed)
    a = rng.laplace(0.0, b, size=(rows, cols))
    n = int(round(outlier_frac * rows * cols))
    if n:
        idx = rng.choice(rows * cols, size=n, replace=False)
        a.reshape(-1)[idx] *= outlier_mult
    return bf16_from_f64(a)


def normal_outlier_cols(rows: int, cols: int, std: float, n_cols: int, mult: float,
                        seed: int) -> torch.Tensor:
    """N(0, std) with n_cols distinct random columns scaled by mult (outlier channels)."""
    rng = np.random.default_rng(seed)
    a = rng.normal(0.0, std, size=(rows, cols))
    cols_idx = rng.choice(cols, size=n_cols, replace=False)
    a[:, cols_idx] *= mult
    return bf16_from_f64(a)


def sign_mask(seed: int) -> int:
    """A random 32-bit sign mask for the random-sign rotation."""
    return int(np.random.default_rng(seed + 7).integers(0, 2 ** 32, dtype=np.uint64))


def random_codes(rows: int, k: int, seed: int) -> np.ndarray:
    """Uniform random packed 4-bit codes [rows, k/2] (all 16 codes, both nibbles)."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)


def random_scales(rows: int, k: int, seed: int, lo: int = 120, hi: int = 134) -> np.ndarray:
    """Random scale bytes [rows * k/32] in [lo, hi] (flat: valid in any scale layout)."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=rows * (k // 32), dtype=np.uint8)


def uniform_f32(rows: int, cols: int, lo: float, hi: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, size=(rows, cols)).astype(np.float32)


# ----------------------------------------------------------------------------
# Device-side generators for workload-sized inputs (the benchmark). Same
# distributions, drawn with torch's seeded CUDA generator, rounded to bf16 RNE.
# ----------------------------------------------------------------------------

def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def dev_normal(rows: int, cols: int, std: float, seed: int, device) -> torch.Tensor:
    g = _gen(device, seed)
    return (torch.randn(rows, cols, generator=g, device=device) * std).to(torch.bfloat16)


def dev_student_t(rows: int, cols: int, df: float, seed: int, device) -> torch.Tensor:
    """t(df) = Z / sqrt(V / df), Z ~ N(0,1), V ~ chi^2(df) = 2 * Gamma(df/2)."""
    g = _gen(device, seed)
    z = torch.randn(rows, cols, generator=g, device=device)
    # chi^2 with integer df as a sum of df squared normals (df is 3 or 4 here)
    v = torch.zeros(rows, cols, device=device)
    for _ in range(int(df)):
        v.addcmul_(t1 := torch.randn(rows, cols, generator=g, device=device), t1)
    return (z / torch.sqrt(v / df)).to(torch.bfloat16)


def dev_laplace(rows: int, cols: int, b: float, seed: int, device, outlier_frac: float = 0.0,
                outlier_mult: float = 100.0) -> torch.Tensor:
    """Laplace(0, b) by inverse CDF; round(outlier_frac * n) distinct entries x outlier_mult."""
    g = _gen(device, seed)
    # u in (-1/2, 1/2): a draw of exactly 0 would give -1/2 and an infinite value
    u = (torch.rand(rows, cols, generator=g, device=device) - 0.5).clamp_(min=-0.5 + 2.0 ** -25)
    a = -b * torch.sign(u) * torch.log1p(-2.0 * u.abs())
    n = int(round(outlier_frac * rows * cols))
    if n:
        idx = torch.randperm(rows * cols, generator=g, device=device)[:n]
        a.view(-1)[idx] *= outlier_mult
    return a.to(torch.bfloat16)
