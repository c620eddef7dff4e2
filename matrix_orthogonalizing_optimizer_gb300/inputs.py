"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle's checks.

This module generates numbers only. It holds none of the method's arithmetic (no
normalisation, no Newton-Schulz, no momentum): the same arrays feed the CUDA path and the
CPU oracle, so both sides see bit-identical inputs.

Storage type of the hot path is bfloat16. `round_to_bf16_bits` turns float values into bf16
bit patterns (round to nearest even) once, at generation time; both sides then decode the
same bits.

Distributions follow the workloads the Dion3 paper and its companion pages use:
  * i.i.d. N(0,1) entries scaled by 1/sqrt(cols) (dense projections, gradient-like);
  * Student-t with nu=4 (heavy-tailed MoE expert gradients), then Frobenius-normalised;
  * an exponentially decaying spectrum sigma_i = 10^(-3 i/(n-1)) with random orthonormal
    singular vectors (the 128x512 synthetic matrix of Dion3 appendix B.1.1; the decay rate
    is not printed there, this one is chosen).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng",
    "gaussian",
    "student_t",
    "exp_spectrum",
    "round_to_bf16_bits",
    "bf16_bits_to_f32",
    "bf16_round",
]


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """Independent generator for (seed, stream): one stream per tensor of a workload."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def gaussian(seed: int, shape, scale: float = 1.0, stream: int = 0) -> np.ndarray:
    """float64 array of N(0, scale^2) entries."""
    return rng(seed, stream).standard_normal(size=shape) * scale


def student_t(seed: int, shape, nu: int = 4, stream: int = 0) -> np.ndarray:
    """float64 Student-t(nu) entries built as Z / sqrt(chi2_nu / nu), chi2 from nu squared normals."""
    g = rng(seed, stream)
    z = g.standard_normal(size=shape)
    chi2 = np.zeros(shape)
    for _ in range(nu):
        chi2 += g.standard_normal(size=shape) ** 2
    return z / np.sqrt(chi2 / nu)


def exp_spectrum(seed: int, n: int, m: int, decades: float = 3.0, stream: int = 0) -> np.ndarray:
    """n x m (n <= m) float64 matrix U diag(sigma) V^T with sigma_i = 10^(-decades*i/(n-1))."""
    assert n <= m
    g = rng(seed, stream)
    u, _ = np.linalg.qr(g.standard_normal(size=(n, n)))
    v, _ = np.linalg.qr(g.standard_normal(size=(m, n)))
    sigma = 10.0 ** (-decades * np.arange(n) / max(n - 1, 1))
    return (u * sigma) @ v.T


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of x (rounded to float32 first, then to bf16 by round-to-nearest-even)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    is_nan = np.isnan(f)
    rounding_bias = ((u >> 16) & 1) + 0x7FFF
    r = ((u + rounding_bias) >> 16).astype(np.uint16)
    r[is_nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """float32 values of bf16 bit patterns (exact)."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float64 copy of x after one rounding to bf16 (the value the GPU receives)."""
    return bf16_bits_to_f32(round_to_bf16_bits(x)).astype(np.float64)
