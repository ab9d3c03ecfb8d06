"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no arithmetic of the quantisation method: it only draws
Llama-shaped BF16 tensors.  Recipe (as stated for the workloads):

* weights  W[N, K] ~ N(0, 0.02^2); a fraction ``outlier_frac`` (1 %) of the
  input channels (columns k) is multiplied by ``outlier_scale`` (x20);
* activations X[M, K] ~ N(0, 1); optionally a fraction ``token_outlier_frac``
  (0.1 %) of the tokens (rows m) is multiplied by ``token_outlier_scale`` (x50);
* every draw is float32 from ``numpy.random.Generator(PCG64)`` and then
  rounded to bfloat16 (round to nearest, ties to even), returned as the raw
  uint16 bit patterns;
* the outlier index sets come from their own stream, ``SeedSequence([seed, 2])``,
  so that changing the outlier fraction does not change the values drawn.

The number of outlier channels is round(frac * K) (5, 41, 82, 143, 287 for
K = 512, 4096, 8192, 14336, 28672) and of outlier tokens round(frac * M).
"""
from __future__ import annotations

import numpy as np

LLAMA3_8B_LAYERS = {            # (K, N) of the four linear layers of one block
    "qkv": (4096, 6144),
    "o_proj": (4096, 4096),
    "gate_up": (4096, 28672),
    "down": (14336, 4096),
}
LLAMA3_70B_LAYERS = {
    "qkv": (8192, 10240),
    "o_proj": (8192, 8192),
    "gate_up": (8192, 57344),
    "down": (28672, 8192),
}
CROSSOVER_LAYERS = {"up": (4096, 14336), "down": (14336, 4096)}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def outlier_indices(count_of: int, frac: float, seed: int) -> np.ndarray:
    n = int(round(frac * count_of))
    if n == 0:
        return np.zeros((0,), np.int64)
    return np.sort(_rng(seed, 2).permutation(count_of)[:n]).astype(np.int64)


def make_weight(N: int, K: int, seed: int = 0, std: float = 0.02,
                outlier_frac: float = 0.01, outlier_scale: float = 20.0) -> np.ndarray:
    """W[N, K] as bf16 bits: N(0, std^2) with round(frac*K) input channels scaled."""
    w = _rng(seed, 0).standard_normal((N, K), dtype=np.float32)
    w *= np.float32(std)
    idx = outlier_indices(K, outlier_frac, seed)
    if idx.size:
        w[:, idx] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(w)


def make_act(M: int, K: int, seed: int = 1, token_outlier_frac: float = 0.0,
             token_outlier_scale: float = 50.0) -> np.ndarray:
    """X[M, K] as bf16 bits: N(0, 1) with round(frac*M) tokens scaled."""
    x = _rng(seed, 1).standard_normal((M, K), dtype=np.float32)
    idx = outlier_indices(M, token_outlier_frac, seed)
    if idx.size:
        x[idx, :] *= np.float32(token_outlier_scale)
    return f32_to_bf16_bits(x)


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
