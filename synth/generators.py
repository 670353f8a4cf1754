"""Seeded generators of bf16 activations, weights and integer codes.

Every tensor gets its own Philox stream, keyed by (seed, tags...) through
numpy's SeedSequence, so a tensor is reproducible on its own whatever else
was drawn before it.  Values are drawn in float32 and stored as bf16 bit
patterns (uint16), rounded to nearest-even.

Recipes (the workloads of the pages' VLA backbones and action experts):
  * activations: N(0,1) or Student-t(nu=4); a fixed, seeded set of outlier
    channels is multiplied by a constant for every token;
  * weights: N(0, std^2); optionally a Bernoulli-selected fraction of entries
    multiplied by a constant ("spikes").
"""
from __future__ import annotations

import zlib

import numpy as np


def _tag_int(tag) -> int:
    if isinstance(tag, (int, np.integer)):
        return int(tag) & 0xFFFFFFFF
    return zlib.crc32(str(tag).encode("utf-8"))


def sub_rng(seed: int, *tags) -> np.random.Generator:
    """An independent Philox stream for (seed, *tags)."""
    ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF] + [_tag_int(t) for t in tags])
    return np.random.Generator(np.random.Philox(ss))


def f32_to_bf16_bits(a) -> np.ndarray:
    """float32 array -> uint16 bf16 bit patterns, round to nearest even."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def outlier_channels(K: int, n: int, rng: np.random.Generator) -> np.ndarray:
    """n distinct channel indices out of K, chosen by a seeded shuffle."""
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(rng.permutation(K)[:n])


def activations(M: int, K: int, *, dist: str = "normal", n_outliers: int = 0,
                outlier_scale: float = 1.0, seed: int = 0, tags=()) -> np.ndarray:
    """bf16 bits [M, K]: token-major activations with fixed outlier channels."""
    rng = sub_rng(seed, "act", M, K, *tags)
    if dist == "normal":
        x = rng.standard_normal((M, K), dtype=np.float32)
    elif dist == "student_t4":
        z = rng.standard_normal((M, K), dtype=np.float32)
        chi2 = rng.chisquare(4.0, size=(M, K)).astype(np.float32)
        x = z / np.sqrt(chi2 / np.float32(4.0))
    else:
        raise ValueError(f"unknown activation distribution {dist!r}")
    ch = outlier_channels(K, n_outliers, rng)
    if ch.size:
        x[:, ch] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(x)


def weights(N: int, K: int, *, std: float = 0.02, spike_frac: float = 0.0,
            spike_scale: float = 1.0, seed: int = 0, tags=()) -> np.ndarray:
    """bf16 bits [N, K]: nn.Linear-layout weights N(0, std^2) with optional spikes."""
    rng = sub_rng(seed, "w", N, K, *tags)
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)
    if spike_frac > 0.0:
        mask = rng.random((N, K), dtype=np.float32) < np.float32(spike_frac)
        w[mask] *= np.float32(spike_scale)
    return f32_to_bf16_bits(w)


def random_codes(shape, lo: int, hi: int, *, seed: int = 0, tags=()) -> np.ndarray:
    """Uniform integer codes in [lo, hi] (inclusive), int8."""
    rng = sub_rng(seed, "codes", *shape, lo, hi, *tags)
    return rng.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.int8)
