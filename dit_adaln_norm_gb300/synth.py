"""Seeded synthetic inputs for the adaLN row kernels.

This module only draws numbers: it holds none of the normalisation or
modulation arithmetic.  The CUDA path and the CPU oracle consume the same
bytes from it.  bf16 tensors are returned as ``np.uint16`` bit patterns; the
fp32 -> bf16 cast of a drawn value is torch's CPU cast (round to nearest even).

Distributions follow the diffusion sites the kernels serve (FLUX.1 image/text
adaLN sites at hidden 3072, ERNIE-Image at 4096, Qwen-Image packed QKV with 24
heads of 128): activations ~ N(0, 1), adaLN scale/shift drawn as chunks of one
embedding row per batch, LayerNorm activations with 1% outlier channels
scaled x20, per-head norm weights ~ 1 + N(0, 0.05), fp32 RoPE tables with
theta = 10000.
"""
from __future__ import annotations

import numpy as np
import torch

SEED_X = 0          # activations
SEED_VEC = 1        # scale / shift / gate / weights
SEED_OUTLIER = 2    # which channels carry outliers


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (torch's round-to-nearest-even cast)."""
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16(shape, seed: int, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    f = _rng(seed).standard_normal(size=shape) * std + mean
    return to_bf16_bits(f.astype(np.float32))


def outlier_rows_bf16(shape, seed: int, outlier_seed: int, frac: float = 0.01,
                      factor: float = 20.0) -> np.ndarray:
    """N(0, 1) rows where round(frac * D) channels (a seeded permutation) are
    multiplied by ``factor`` before the bf16 cast."""
    D = shape[-1]
    f = _rng(seed).standard_normal(size=shape)
    k = int(round(frac * D))
    ch = _rng(outlier_seed).permutation(D)[:k]
    f[..., ch] *= factor
    return to_bf16_bits(f.astype(np.float32))


def adaln_vectors(B: int, D: int, n: int, seed: int, std: float, chunks: int = 6):
    """``n`` per-batch vectors [B, D] taken as the first ``n`` chunks of one
    embedding row of ``chunks * D`` values per batch (the adaLN projection
    output), so each view has batch stride ``chunks * D``."""
    chunks = max(chunks, n)
    emb = normal_bf16((B, chunks * D), seed, std)
    return [emb[:, i * D:(i + 1) * D] for i in range(n)]


def rope_table(T: int, head_dim: int = 128, theta: float = 10000.0,
               pos0: int = 0) -> np.ndarray:
    """fp32 [T, head_dim] rows [cos_0..cos_{h/2-1} | sin_0..sin_{h/2-1}] for
    positions pos0..pos0+T-1, built in fp64 and rounded once to fp32."""
    half = head_dim // 2
    inv_freq = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / head_dim)
    ang = np.arange(pos0, pos0 + T, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def head_weights(n: int, seed: int, head_dim: int = 128, std: float = 0.05):
    f = 1.0 + _rng(seed).standard_normal(size=(n, head_dim)) * std
    bits = to_bf16_bits(f.astype(np.float32))
    return [bits[i] for i in range(n)]


def packed_qkv(T: int, heads: int, seed: int, head_dim: int = 128) -> np.ndarray:
    """A packed QKV GEMM output [T, 3 * heads * head_dim] ~ N(0, 1); Q, K, V
    are its column slices (zero-copy strided views)."""
    return normal_bf16((T, 3 * heads * head_dim), seed)


def split_qkv(packed: np.ndarray, heads: int, head_dim: int = 128):
    w = heads * head_dim
    return packed[:, :w], packed[:, w:2 * w], packed[:, 2 * w:3 * w]
