"""Seeded synthetic inputs shaped like the workloads of the MXFP4 dense linear.

This module draws random numbers and builds bit patterns; it holds none of
the method's arithmetic (no quantization, no dequantization, no products).
Both the CUDA path and the CPU oracle consume exactly the arrays made here.

Every tensor gets its own independent stream: ``numpy.random.Generator``
(PCG64) seeded with ``SeedSequence([seed, tensor_id])``.

Recipes (stand-ins for the pages' model checkpoints, which are not available):

* activations: N(0, 1) in float32, rounded to bfloat16; optionally a seeded
  1% of the K-columns multiplied by 20 before rounding (outlier channels);
* weights: FP4 codes uniform over all 16 nibbles (two per byte), E8M0 scale
  bytes 127 + U{lo..hi};
* bias: N(0, 0.1) rounded to bfloat16;
* RMSNorm weights: uniform in [0.25, 2) rounded to bfloat16; residual
  stream: N(0, 16) rounded to bfloat16;
* edge rows: all +0, all -0, blocks whose largest magnitude is exactly 2**k or
  the bfloat16 just below it, blocks holding every rounding tie, blocks with
  values in (6, 8) times a power of two, and blocks of bfloat16 subnormals.
"""

from __future__ import annotations

import numpy as np
import torch

BLOCK = 32


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 data to bfloat16 (torch's CPU conversion) and return the bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    """CPU bfloat16 tensor viewing a uint16 bit array."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def activations(M: int, K: int, seed: int, tensor_id: int = 1,
                outlier_frac: float = 0.0, outlier_scale: float = 20.0) -> np.ndarray:
    """bf16 bits [M, K] of N(0,1) samples, with optional outlier columns."""
    g = rng(seed, tensor_id)
    x = g.standard_normal((M, K), dtype=np.float32)
    if outlier_frac > 0.0:
        n_out = int(round(outlier_frac * K))
        cols = g.choice(K, size=n_out, replace=False)
        x[:, cols] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(x)


def weight_codes(N: int, K: int, seed: int, tensor_id: int = 2, batch: int | None = None) -> np.ndarray:
    """Uniform random packed FP4 bytes [N, K//2] (or [batch, N, K//2])."""
    shape = (N, K // 2) if batch is None else (batch, N, K // 2)
    return rng(seed, tensor_id).integers(0, 256, size=shape, dtype=np.uint8)


def weight_scales(N: int, K: int, lo: int, hi: int, seed: int, tensor_id: int = 3,
                  batch: int | None = None) -> np.ndarray:
    """E8M0 bytes 127 + U{lo..hi}, shape [N, ceil(K/32)] (or batched)."""
    nb = -(-K // BLOCK)
    shape = (N, nb) if batch is None else (batch, N, nb)
    u = rng(seed, tensor_id).integers(lo, hi + 1, size=shape)
    return (127 + u).astype(np.uint8)


def bias(N: int, seed: int, tensor_id: int = 4, sigma: float = 0.1) -> np.ndarray:
    g = rng(seed, tensor_id)
    return f32_to_bf16_bits(g.standard_normal(N, dtype=np.float32) * np.float32(sigma))


def norm_gamma(K: int, seed: int, tensor_id: int = 7) -> np.ndarray:
    """bf16 bits [K] of RMSNorm weights, uniform in [0.25, 2)."""
    return f32_to_bf16_bits(rng(seed, tensor_id).uniform(0.25, 2.0, K).astype(np.float32))


def residual(M: int, K: int, seed: int, tensor_id: int = 8, sigma: float = 4.0) -> np.ndarray:
    """bf16 bits [M, K] of a residual stream, N(0, sigma^2)."""
    return f32_to_bf16_bits(rng(seed, tensor_id).standard_normal((M, K), dtype=np.float32) * np.float32(sigma))


def bmm_activations(B: int, M: int, K: int, seed: int, tensor_id: int = 5) -> np.ndarray:
    g = rng(seed, tensor_id)
    return f32_to_bf16_bits(g.standard_normal((B, M, K), dtype=np.float32))


# --------------------------------------------------------------------------
# structured edge rows
# --------------------------------------------------------------------------
def _pow2_bits(k: int) -> int:
    """bfloat16 bit pattern of 2**k for k in [-133, 127]."""
    if k >= -126:
        return (k + 127) << 7
    return 1 << (k + 133)           # subnormal: one quantum of 2**-133 shifted


def _block_pow2(g: np.random.Generator, k: int, just_below: bool) -> np.ndarray:
    """A block whose largest magnitude is 2**k (or the bf16 just below it)."""
    top = _pow2_bits(k) - (1 if just_below else 0)
    top_val = np.float32(np.array([top << 16], dtype=np.uint32).view(np.float32)[0])
    vals = (g.uniform(-1.0, 1.0, BLOCK) * float(top_val) * 0.9).astype(np.float32)
    bits = f32_to_bf16_bits(vals)
    pos = g.integers(0, BLOCK)
    bits[pos] = top | (0x8000 if g.integers(0, 2) else 0)
    return bits


def _block_ties(E: int) -> np.ndarray:
    """Largest magnitude 4 * 2**E plus every rounding tie t * 2**E (both signs)."""
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    vals = [4.0] + ties + [-t for t in ties] + [0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0 * 0.5, -4.0]
    vals = (vals + [0.0] * BLOCK)[:BLOCK]
    return f32_to_bf16_bits(np.ldexp(np.array(vals, dtype=np.float64), E).astype(np.float32))


def _block_saturating(E: int) -> np.ndarray:
    """Values in (6, 8) * 2**E, which fall beyond the largest code 6."""
    vals = [6.5, 7.0, 7.5, 7.96875, -6.25, -7.25, 6.125, -7.96875]
    vals = (vals * 4)[:BLOCK]
    return f32_to_bf16_bits(np.ldexp(np.array(vals, dtype=np.float64), E).astype(np.float32))


def _block_subnormal(g: np.random.Generator) -> np.ndarray:
    mant = g.integers(1, 0x80, size=BLOCK, dtype=np.uint16)
    sign = (g.integers(0, 2, size=BLOCK).astype(np.uint16) << 15).astype(np.uint16)
    return (mant | sign).astype(np.uint16)


def edge_rows(K: int, seed: int, tensor_id: int = 6) -> list[np.ndarray]:
    """Rows of bf16 bits (length K) built from the structured edge blocks."""
    g = rng(seed, tensor_id)
    nb = -(-K // BLOCK)
    zeros = np.zeros(K, dtype=np.uint16)
    negzeros = np.full(K, 0x8000, dtype=np.uint16)
    patterns = []
    for k in (-130, -20, 0, 5, 100):
        patterns.append(_block_pow2(g, k, False))
        patterns.append(_block_pow2(g, k, True))
    for E in (-3, 0, 7):
        patterns.append(_block_ties(E))
        patterns.append(_block_saturating(E))
    patterns.append(_block_subnormal(g))
    rows = [zeros, negzeros]
    for shift in range(3):
        row = np.concatenate([patterns[(b + shift * 7) % len(patterns)] for b in range(nb)])
        rows.append(row[:K].copy())
    return rows


def with_edge_rows(x_bits: np.ndarray, seed: int) -> np.ndarray:
    """Copy of ``x_bits`` [M, K] with edge rows placed at first/middle/last and spread rows."""
    M, K = x_bits.shape
    out = x_bits.copy()
    rows = edge_rows(K, seed)
    positions = sorted(set([0, M // 2, M - 1] + [i * M // len(rows) for i in range(len(rows))]))
    for idx, p in enumerate(positions):
        out[p] = rows[idx % len(rows)]
    return out
