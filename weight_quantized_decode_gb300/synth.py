"""Seeded synthetic inputs shaped like the pages' decode workloads.

This module only draws random numbers and lays them out as GGUF blocks; it
holds none of the dequantise/dot arithmetic.  The tests, the oracle runs and
the benchmark all take their inputs from here.

Value distributions (the configurations the library is measured on):
  * Q4_0: codes uniform in 0..15 (every qs byte uniform in 0..255), per-32
    fp16 scale d uniform in [0.005, 0.02];
  * Q8_0: int8 codes uniform in -127..127, per-32 fp16 scale in [0.001, 0.01];
  * plain 2-bit: codes uniform in 0..3 (every code byte uniform), per-32 fp16
    scale in [0.01, 0.04];
  * activations: fp16 (or fp32) N(0, 1); optional plants of large values
    (+-20000..60000 in ~1 % of entries, like real down_proj inputs) or of tiny
    ones (~1e-4), as in volta-kernel-bakeoff, "A few tokens at once".
"""
from __future__ import annotations

import zlib

import numpy as np

Q4_0 = "q4_0"
Q8_0 = "q8_0"
Q2W = "q2w"
BLOCK = 32
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q2W: 10}


def seed_for(name: str, copy: int = 0) -> int:
    """Deterministic seed for a named workload and copy index."""
    return (zlib.crc32(name.encode()) + 1000003 * copy) & 0x7FFFFFFF


def row_bytes(fmt: str, K: int) -> int:
    return (K // BLOCK) * BLOCK_BYTES[fmt]


def _scales(rng: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float16)


def q4_0_weights(N: int, K: int, seed: int, d_lo: float = 0.005, d_hi: float = 0.02) -> np.ndarray:
    """GGUF Q4_0 bytes for an N x K matrix: uint8 array [N, K/32*18]."""
    assert K % BLOCK == 0
    rng = np.random.Generator(np.random.PCG64(seed))
    nb = K // BLOCK
    blocks = np.empty((N, nb, 18), dtype=np.uint8)
    d = _scales(rng, (N, nb), d_lo, d_hi)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)   # little-endian fp16
    blocks[:, :, 2:18] = rng.integers(0, 256, size=(N, nb, 16), dtype=np.uint8)
    return blocks.reshape(N, nb * 18)


def q8_0_weights(N: int, K: int, seed: int, d_lo: float = 0.001, d_hi: float = 0.01) -> np.ndarray:
    """GGUF Q8_0 bytes for an N x K matrix: uint8 array [N, K/32*34]."""
    assert K % BLOCK == 0
    rng = np.random.Generator(np.random.PCG64(seed))
    nb = K // BLOCK
    blocks = np.empty((N, nb, 34), dtype=np.uint8)
    d = _scales(rng, (N, nb), d_lo, d_hi)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    codes = rng.integers(-127, 128, size=(N, nb, 32), dtype=np.int16).astype(np.int8)
    blocks[:, :, 2:34] = codes.view(np.uint8)
    return blocks.reshape(N, nb * 34)


def q2w_weights(N: int, K: int, seed: int, d_lo: float = 0.01, d_hi: float = 0.04) -> np.ndarray:
    """Plain 2-bit bytes (fp16 d, then 8 code bytes per 32 weights) for an N x K
    matrix: uint8 array [N, K/32*10]."""
    assert K % BLOCK == 0
    rng = np.random.Generator(np.random.PCG64(seed))
    nb = K // BLOCK
    blocks = np.empty((N, nb, 10), dtype=np.uint8)
    d = _scales(rng, (N, nb), d_lo, d_hi)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(N, nb, 2)
    blocks[:, :, 2:10] = rng.integers(0, 256, size=(N, nb, 8), dtype=np.uint8)
    return blocks.reshape(N, nb * 10)


def weights(fmt: str, N: int, K: int, seed: int) -> np.ndarray:
    if fmt == Q4_0:
        return q4_0_weights(N, K, seed)
    if fmt == Q8_0:
        return q8_0_weights(N, K, seed)
    if fmt == Q2W:
        return q2w_weights(N, K, seed)
    raise ValueError(fmt)


def activations(M: int, K: int, seed: int, plant: str | None = None, dtype=np.float16) -> np.ndarray:
    """Activations [M, K], N(0,1), with optional 'large' or 'tiny' plants; fp16
    by default, or the same draws rounded to fp32 (dtype=np.float32)."""
    rng = np.random.Generator(np.random.PCG64(seed ^ 0x5A5A5A5A))
    x = rng.standard_normal((M, K))
    if plant == "large":
        mask = rng.random((M, K)) < 0.01
        mag = rng.uniform(20000.0, 60000.0, size=(M, K))
        sign = np.where(rng.random((M, K)) < 0.5, -1.0, 1.0)
        x = np.where(mask, sign * mag, x)
    elif plant == "tiny":
        x = x * 1e-4
    elif plant is not None:
        raise ValueError(plant)
    return x.astype(dtype)


def expert_indices(n_calls: int, n_slots: int, n_experts: int, seed: int) -> np.ndarray:
    """Per call, n_slots distinct expert indices drawn uniformly: int32 [n_calls, n_slots]."""
    rng = np.random.Generator(np.random.PCG64(seed ^ 0x3C3C3C3C))
    out = np.empty((n_calls, n_slots), dtype=np.int32)
    for c in range(n_calls):
        out[c] = rng.choice(n_experts, size=n_slots, replace=False)
    return out
