"""Seeded synthetic inputs for the Q4_K hot path.

This module is shared by the tests, the benchmark and the smoke check; it holds
no arithmetic of the method (no dequantization, no dot products).  It only
draws bytes and numbers with numpy's published bit generators (PCG64 seeded
through SeedSequence), so the CUDA path and the CPU oracle always consume the
very same buffers.

Weight recipe (one Q4_K super-block = 144 bytes, 256 weights):
  bytes 0-1  d    : uniform float in [d_lo, d_hi], rounded to binary16 (RNE)
  bytes 2-3  dmin : same distribution, independent
  bytes 4-143     : uniform random bytes.
The last 140 bytes hold the eight 6-bit scales, eight 6-bit mins and 256 4-bit
quants; every bit of them belongs to exactly one of those fields, so uniform
bytes are exactly "scales and mins uniform on 0..63, quants uniform on 0..15".
(A test decodes generated blocks with the oracle and checks these marginals.)
"""
from __future__ import annotations

import numpy as np

QK = 256
QBYTES = 144

# Matrix ids used to derive independent streams per (layer, matrix).
QWEN_MATRICES = ("q", "k", "v", "o", "gate", "up", "down")


def rng(*tags: int) -> np.random.Generator:
    """Independent PCG64 stream for a tuple of integer tags."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(t) & 0xFFFFFFFF for t in tags])))


def q4k_weights(N: int, K: int, seed, d_lo: float = 2e-4, d_hi: float = 2e-3) -> np.ndarray:
    """Random Q4_K matrix, uint8 [N, K/256*144] (row-major, block-contiguous rows)."""
    assert K % QK == 0 and K > 0 and N >= 0
    nb = K // QK
    g = rng(*(seed if isinstance(seed, tuple) else (seed,)))
    nblk = N * nb
    out = np.empty((nblk, QBYTES), np.uint8)
    if nblk:
        raw = g.bit_generator.random_raw((nblk * 140 + 7) // 8)
        out[:, 4:] = raw.view(np.uint8)[: nblk * 140].reshape(nblk, 140)
        d = g.uniform(d_lo, d_hi, size=nblk).astype(np.float16)
        dm = g.uniform(d_lo, d_hi, size=nblk).astype(np.float16)
        out[:, 0:2] = d.view(np.uint8).reshape(nblk, 2)
        out[:, 2:4] = dm.view(np.uint8).reshape(nblk, 2)
    return out.reshape(N, nb * QBYTES)


Q6BYTES = 210


def q6k_weights(N: int, K: int, seed, d_lo: float = 2e-4, d_hi: float = 2e-3) -> np.ndarray:
    """Random Q6_K matrix, uint8 [N, K/256*210]: uniform bytes for the 6-bit
    codes and the int8 scales (all signs), d ~ U[d_lo, d_hi] rounded to fp16."""
    assert K % QK == 0 and K > 0 and N >= 0
    nb = K // QK
    g = rng(*(seed if isinstance(seed, tuple) else (seed,)))
    nblk = N * nb
    out = np.empty((nblk, Q6BYTES), np.uint8)
    if nblk:
        raw = g.bit_generator.random_raw((nblk * 208 + 7) // 8)
        out[:, :208] = raw.view(np.uint8)[: nblk * 208].reshape(nblk, 208)
        d = g.uniform(d_lo, d_hi, size=nblk).astype(np.float16)
        out[:, 208:210] = d.view(np.uint8).reshape(nblk, 2)
    return out.reshape(N, nb * Q6BYTES)


def normal_f32(shape, seed) -> np.ndarray:
    """N(0, 1) float32 samples."""
    g = rng(*(seed if isinstance(seed, tuple) else (seed,)))
    return g.standard_normal(size=shape, dtype=np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    nan = np.isnan(np.asarray(a, np.float32))
    r = np.where(nan, 0x7FC0, r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16_bits(shape, seed) -> np.ndarray:
    """N(0, 1) samples rounded to bfloat16, as uint16 bit patterns."""
    return f32_to_bf16_bits(normal_f32(shape, seed))


def qwen25_7b_shapes(hidden: int = 3584, kv: int = 512, ffn: int = 18944):
    """(name, N, K) of the seven Q4_K matrices of one Qwen2.5-7B-shaped layer."""
    return [("q", hidden, hidden), ("k", kv, hidden), ("v", kv, hidden), ("o", hidden, hidden),
            ("gate", ffn, hidden), ("up", ffn, hidden), ("down", hidden, ffn)]


def llama3_8b_prefill_shapes():
    """(name, N, K) of the Llama-3-8B-shaped prefill matrices."""
    return [("sq", 4096, 4096), ("kv", 1024, 4096), ("ffn_up", 14336, 4096), ("ffn_down", 4096, 14336)]


def qwen_layer_weights(layer: int, base_seed: int = 0):
    """Seeded weights of one Qwen2.5-7B-shaped layer: list of (name, N, K, W)."""
    out = []
    for mid, (name, N, K) in enumerate(qwen25_7b_shapes()):
        out.append((name, N, K, q4k_weights(N, K, (base_seed, 1, layer, mid))))
    return out


def plant_row(W: np.ndarray, row: int, block_row: np.ndarray) -> np.ndarray:
    """Copy of W with one row replaced by the given encoded blocks."""
    W2 = W.copy()
    W2[row] = block_row
    return W2
