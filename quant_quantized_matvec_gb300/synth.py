"""Seeded synthetic inputs for the K-quant matvec.

This module is the one piece both the CUDA path's tests/benchmark and the CPU
oracle consume.  It holds no dequantization or matvec arithmetic: it only
fills byte buffers with random values at the field offsets the block layouts
fix ("Chapter 6 - The kquant family on the reference lane", Figures 6.2, 6.4
and 6.5) and draws f32 activations.

Recipe (the synthetic stand-in for the Muse Glimmer weights the pages
measure, which are not available):
  * Q4_K / Q5_K blocks: every byte uniform random, then d and dmin (bytes 0..3)
    overwritten with f16 values drawn from U[1e-3, 1e-2] and rounded to f16
    (round to nearest even).  Twelve uniform scale bytes give uniform 6-bit
    scales and mins; qs (and Q5_K's qh) stay uniform random.
  * Q6_K blocks: ql and qh uniform random, the sixteen int8 sub-block scales
    (bytes 192..207) uniform on {-32..31}, d (bytes 208..209) f16 from
    U[1e-3, 1e-2].
  * activations: f32 from N(0, 1), shape [ntok, cols].
Generators are numpy PCG64 seeded from a CRC-32 of a text label, so every run
on every machine produces the same bytes.
"""
from __future__ import annotations

import zlib

import numpy as np

Q4_K, Q5_K, Q6_K = 12, 13, 14
BLOCK_BYTES = {Q4_K: 144, Q5_K: 176, Q6_K: 210}
FMT_NAMES = {Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K"}
FMT_BY_NAME = {v: k for k, v in FMT_NAMES.items()}


def seed_of(label: str) -> int:
    """Stable 32-bit seed for a text label (CRC-32)."""
    return zlib.crc32(label.encode("utf-8")) & 0xFFFFFFFF


def _rng(seed) -> np.random.Generator:
    if isinstance(seed, str):
        seed = seed_of(seed)
    return np.random.Generator(np.random.PCG64(int(seed)))


def _f16_bits(values: np.ndarray) -> np.ndarray:
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(
        np.uint16)


def row_bytes(fmt: int, cols: int) -> int:
    return cols // 256 * BLOCK_BYTES[fmt]


def kquant_matrix(fmt: int, rows: int, cols: int, seed) -> np.ndarray:
    """A row-major [rows, row_bytes] uint8 matrix of random super-blocks."""
    if cols % 256 != 0 or cols <= 0 or rows <= 0:
        raise ValueError("cols must be a positive multiple of 256")
    bb = BLOCK_BYTES[fmt]
    nblk = rows * (cols // 256)
    rng = _rng(seed)
    W = rng.integers(0, 256, size=nblk * bb, dtype=np.uint8)
    blocks = W.reshape(nblk, bb)
    if fmt in (Q4_K, Q5_K):
        hdr = _f16_bits(rng.uniform(1e-3, 1e-2, size=(nblk, 2)))
        blocks[:, 0:4] = hdr.view(np.uint8).reshape(nblk, 4)
    elif fmt == Q6_K:
        sc = rng.integers(-32, 32, size=(nblk, 16), dtype=np.int8)
        blocks[:, 192:208] = sc.view(np.uint8)
        d = _f16_bits(rng.uniform(1e-3, 1e-2, size=nblk))
        blocks[:, 208:210] = d.view(np.uint8).reshape(nblk, 2)
    else:
        raise ValueError(f"unknown format {fmt}")
    return W.reshape(rows, cols // 256 * bb)


def activations(ntok: int, cols: int, seed) -> np.ndarray:
    """x ~ N(0, 1) as f32, shape [ntok, cols]."""
    rng = _rng(seed)
    return rng.standard_normal((ntok, cols)).astype(np.float32)
