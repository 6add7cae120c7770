"""Seeded synthetic weights shaped like the workloads on the pages.

This module only draws inputs: it holds none of the conversion arithmetic,
and both the CUDA path and the CPU oracle receive exactly the bytes it
returns.  Everything is numpy (PCG64) on the host.  bf16 weights are drawn
in fp32 and rounded to bf16 (nearest, ties to even) -- an input recipe, not
a step of the method.

Workloads (TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling
recipes", "Test results (B200)"; TE PR #3790 "export_components",
Description and test list):

* ``exhaustive_bf16``: all 65536 bf16 patterns in ascending order, one 1x32
  block per row (2048 x 32).
* ``partial_block_fp32``: fp32 N(0, 0.02) weights of shapes (100, 48),
  (64, 16), (128, 96), each 1x32 block (the last one may hold 16) scaled by
  2^U{-20..20}.
* ``normal_bf16``: N(0, 0.02) bf16 of any shape (8192 x 8192 is the
  headline weight).
* ``spread_tiles_fp32``: 128x128 tiles of E2M1 grid payloads whose 1x32
  block exponents spread by d ~ U{0..16} around a base 2^U{-120..120}, with
  planted zero, -0 and 2^-127 tiles.
* ``moe_expert_bf16``: one expert of a 32 x 4096 x 7184 stack, N(0, 0.02)
  times 2^U{-8..8} per expert; experts are seeded independently so a test
  can regenerate any one of them.
"""

from __future__ import annotations

import numpy as np

SEED_BASE = 1000  # workload k uses seed 1000 + k

PARTIAL_BLOCK_SHAPES = ((100, 48), (64, 16), (128, 96))
MOE_EXPERTS, MOE_ROWS, MOE_K = 32, 4096, 7184

# Planted tiles of the spread sweep: (tile row, tile col) -> kind
PLANTED_TILES = {(0, 0): "zero", (0, 1): "negzero", (0, 2): "min_subnormal_scale"}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 to bf16 bit patterns (nearest, ties to even)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def exhaustive_bf16() -> np.ndarray:
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(2048, 32)


def partial_block_fp32(shape, seed: int = SEED_BASE + 2) -> np.ndarray:
    rows, K = shape
    g = rng(seed * 1000 + rows * 7 + K)
    w = (g.standard_normal((rows, K), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    nb = (K + 31) // 32
    k = g.integers(-20, 21, size=(rows, nb))
    mult = np.ldexp(np.float32(1.0), k).astype(np.float32)
    w *= np.repeat(mult, 32, axis=1)[:, :K]
    return w


def normal_bf16(rows: int, K: int, seed: int = SEED_BASE + 3, std: float = 0.02) -> np.ndarray:
    g = rng(seed)
    out = np.empty((rows, K), dtype=np.uint16)
    step = max(1, (1 << 24) // max(K, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        out[r0:r1] = f32_to_bf16_bits(g.standard_normal((r1 - r0, K), dtype=np.float32) * np.float32(std))
    return out


E2M1_SIGNED = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0, 0.0, -0.0],
                       dtype=np.float32)


def spread_tiles_fp32(rows: int = 8192, K: int = 8192, seed: int = SEED_BASE + 4, max_spread: int = 16):
    """(weights, per-tile spread d).  Payloads are uniform over the 15 signed
    grid values plus -0; block exponents are base - U{0..d}, with one block
    at base and one at base - d in every tile."""
    g = rng(seed)
    tr, tc = rows // 128, K // 128
    d = g.integers(0, max_spread + 1, size=(tr, tc))
    base = g.integers(-120, 121, size=(tr, tc))
    nbt = 128 * 4  # 1x32 blocks per tile
    off = g.integers(0, 1 << 30, size=(tr, tc, nbt)) % (d[..., None] + 1)
    off[..., 0] = 0
    off[..., 1] = d
    gexp = base[..., None] - off  # (tr, tc, 512)
    pay = E2M1_SIGNED[g.integers(0, 16, size=(tr, tc, 128, 128))]
    # block (ti, tj, r, b) covers columns 32b..32b+31 of tile row r
    gexp = gexp.reshape(tr, tc, 128, 4)
    mult = np.ldexp(np.float64(1.0), np.repeat(gexp, 32, axis=3))
    w = (pay.astype(np.float64) * mult).astype(np.float32)
    w = w.transpose(0, 2, 1, 3).reshape(rows, K)
    for (ti, tj), kind in PLANTED_TILES.items():
        if ti < tr and tj < tc:
            t = w[ti * 128:(ti + 1) * 128, tj * 128:(tj + 1) * 128]
            if kind == "zero":
                t[:] = 0.0
            elif kind == "negzero":
                t[:] = -0.0
            else:
                t[:] = np.float32(np.ldexp(1.0, -127))
                t[1::2] = -t[1::2]
    return np.ascontiguousarray(w), d


def moe_expert_bf16(expert: int, rows: int = MOE_ROWS, K: int = MOE_K, seed: int = SEED_BASE + 5) -> np.ndarray:
    g = rng(seed * 1000 + expert)
    k = int(g.integers(-8, 9))
    w = g.standard_normal((rows, K), dtype=np.float32) * np.float32(0.02 * 2.0 ** k)
    return f32_to_bf16_bits(w)
