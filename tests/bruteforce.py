"""Exact-rational brute force of the MXFP4 projection, used to pin the oracle.

Independent of the oracle's formulation: values are exact Fractions, the
scale exponent is the smallest integer e with amax <= 6 * 2^e (the
definition of ceil(log2(amax/6))), and each element takes the nearest of
the eight grid points times 2^e by exhaustive comparison, ties to the even
code (TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling
recipes", Description, mode 1).  Pure Python: small inputs only.
"""

import math
import struct
from fractions import Fraction

GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def bf16_to_float(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (b & 0xFFFF) << 16))[0]


def f32_bits_to_float(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def float_to_f32_bits(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def ceil_log2_over6(amax: Fraction) -> int:
    """Smallest integer e with amax <= 6 * 2^e (amax > 0)."""
    e = math.frexp(float(amax))[1] - 5
    while Fraction(6) * Fraction(2) ** e < amax:
        e += 1
    while Fraction(6) * Fraction(2) ** (e - 1) >= amax:
        e -= 1
    return e


def scale_exponent(amax: Fraction) -> int:
    if amax == 0:
        return -126
    return max(-126, min(125, ceil_log2_over6(amax)))


def nearest_grid(a: Fraction, e: int) -> Fraction:
    s = Fraction(2) ** e
    best = min(range(8), key=lambda c: (abs(a - GRID[c] * s), c % 2))
    return GRID[best] * s


def project_block(values):
    """values: Python floats of one block.  Returns projected floats or None
    when the block holds a NaN or an Inf."""
    if any(math.isnan(v) or math.isinf(v) for v in values):
        return None
    amax = max(Fraction(abs(v)) for v in values)
    e = scale_exponent(amax)
    out = []
    for v in values:
        y = float(nearest_grid(Fraction(abs(v)), e))
        out.append(math.copysign(y, v))
    return out


def project_bf16_rows(rows_bits):
    """rows_bits: list of lists of bf16 patterns (one block per list)."""
    res = []
    for blk in rows_bits:
        vals = [bf16_to_float(b) for b in blk]
        y = project_block(vals)
        if y is None:
            res.append([0x7FC0] * len(blk))
            continue
        row = []
        for v in y:
            u = float_to_f32_bits(v)
            assert u & 0xFFFF == 0
            row.append(u >> 16)
        res.append(row)
    return res


def project_f32_rows(rows_bits, block=32):
    """rows_bits: list of lists of fp32 patterns; blocks of 32 along each row."""
    res = []
    for rb in rows_bits:
        out = []
        for j0 in range(0, len(rb), block):
            blk = rb[j0:j0 + block]
            vals = [f32_bits_to_float(u) for u in blk]
            y = project_block(vals)
            if y is None:
                out.extend([0x7FC00000] * len(blk))
            else:
                out.extend(float_to_f32_bits(v) for v in y)
        res.append(out)
    return res
