"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties an oracle function to something it does not compute itself:
numbers the pages print (fixtures under tests/golden/, each cited), exact
rational brute force, closed forms, or a library conversion (torch's fp8,
e8m0 and bf16 casts on the CPU).
"""

import math
import struct

import numpy as np
import pytest
import torch

import oracle
from block_scaled_precision_x32_gb300 import synthetic as syn
from tests import bruteforce as bf
from tests.golden_io import kv, rows

BF16, FP32 = oracle.BF16, oracle.FP32


# ------------------------------------------------------------ scale rule

def test_block_exponent_every_bf16_amax():
    """e = clamp(ceil(log2(amax/6)), -126, 125) for every finite bf16 amax
    (TE PR #3264, Description, mode 1), against the exact definition."""
    from fractions import Fraction
    for b in range(0, 0x7F80):
        want = bf.scale_exponent(Fraction(bf.bf16_to_float(b)))
        assert oracle.block_exponent(b, BF16) == want, hex(b)


def test_block_exponent_fp32_triples_and_fuzz():
    """The 1.5*2^k +-1 ulp triples of the test list ("Test results (B200)"),
    where ceil(log2(amax/6)) steps, plus random fp32 amax patterns."""
    from fractions import Fraction
    pats = []
    for k in range(-126, 128):
        c = bf.float_to_f32_bits(1.5 * 2.0 ** k)
        pats += [c - 1, c, c + 1]
    g = np.random.default_rng(7)
    pats += [int(u) for u in g.integers(0, 0x7F800000, size=4000)]
    for u in pats:
        if not 0 <= u < 0x7F800000:
            continue
        want = bf.scale_exponent(Fraction(bf.f32_bits_to_float(u)))
        assert oracle.block_exponent(u, FP32) == want, hex(u)
    # closed form at the step: 1.5*2^k gives k-2, one ulp above gives k-1
    for k in range(-100, 100):
        c = bf.float_to_f32_bits(1.5 * 2.0 ** k)
        assert oracle.block_exponent(c, FP32) == max(-126, min(125, k - 2))
        assert oracle.block_exponent(c + 1, FP32) == max(-126, min(125, k - 1))


def test_e2m1_rtne_points():
    for v, want in rows("e2m1_rtne_points.txt"):
        code = oracle.e2m1_rtne_code(float(v))
        assert [0, 0.5, 1, 1.5, 2, 3, 4, 6][code] == float(want), v


# -------------------------------------------------------------- projection

def test_projection_bf16_exhaustive_bruteforce():
    """All 65536 bf16 patterns against the exact-rational brute force."""
    x = syn.exhaustive_bf16()
    y = oracle.fake_quant_mxfp4(x)
    want = np.array(bf.project_bf16_rows(x.tolist()), dtype=np.uint16)
    np.testing.assert_array_equal(y, want)


def test_projection_bf16_exhaustive_counts():
    """2036/2048 rows are finite and below saturation; 8 are poisoned and 4
    saturate (TE PR #3264, "Test results (B200)", cross-validation)."""
    g = kv("bf16_exhaustive_counts.txt")
    x = syn.exhaustive_bf16()
    y = oracle.fake_quant_mxfp4(x)
    poisoned = np.all(y == 0x7FC0, axis=1)
    cap = 0x7F40  # 6*2^125
    mag = x & 0x7FFF
    finite = mag < 0x7F80
    over = np.any(finite & (mag > cap), axis=1) & ~poisoned
    assert int(poisoned.sum()) == int(g["poisoned_rows"])
    assert int(over.sum()) == int(g["saturating_rows"])
    assert int((~poisoned & ~over).sum()) == int(g["shared_domain_rows"])
    assert x.shape[0] == int(g["rows"])
    # saturating rows: every value above the cap lands on +-6*2^125
    # ("Known limitations": the projection saturates at the cap)
    sel = finite & (mag > cap)
    assert np.all((y[sel] & 0x7FFF) == cap)
    assert np.all((y[sel] & 0x8000) == (x[sel] & 0x8000))


def test_projection_fp32_fuzz_bruteforce():
    g = np.random.default_rng(11)
    n_rows = 48
    u = g.integers(0, 0x7F800000, size=(n_rows, 32), dtype=np.uint64).astype(np.uint32)
    # rows of a common binade so that blocks are not all dominated by one value
    for r in range(0, n_rows, 3):
        e = int(g.integers(1, 254))
        u[r] = (np.uint32(e) << np.uint32(23)) | (u[r] & np.uint32(0x7FFFFF))
        u[r] -= (g.integers(0, 40, size=32) << 23).astype(np.uint32) * (u[r] >> 23 > 40)
    u |= (g.integers(0, 2, size=u.shape).astype(np.uint32) << np.uint32(31))
    u[5, 3] = 0x7F800000  # Inf poisons its block
    u[7, 9] = 0x7FC00001  # NaN too
    u[9, :] = 0x80000000  # -0 block
    x = u.view(np.float32)
    y = oracle.fake_quant_mxfp4(x).view(np.uint32)
    want = np.array(bf.project_f32_rows(u.tolist()), dtype=np.uint32)
    np.testing.assert_array_equal(y, want)


def test_projection_partial_blocks_bruteforce():
    """K % 32 = 16: the last block holds 16 values and has its own scale."""
    for shape in syn.PARTIAL_BLOCK_SHAPES:
        x = syn.partial_block_fp32(shape)
        y = oracle.fake_quant_mxfp4(x).view(np.uint32)
        want = np.array(bf.project_f32_rows(x.view(np.uint32).tolist()), dtype=np.uint32)
        np.testing.assert_array_equal(y, want)


def test_subnormal_ladder_and_tie():
    for k, xb, yb, code, pay in rows("subnormal_ladder.txt"):
        x = np.zeros((1, 32), dtype=np.uint16)
        x[0, 0] = int(xb, 16)
        y = oracle.fake_quant_mxfp4(x)
        assert int(y[0, 0]) == int(yb, 16), k
        d, s = oracle.mxfp8_row_direct(x)
        assert int(s[0, 0]) == int(code) and int(d[0, 0]) == int(pay, 16), k
        # negative: sign kept, zero keeps its sign too
        x[0, 0] |= 0x8000
        y = oracle.fake_quant_mxfp4(x)
        assert int(y[0, 0]) == (int(yb, 16) | 0x8000), k


def _grid_decompose(y_f64, e):
    return np.abs(y_f64) / np.ldexp(1.0, e)


def test_projection_idempotent_and_on_grid():
    """Every projected value is a grid point p*2^e and projecting again
    changes nothing (TE PR #3264, Description, mode 1)."""
    g = np.random.default_rng(3)
    x = (g.standard_normal((64, 96)) * np.ldexp(1.0, g.integers(-60, 60, size=(64, 1)))).astype(np.float32)
    y = oracle.fake_quant_mxfp4(x)
    y2 = oracle.fake_quant_mxfp4(y)
    np.testing.assert_array_equal(y.view(np.uint32), y2.view(np.uint32))
    grid = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}
    for r in range(x.shape[0]):
        for j0 in range(0, 96, 32):
            blk = x[r, j0:j0 + 32].view(np.uint32) & np.uint32(0x7FFFFFFF)
            e = oracle.block_exponent(int(blk.max()), FP32)
            p = _grid_decompose(y[r, j0:j0 + 32].astype(np.float64), e)
            assert set(p.tolist()) <= grid


# ------------------------------------------------------------- fp8 codes

def test_fp8_decode_matches_torch_all_codes():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    for kind, dt in ((oracle.E4M3, torch.float8_e4m3fn), (oracle.E5M2, torch.float8_e5m2)):
        ref = b.view(dt).to(torch.float64).numpy()
        got = np.array([oracle.fp8_value(i, kind) for i in range(256)])
        np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
        ok = ~np.isnan(ref)
        np.testing.assert_array_equal(got[ok], ref[ok])
        np.testing.assert_array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e8m0_decode_golden_and_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([oracle.e8m0_value(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    np.testing.assert_array_equal(got[:255], ref[:255])
    for c, bits in rows("ue8m0_decode.txt"):
        v = oracle.e8m0_value(int(c))
        if bits == "nan":
            assert math.isnan(v)
        else:
            assert struct.unpack("<I", struct.pack("<f", v))[0] == int(bits, 16)


def _e4m3_probe_values():
    vals = []
    pos = [oracle.fp8_value(c, oracle.E4M3) for c in range(127)]
    for a, b in zip(pos[:-1], pos[1:]):
        m = (a + b) / 2
        mb = bf.float_to_f32_bits(m)
        vals += [m, bf.f32_bits_to_float(mb - 1), bf.f32_bits_to_float(mb + 1), a, b]
    g = np.random.default_rng(5)
    vals += g.uniform(0, 448, 3000).astype(np.float32).tolist()
    vals += (g.uniform(0, 1, 3000) * 2.0 ** -6).astype(np.float32).tolist()
    vals += [2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11, 2.0 ** -30, 0.0]
    vals = [float(np.float32(v)) for v in vals]
    return vals + [-v for v in vals]


def test_e4m3_rtne_matches_torch_cast():
    """Round-to-nearest-even onto E4M3 with subnormals (the blockwise payload
    rounding) against torch's float32 -> float8_e4m3fn conversion."""
    vals = _e4m3_probe_values()
    ref = torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_rtne(v) for v in vals], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_f32_to_bf16_matches_torch_cast():
    g = np.random.default_rng(9)
    u = g.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    u = np.concatenate([u, np.array([0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0x00008000, 0x00018000, 0x80008000,
                                     0x3F808000, 0x3F818000, 0x7F800000, 0xFF800000], dtype=np.uint32)])
    f = u.view(np.float32)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(int(b)) for b in u], dtype=np.uint16)
    nan = np.isnan(f)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert np.all(got[nan] == 0x7FC0)


# ------------------------------------------------------------ direct row

def test_row_direct_decodes_to_projection_exhaustive():
    """MXFP8 rowwise payload/scale bytes decode back to the projected weight,
    2^-127 at code 0 included (TE PR #3264, "Test results (B200)")."""
    x = syn.exhaustive_bf16()
    y = oracle.fake_quant_mxfp4(x)
    d, s = oracle.mxfp8_row_direct(x)
    back16 = oracle.dequant_mxfp8(d, s, oracle.COMPACT, oracle.E4M3, BF16)
    np.testing.assert_array_equal(back16, y)
    back32 = oracle.dequant_mxfp8(d, s, oracle.COMPACT, oracle.E4M3, FP32)
    np.testing.assert_array_equal(back32.view(np.uint32), syn.bf16_bits_to_f32(y).view(np.uint32))
    poisoned = np.all(y == 0x7FC0, axis=1)
    assert np.all(s[poisoned, 0] == 0xFF) and np.all(d[poisoned] == 0x7F)
    assert np.any(s[~poisoned, 0] == 0)  # the code-0 absorption domain is present


def test_row_direct_shift6_and_clamp_closed_form():
    """Unclamped blocks: code = e + 121 and payload = p*2^6, i.e. E4M3
    exponent field = grid exponent + 6 + 7; clamped (e < -121): code 0."""
    x = syn.exhaustive_bf16()
    d, s = oracle.mxfp8_row_direct(x)
    for r in range(0, 2048, 37):
        mag = x[r] & 0x7FFF
        if np.any(mag >= 0x7F80):
            continue
        e = oracle.block_exponent(int(mag.max()), BF16)
        assert int(s[r, 0]) == max(e + 121, 0)
        if e + 121 >= 0:
            # amax/2^e lies in (3, 6], so the largest payload is p*2^6 with p in {3, 4, 6}
            top = max(oracle.fp8_value(int(b), oracle.E4M3) for b in d[r] & 0x7F)
            assert top in (192.0, 256.0, 384.0) or int(mag.max()) < 0x0080


def test_row_direct_fp32_partial_blocks():
    for shape in syn.PARTIAL_BLOCK_SHAPES:
        x = syn.partial_block_fp32(shape)
        y = oracle.fake_quant_mxfp4(x)
        d, s = oracle.mxfp8_row_direct(x)
        assert s.shape == (shape[0], -(-shape[1] // 32))
        back = oracle.dequant_mxfp8(d, s, oracle.COMPACT, oracle.E4M3, FP32)
        np.testing.assert_array_equal(back.view(np.uint32), y.view(np.uint32))


# ----------------------------------------------------------- 128x128 tiles

def _spread_tile(d, base=0):
    """One 128x128 fp32 tile: block (row 0, cols 0..31) at exponent base
    (it holds 6*2^base), every other block holds the full signed grid and
    6*2^(base-d), so its scale exponent is base - d."""
    grid = [0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6, 0.0, 6]
    t = np.zeros((128, 128), dtype=np.float64)
    blk = np.array(grid * 2, dtype=np.float64)
    for r in range(128):
        for b in range(4):
            t[r, 32 * b:32 * b + 32] = blk * 2.0 ** (base - d)
    t[0, 0:32] = np.array(grid * 2) * 2.0 ** base
    return t.astype(np.float32)


def _e4m3_representable(w):
    """E4M3 lattice: 4 significant bits for w >= 2^-6, multiples of 2^-9 below."""
    w = abs(w)
    if w == 0:
        return True
    if w < 2.0 ** -6:
        return (w / 2.0 ** -9) == int(w / 2.0 ** -9)
    m, e = math.frexp(w)
    return (m * 16) == int(m * 16)


def test_blockwise_exactness_boundary():
    """Exact through spread 2^14, first loss at 2^15, and every element's
    loss predicted by the E4M3 lattice (TE PR #3264, "Test results (B200)")."""
    g = kv("blockwise_exactness_boundary.txt")
    exact_upto, first_loss = int(g["exact_through_spread"]), int(g["first_loss_spread"])
    results = {}
    for base in (0, 57, -100):
        for d in range(int(g["max_spread_tested"]) + 1):
            x = _spread_tile(d, base)
            y = oracle.fake_quant_mxfp4(x)
            data, sinv = oracle.fp8_block128_direct(x)
            assert sinv[0, 0] == np.float32(2.0 ** (base - 6))
            back = oracle.dequant_block128(data, sinv, FP32)
            exact = np.array_equal(back.view(np.uint32), y.view(np.uint32))
            results[(base, d)] = exact
            # per-element prediction: p*2^(e_b - T) on the E4M3 lattice
            pay = y.astype(np.float64) / 2.0 ** (base - 6)
            pred = np.vectorize(_e4m3_representable)(pay)
            np.testing.assert_array_equal(back == y, pred)
        assert all(results[(base, d)] for d in range(exact_upto + 1))
        assert not results[(base, first_loss)]


def test_blockwise_clamp_and_planted_tiles():
    """Tile scale clamps at 2^-127 (fp32 0x00400000); zero, -0 and 2^-127
    tiles (the spread-sweep workload) encode exactly."""
    x, _ = syn.spread_tiles_fp32(rows=128, K=512)
    data, sinv = oracle.fp8_block128_direct(x)
    s = sinv.view(np.uint32)
    assert s[0, 0] == 0x00400000 and s[0, 1] == 0x00400000 and s[0, 2] == 0x00400000
    assert np.all(data[:, :128] == 0) and np.all(data[:, 128:256] == 0x80)
    y = oracle.fake_quant_mxfp4(x[:, 256:384])
    back = oracle.dequant_block128(data[:, 256:384], sinv[:, 2:3], FP32)
    np.testing.assert_array_equal(back.view(np.uint32), y.view(np.uint32))
    # 2^-127 at e = -126 is 0.5*2^-126: T = -127, payload 1.0 = 0x38 (sign kept)
    assert set(np.unique(data[:, 256:384]).tolist()) == {0x38, 0xB8}


def test_blockwise_poisoned_block_left_out_of_tile_max():
    """Reading of "non-finite block poisoning" for the 128x128 form: a
    poisoned block gives payloads 0x7F and does not enter the tile maximum,
    so the finite blocks still encode their projection exactly."""
    x = np.zeros((128, 128), dtype=np.float32)
    x[:, :] = np.float32(2.0 ** -50) * np.tile(np.array([6, -3, 1.5, 0.5], dtype=np.float32), 32)
    x[5, 32:64] = np.nan
    x[70, 0] = np.inf
    data, sinv = oracle.fp8_block128_direct(x)
    e_fin = oracle.block_exponent(int(np.float32(6 * 2.0 ** -50).view(np.uint32)), FP32)
    assert sinv[0, 0] == np.float32(2.0 ** (e_fin - 6))
    assert np.all(data[5, 32:64] == 0x7F) and np.all(data[70, 0:32] == 0x7F)
    y = oracle.fake_quant_mxfp4(x)
    back = oracle.dequant_block128(data, sinv, FP32)
    finite = np.ones_like(x, dtype=bool)
    finite[5, 32:64] = False
    finite[70, 0:32] = False
    np.testing.assert_array_equal(back.view(np.uint32)[finite], y.view(np.uint32)[finite])


# ------------------------------------------------ MXFP8 columnwise (32x1)

def test_mxfp8_host_exponent_is_ceil_log2_amax_over_448():
    """The host rule read for "fresh 32x1 quantization": the smallest s with
    amax <= 448 * 2^s, clamped to [-127, 127]; zero gives -127."""
    from fractions import Fraction
    g = np.random.default_rng(12)
    vals = [p * 2.0 ** k for p in (0.5, 1, 1.5, 2, 3, 4, 6) for k in range(-133, 126)]
    vals += [float(v) for v in g.uniform(0, 1, 3000).astype(np.float32) * np.ldexp(1.0, g.integers(-140, 120, 3000))]
    vals += [448.0, 448.0 * 2 ** -20, 449.0, 447.9999, 2.0 ** -149, 3.0e38]
    for v in vals:
        if v == 0:
            continue
        a = Fraction(v)
        s_ = 0
        while Fraction(448) * Fraction(2) ** s_ < a:
            s_ += 1
        while Fraction(448) * Fraction(2) ** (s_ - 1) >= a:
            s_ -= 1
        assert oracle.mxfp8_host_exponent(v) == max(-127, min(127, s_)), v
    assert oracle.mxfp8_host_exponent(0.0) == -127


def test_mxfp8_columnwise_exact_for_uniform_row_exponents():
    """When every 1x32 block of a column block shares one exponent, the
    projected values p*2^e re-encode exactly (payload p*2^6 or p*2^7, s =
    e - 6 or e - 7): decode(columnwise(x)) == projection(x)."""
    g = np.random.default_rng(4)
    grid = np.array([0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6, 0], dtype=np.float64)
    for e in (-126, -100, -3, 0, 17, 118):
        p = grid[g.integers(0, 15, size=(96, 64))]
        p[:, ::32] = 6.0  # every 1x32 block reaches 6, so its exponent is exactly e
        x = (p * 2.0 ** e).astype(np.float32)
        y = oracle.fake_quant_mxfp4(x)
        data, sc = oracle.mxfp8_col_direct(x)
        assert sc.shape == (64, 3)
        back = oracle.dequant_mxfp8(np.ascontiguousarray(data.T), sc, oracle.COMPACT, oracle.E4M3, FP32).T
        np.testing.assert_array_equal(np.ascontiguousarray(back).view(np.uint32), y.view(np.uint32))


def test_mxfp8_columnwise_error_bound_and_poison():
    """Mixed row exponents: every decoded value is the E4M3 rounding of y /
    2^s (relative error <= 2^-4, absolute <= 2^(s-10) in the subnormal range);
    a NaN in a 1x32 block poisons each 32x1 block it touches."""
    x = syn.partial_block_fp32((100, 48))
    y = oracle.fake_quant_mxfp4(x).astype(np.float64)
    data, sc = oracle.mxfp8_col_direct(x)
    assert sc.shape == (48, 4) and data.shape == (100, 48)
    back = oracle.dequant_mxfp8(np.ascontiguousarray(data.T), sc, oracle.COMPACT, oracle.E4M3, FP32).T.astype(np.float64)
    s_of = np.ldexp(1.0, sc.astype(np.int64).T - 127)  # (4, 48)
    bound = np.maximum(np.abs(y) * 2.0 ** -4, np.repeat(s_of, 32, axis=0)[:100] * 2.0 ** -10)
    assert np.all(np.abs(back - y) <= bound)
    x[40, 5] = np.nan  # poisons row 40's first 1x32 block (columns 0..31)
    data, sc = oracle.mxfp8_col_direct(x)
    assert np.all(sc[:32, 1] == 0xFF) and np.all(sc[32:, 1] != 0xFF)
    assert np.all(data[32:64, :32] == 0x7F)


# ------------------------------------------------------ packed MXFP4

def test_packed_mxfp4_decodes_to_projection_and_moves_past_the_cap():
    """The packed deployment form decodes exactly to the projection wherever
    amax <= 6*2^125; above it the scale moves to 2^126 and the nibbles are
    the nearest grid points of |x|/2^126 (TE PR #3264, Description and
    "Known limitations")."""
    from fractions import Fraction
    g = kv("mxfp4_packed_saturation.txt")
    x = syn.exhaustive_bf16()
    packed, scales = oracle.mxfp4_pack(x)
    y = oracle.fake_quant_mxfp4(x)
    back = oracle.dequant_mxfp4(packed, scales, oracle.COMPACT, 32, BF16)
    mag = x & 0x7FFF
    poisoned = np.any(mag >= 0x7F80, axis=1)
    over = np.any((mag > 0x7F40) & (mag < 0x7F80), axis=1) & ~poisoned
    ok = ~poisoned & ~over
    assert int(ok.sum()) == 2036
    np.testing.assert_array_equal(back[ok], y[ok])
    assert np.all(scales[poisoned, 0] == 0xFF) and np.all(packed[poisoned] == 0)
    assert np.all(scales[over, 0] == int(g["saturating_scale_code"]))
    # nibbles of the saturating rows: nearest grid point of |x| / 2^126, ties to even
    for r in np.nonzero(over)[0]:
        for i in range(32):
            v = Fraction(bf.bf16_to_float(int(x[r, i])))
            a = abs(v) / Fraction(2) ** 126
            c = min(range(8), key=lambda k: (abs(a - bf.GRID[k]), k % 2))
            nib = (int(packed[r, i // 2]) >> ((i % 2) * 4)) & 15
            assert nib == (c | (8 if v < 0 or (v == 0 and x[r, i] & 0x8000) else 0)), (r, i)
    # the projection instead holds those rows at the cap 2^125 * 6 (scale code 252)
    _, row_scales = oracle.mxfp8_row_direct(x[over])
    assert np.all(row_scales[:, 0] + 6 == int(g["projection_cap_scale_code"]))


def test_packed_mxfp4_nibble_order_and_partial_blocks():
    """Element 2i in the low nibble, 2i+1 in the high nibble; a short last
    block keeps its own scale (K = 48 -> 24 bytes, 2 scales)."""
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :4] = [0.5, 6.0, -1.0, 3.0]  # amax 6 -> e = 0, codes 1, 7, 8|2, 5
    packed, scales = oracle.mxfp4_pack(x)
    assert scales[0, 0] == 127
    assert packed[0, 0] == 0x71 and packed[0, 1] == 0x5A
    for shape in ((100, 48), (64, 16)):
        xx = syn.partial_block_fp32(shape)
        packed, scales = oracle.mxfp4_pack(xx)
        assert packed.shape == (shape[0], shape[1] // 2) and scales.shape == (shape[0], -(-shape[1] // 32))
        back = oracle.dequant_mxfp4(packed, scales, oracle.COMPACT, shape[1], FP32)
        np.testing.assert_array_equal(back.view(np.uint32), oracle.fake_quant_mxfp4(xx).view(np.uint32))


def test_e2m1_nibble_values():
    vals = [oracle.e2m1_value(n) for n in range(16)]
    assert vals[:8] == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert vals[8:] == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]
    assert math.copysign(1.0, vals[8]) == -1.0


# ---------------------------------------------------------------- layouts

def test_swizzle_offsets_golden_and_bijective():
    for nb, r, j, off in rows("swizzle_offsets.txt"):
        assert oracle.scale_offset(int(r), int(j), int(nb), oracle.SWIZZLED) == int(off)
    for rows_, nb in ((256, 8), (128, 225), (384, 12)):
        cp = -(-nb // 4) * 4
        offs = {oracle.scale_offset(r, j, nb, oracle.SWIZZLED) for r in range(rows_) for j in range(cp)}
        assert offs == set(range(rows_ * cp))


def test_scale_columns_ceil():
    """ceil(K/32) columns: K = 48 -> 2 and K = 16 -> 1; K // 32 would give 1
    and 0 (TE PR #3790, partial-block regression)."""
    for K, nb in ((48, 2), (16, 1), (96, 3), (7184, 225), (8192, 256)):
        assert oracle.scale_cols(K) == nb
    assert oracle.scale_bytes(100, 48, oracle.PADDED) == 128 * 4
    assert oracle.scale_bytes(100, 48, oracle.COMPACT) == 200


@pytest.mark.parametrize("shape", [(100, 48), (64, 16), (128, 96), (300, 7184 // 4)])
def test_export_swizzle_invariance_and_dequant(shape):
    """Exported compact scales are the same from compact, padded and
    swizzled storage, and the export decodes exactly to dequantize()
    (TE PR #3790, Description and its test list)."""
    rows_, K = shape
    x = syn.partial_block_fp32(shape) if rows_ <= 128 else syn.bf16_bits_to_f32(syn.normal_bf16(rows_, K, seed=99))
    x = np.ascontiguousarray(x, dtype=np.float32)
    d, s_c = oracle.mxfp8_row_direct(x, oracle.COMPACT)
    for lay in (oracle.PADDED, oracle.SWIZZLED):
        _, s_l = oracle.mxfp8_row_direct(x, lay)
        ex = oracle.export_scales(s_l, lay, rows_, K)
        np.testing.assert_array_equal(ex, s_c)
        for kind in (oracle.E4M3, oracle.E5M2):
            a = oracle.dequant_mxfp8(d, ex, oracle.COMPACT, kind, FP32)
            b = oracle.dequant_mxfp8(d, s_l, lay, kind, FP32)
            np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))
        nb = -(-K // 32)
        if lay == oracle.PADDED:  # a plain row-major (Rp, Cp) matrix
            Rp, Cp = -(-rows_ // 128) * 128, -(-nb // 4) * 4
            np.testing.assert_array_equal(s_l.reshape(Rp, Cp)[:rows_, :nb], s_c)
        # padding bytes are zero
        mask = np.ones(s_l.size, dtype=bool)
        for r in range(rows_):
            for j in range(nb):
                mask[oracle.scale_offset(r, j, nb, lay)] = False
        assert np.all(s_l[mask] == 0)


def test_dequant_planted_codes():
    """Planted extreme scale codes through dequantize: 0 -> 2^-127, 255 -> NaN
    (TE PR #3264, "Test results (B200)")."""
    d = np.array([[0x38] * 32 + [0x38] * 32], dtype=np.uint8)
    s = np.array([[0, 255]], dtype=np.uint8)
    out = oracle.dequant_mxfp8(d, s, oracle.COMPACT, oracle.E4M3, FP32).view(np.uint32)
    assert np.all(out[0, :32] == 0x00400000)
    assert np.all(out[0, 32:] == 0x7FC00000)
    out16 = oracle.dequant_mxfp8(d, s, oracle.COMPACT, oracle.E4M3, BF16)
    assert np.all(out16[0, :32] == 0x0040) and np.all(out16[0, 32:] == 0x7FC0)
    # E5M2 Inf payload times a finite scale stays Inf; the largest finite
    # payload times 2^127 overflows to Inf
    d = np.array([[0x7C] * 16 + [0x7B] * 16], dtype=np.uint8)
    out = oracle.dequant_mxfp8(d, np.array([[254]], np.uint8), oracle.COMPACT, oracle.E5M2, FP32)
    assert np.all(np.isinf(out))
