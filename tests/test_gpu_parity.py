"""GPU parity: every conversion of libmxq against the CPU oracle, byte for
byte (tolerance 0: payload bytes, scale bytes and output bit patterns must
be equal).  Small cases are compared in full, the 8192 x 8192 and MoE
workloads on sampled rows and tiles plus properties checked over the whole
tensor.  All calls go through the C ABI via the Python binding."""

import zlib

import numpy as np
import pytest
import torch

import block_scaled_precision_x32_gb300 as mxq
import oracle
from block_scaled_precision_x32_gb300 import synthetic as syn
from tests.gpu_util import Guarded, dev_bf16, dev_f32, dev_input, host_bits, oracle_bits

pytestmark = pytest.mark.gpu

LAYOUTS = (oracle.COMPACT, oracle.PADDED, oracle.SWIZZLED)


@pytest.fixture(scope="module")
def mx():
    return mxq.library()


def _rows_k(a):
    K = a.shape[-1]
    return (a.size // K if K else 0), K


def run_all_and_compare(mx, x_np, layouts=LAYOUTS, block128=True, guard=True):
    """Projection, MXFP8 row (every layout), 128x128 blockwise, export and
    dequantize of one input, each against the oracle."""
    x = dev_input(x_np)
    rows, K = _rows_k(x_np)
    dtype = x.dtype

    # projection
    y = Guarded(x.shape, dtype) if guard else None
    got = mx.fake_quant_mxfp4(x, out=y.t if y else None)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(got), oracle_bits(oracle.fake_quant_mxfp4(x_np)))
    if y:
        assert y.intact()

    # MXFP8 rowwise, each scale layout, then export and dequantize
    ref_data, ref_compact = oracle.mxfp8_row_direct(x_np, oracle.COMPACT)
    for lay in layouts:
        nbytes = mx.scale_bytes(rows, K, lay)
        d = Guarded(x.shape, torch.uint8)
        s = Guarded((max(nbytes, 1),), torch.uint8)
        mx.mxfp8_row_direct(x, lay, data=d.t, scales=s.t)
        torch.cuda.synchronize()
        assert d.intact() and s.intact()
        np.testing.assert_array_equal(host_bits(d.t), ref_data)
        ref_lay = ref_compact.reshape(-1) if lay == oracle.COMPACT else oracle.scales_to_layout(ref_compact, rows, K, lay)
        np.testing.assert_array_equal(host_bits(s.t)[:nbytes], ref_lay)
        for kind in ("e4m3", "e5m2"):
            comp = mx.export_mxfp8(d.t, s.t[:nbytes], shape=x.shape, layout=lay, fp8=kind)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(host_bits(comp.scale_inv).reshape(rows, -1), ref_compact.reshape(rows, -1))
            assert comp.data.dtype == (torch.float8_e4m3fn if kind == "e4m3" else torch.float8_e5m2)
            assert comp.data.data_ptr() == d.t.data_ptr()
            nb = (K + 31) // 32
            assert comp.is_view == (lay == oracle.COMPACT or (lay == oracle.PADDED and nb % 4 == 0))
            for odt, ocode in ((torch.float32, oracle.FP32), (torch.bfloat16, oracle.BF16)):
                ok = oracle.E4M3 if kind == "e4m3" else oracle.E5M2
                want = oracle_bits(oracle.dequant_mxfp8(ref_data, ref_compact, oracle.COMPACT, ok, ocode))
                a = mx.dequantize(d.t, scales=s.t[:nbytes], layout=lay, fp8=kind, out_dtype=odt)
                b = mx.dequantize(comp.data.view(torch.uint8), scales=comp.scale_inv.contiguous(), layout="compact",
                                  fp8=kind, out_dtype=odt)
                torch.cuda.synchronize()
                np.testing.assert_array_equal(host_bits(a), want)
                np.testing.assert_array_equal(host_bits(b), want)  # export decodes to dequantize()

    # MXFP8 columnwise (32x1 blocks of the projection), each layout, and its dequantize
    ref_cd, ref_cs = oracle.mxfp8_col_direct(x_np, oracle.COMPACT)
    x2 = x if x.dim() == 2 else x.reshape(rows, K)
    for lay in layouts:
        nbytes = mx.scale_bytes(K, rows, lay)
        d = Guarded((rows, K), torch.uint8)
        s = Guarded((max(nbytes, 1),), torch.uint8)
        mx.mxfp8_col_direct(x2, lay, data=d.t, scales=s.t)
        torch.cuda.synchronize()
        assert d.intact() and s.intact()
        np.testing.assert_array_equal(host_bits(d.t), ref_cd)
        ref_lay = ref_cs.reshape(-1) if lay == oracle.COMPACT else oracle.scales_to_layout(ref_cs, K, rows, lay)
        np.testing.assert_array_equal(host_bits(s.t)[:nbytes], ref_lay)
        for odt, ocode in ((torch.float32, oracle.FP32), (torch.bfloat16, oracle.BF16)):
            got = mx.dequantize(d.t, scales=s.t[:nbytes], layout=lay, out_dtype=odt, columnwise=True)
            torch.cuda.synchronize()
            want = oracle.dequant_mxfp8(np.ascontiguousarray(ref_cd.T), ref_cs, oracle.COMPACT, oracle.E4M3, ocode).T
            np.testing.assert_array_equal(host_bits(got), oracle_bits(np.ascontiguousarray(want)))

    # packed MXFP4 (deployment form), each scale layout, and its dequantize
    ref_p, ref_pc = oracle.mxfp4_pack(x_np, oracle.COMPACT)
    for lay in layouts:
        nbytes = mx.scale_bytes(rows, K, lay)
        p = Guarded((rows, (K + 1) // 2), torch.uint8)
        s = Guarded((max(nbytes, 1),), torch.uint8)
        x2 = x if x.dim() == 2 else x.reshape(rows, K)
        mx.mxfp4_pack(x2, lay, packed=p.t, scales=s.t)
        torch.cuda.synchronize()
        assert p.intact() and s.intact()
        np.testing.assert_array_equal(host_bits(p.t), ref_p)
        ref_lay = ref_pc.reshape(-1) if lay == oracle.COMPACT else oracle.scales_to_layout(ref_pc, rows, K, lay)
        np.testing.assert_array_equal(host_bits(s.t)[:nbytes], ref_lay)
        for odt, ocode in ((torch.float32, oracle.FP32), (torch.bfloat16, oracle.BF16)):
            got = mx.dequantize(p.t, scales=s.t[:nbytes], layout=lay, out_dtype=odt, mxfp4_K=K)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(host_bits(got).reshape(rows, K),
                                          oracle_bits(oracle.dequant_mxfp4(ref_p, ref_pc, oracle.COMPACT, K, ocode)))

    if block128:
        ref_d, ref_s = oracle.fp8_block128_direct(x_np)
        d = Guarded(x.shape, torch.uint8)
        s = Guarded((max(mx.tile_scale_count(rows, K), 1),), torch.float32)
        mx.fp8_block128_direct(x, data=d.t, tile_scale_inv=s.t)
        torch.cuda.synchronize()
        assert d.intact() and s.intact()
        np.testing.assert_array_equal(host_bits(d.t), ref_d)
        np.testing.assert_array_equal(host_bits(s.t)[:ref_s.size], ref_s.view(np.uint32).reshape(-1))
        for odt, ocode in ((torch.float32, oracle.FP32), (torch.bfloat16, oracle.BF16)):
            got = mx.dequantize(d.t, tile_scale_inv=s.t, out_dtype=odt)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(host_bits(got), oracle_bits(oracle.dequant_block128(ref_d, ref_s, ocode)))


# ------------------------------------------------ exhaustive bf16 corpus

def test_exhaustive_bf16_corpus(mx):
    """All 65536 bf16 patterns, one block per row: projection, MXFP8 rowwise,
    export, dequantize and (with partial 32-column tiles) blockwise."""
    run_all_and_compare(mx, syn.exhaustive_bf16())


# ------------------------------------------------ partial-block fp32 set

@pytest.mark.parametrize("shape", syn.PARTIAL_BLOCK_SHAPES)
def test_partial_block_fp32(mx, shape):
    run_all_and_compare(mx, syn.partial_block_fp32(shape))


# ---------------------------------------------------------- edge shapes

@pytest.mark.parametrize("shape", [(1, 1), (1, 17), (3, 33), (129, 130), (2, 16), (5, 48), (257, 264), (130, 7184)])
@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_edge_shapes(mx, shape, dt):
    g = np.random.default_rng(zlib.crc32(repr((shape, dt)).encode()))
    w = (g.standard_normal(shape) * np.ldexp(1.0, g.integers(-30, 30, size=(shape[0], 1)))).astype(np.float32)
    x = syn.f32_to_bf16_bits(w) if dt == "bf16" else w
    run_all_and_compare(mx, x)


@pytest.mark.parametrize("shape", [(1, 32), (32, 64), (33, 96), (100, 160), (257, 320), (70, 4096)])
@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_columnwise_tile_path(mx, shape, dt):
    """K % 32 == 0: the 32x64 warp-tile columnwise path (fp32 through the
    E2M1 conversion).  Odd and half-filled column tiles, ragged bands, row
    and column exponent spreads of 2^+-40 (so 32x1 payloads fall into E4M3
    subnormals), blocks at the upper clamp, and NaN / Inf / zero blocks."""
    rows, K = shape
    g = np.random.default_rng(zlib.crc32(repr(("tile64", shape)).encode()))
    w = g.standard_normal(shape) * np.ldexp(1.0, g.integers(-40, 40, size=(rows, 1)))
    w *= np.ldexp(1.0, g.integers(-8, 8, size=(1, K)))
    w = w.astype(np.float32)
    if dt == "bf16":
        x = syn.f32_to_bf16_bits(w)
        if rows > 2:
            x[1, :] = np.where(np.arange(K) % 3 == 0, 0x7F7F, 0xFF70)  # near 6 * 2^125: the upper clamp
            x[2, :32] = 0
        if rows > 40 and K > 40:
            x[37, 5] = 0x7FC0   # NaN block
            x[40, 33] = 0xFF80  # -Inf block
    else:
        x = w
        u = x.view(np.uint32)
        if rows > 2:
            u[1, :] = np.where(np.arange(K) % 3 == 0, 0x7F7FFFFF, 0xFF6FFFFF)  # near the fp32 maximum: the clamp
            x[2, :32] = 0.0
        if rows > 40 and K > 40:
            u[37, 5] = 0x7FC00001   # NaN block
            u[40, 33] = 0xFF800000  # -Inf block
    run_all_and_compare(mx, x)


def test_fp32_random_bit_patterns(mx):
    """Finite fp32 bit patterns over every exponent range, with Inf/NaN
    planted in a few blocks (non-finite block poisoning)."""
    g = np.random.default_rng(21)
    u = g.integers(0, 0x7F800000, size=(384, 160), dtype=np.uint64).astype(np.uint32)
    for r in range(0, 384, 2):  # rows of one binade band, so scales span 2^-126..2^125
        e = int(g.integers(1, 255))
        u[r] = (np.uint32(e) << np.uint32(23)) | (u[r] & np.uint32(0x7FFFFF))
    u |= g.integers(0, 2, size=u.shape).astype(np.uint32) << np.uint32(31)
    u[3, 5] = 0x7F800000
    u[40, 100] = 0xFF800000
    u[77, 0] = 0x7FC00001
    u[200, 159] = 0xFFFFFFFF
    run_all_and_compare(mx, u.view(np.float32))


def test_bf16_edge_values(mx):
    """Ladder 2^-127..2^-133, the 2^-128 tie, 1.5*2^k +-1 ulp, saturation
    past 6*2^125 and signed zeros (TE PR #3264, "Test results (B200)")."""
    rows = []
    for k in range(-133, -126):
        r = np.zeros(32, dtype=np.uint16)
        r[3] = syn.f32_to_bf16_bits(np.array([np.ldexp(1.0, k)], dtype=np.float32))[0]
        r[4] = r[3] | 0x8000
        rows.append(r)
    for k in range(-120, 128, 7):
        c = int(syn.f32_to_bf16_bits(np.array([1.5 * 2.0 ** k], dtype=np.float32))[0])
        r = np.zeros(32, dtype=np.uint16)
        r[:3] = [c - 1, c, c + 1]
        r[3:6] = [c - 0x40, c - 0x3F, c - 0x41]
        rows.append(r)
    sat = np.arange(0x7F38, 0x7F80, dtype=np.uint16)[:32]
    rows.append(sat)
    rows.append(sat | 0x8000)
    rows.append(np.array([0x8000] * 16 + [0] * 16, dtype=np.uint16))
    run_all_and_compare(mx, np.stack(rows))


# -------------------------------------------------- views and in place

@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_misaligned_and_strided_views(mx, dt):
    """Views that start one element late and rows with padding take the
    scalar path and give the same bytes (TE PR #3264: misaligned views)."""
    g = np.random.default_rng(5)
    rows, K = 67, 200
    w = (g.standard_normal((rows, K + 9)) * 0.02).astype(np.float32)
    base = dev_bf16(syn.f32_to_bf16_bits(w)) if dt == "bf16" else dev_f32(w)
    for view in (base[:, 1:K + 1], base[:, :K], base[:, 3:3 + 64]):
        x_np = host_bits(view.contiguous())
        x_np = x_np if dt == "bf16" else x_np.view(np.float32)
        np.testing.assert_array_equal(host_bits(mx.fake_quant_mxfp4(view)), oracle_bits(oracle.fake_quant_mxfp4(x_np)))
        d, s = mx.mxfp8_row_direct(view, "compact")
        rd, rs = oracle.mxfp8_row_direct(x_np)
        np.testing.assert_array_equal(host_bits(d), rd)
        np.testing.assert_array_equal(host_bits(s), rs)
        d, s = mx.fp8_block128_direct(view)
        rd, rs = oracle.fp8_block128_direct(x_np)
        np.testing.assert_array_equal(host_bits(d), rd)
        np.testing.assert_array_equal(host_bits(s), rs.view(np.uint32))


def test_in_place_projection(mx):
    x_np = syn.partial_block_fp32((128, 96))
    x = dev_f32(x_np)
    out = mx.fake_quant_mxfp4(x, out=x)
    assert out.data_ptr() == x.data_ptr()
    np.testing.assert_array_equal(host_bits(x), oracle_bits(oracle.fake_quant_mxfp4(x_np)))


def test_fp16_and_cpu_rejected(mx):
    with pytest.raises(mxq.MXQError) as ei:
        mx.fake_quant_mxfp4(torch.zeros(4, 32, dtype=torch.float16, device="cuda"))
    assert ei.value.status == 2
    with pytest.raises(mxq.MXQError):
        mx.dequantize(torch.zeros(4, 32, dtype=torch.uint8, device="cuda"),
                      scales=torch.zeros(4, 1, dtype=torch.uint8, device="cuda"),
                      out=torch.empty(4, 32, dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError):
        mx.fake_quant_mxfp4(torch.zeros(4, 32, dtype=torch.bfloat16))


def test_empty_tensors(mx):
    for shape in ((0, 32), (4, 0), (0, 0)):
        x = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        assert mx.fake_quant_mxfp4(x).shape == shape
        d, s = mx.mxfp8_row_direct(x, "swizzled")
        assert d.shape == shape
        c = mx.export_mxfp8(d, s, shape=shape, layout="swizzled")
        assert c.scale_inv.shape == (shape[0], (shape[1] + 31) // 32)


def test_export_without_rowwise_data(mx):
    with pytest.raises(mxq.MXQError) as ei:
        mx.export_mxfp8(None, torch.zeros(128, 4, dtype=torch.uint8, device="cuda"), shape=(100, 48),
                        layout="padded")
    assert ei.value.status == 3


# ----------------------------------------------------- dequantize alone

@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("kind", [oracle.E4M3, oracle.E5M2])
def test_dequant_every_payload_and_scale_code(mx, lay, kind):
    """Every payload byte against every 16th scale code plus codes 0, 1,
    127, 254 and 255 (TE PR #3264: planted extreme scale codes)."""
    codes = sorted(set(range(0, 256, 16)) | {0, 1, 127, 254, 255})
    rows, K = len(codes) * 4, 256 + 16
    g = np.random.default_rng(kind * 10 + lay)
    data = np.tile(np.arange(256, dtype=np.uint8), (rows, 2))[:, :K].copy()
    g.shuffle(data, axis=1)
    nb = (K + 31) // 32
    compact = np.repeat(np.array(codes, dtype=np.uint8), 4)[:, None].repeat(nb, axis=1)
    compact[:, 1] = g.integers(0, 256, size=rows, dtype=np.uint8)
    scales = compact.reshape(-1) if lay == oracle.COMPACT else oracle.scales_to_layout(compact, rows, K, lay)
    d = torch.from_numpy(data).cuda()
    s = torch.from_numpy(scales).cuda()
    for odt, ocode in ((torch.float32, oracle.FP32), (torch.bfloat16, oracle.BF16)):
        got = mx.dequantize(d, scales=s, layout=lay, fp8="e4m3" if kind == oracle.E4M3 else "e5m2", out_dtype=odt)
        np.testing.assert_array_equal(host_bits(got), oracle_bits(oracle.dequant_mxfp8(data, compact, oracle.COMPACT, kind, ocode)))


@pytest.mark.parametrize("K", [256, 272])
@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("kind", [oracle.E4M3, oracle.E5M2])
def test_dequant_columnwise_every_payload_and_scale_code(mx, K, lay, kind):
    """Columnwise form: every payload byte in every column, each column with
    its own scale codes (all 256 codes appear, 255 and the small codes that
    leave bf16's normal range for fp32 output included); K = 256 takes the
    warp-tile kernel, K = 272 the element-wise one; 100 rows end in a
    ragged band."""
    rows = 100
    g = np.random.default_rng(K * 10 + kind * 3 + lay)
    data = np.tile(np.arange(256, dtype=np.uint8), (rows, 2))[:, :K].copy()
    g.shuffle(data, axis=1)
    nbr = (rows + 31) // 32
    cs = ((np.arange(K)[:, None] * 37 + np.arange(nbr)[None, :] * 101) % 256).astype(np.uint8)  # K x nbr codes
    scales = cs.reshape(-1) if lay == oracle.COMPACT else oracle.scales_to_layout(cs, K, rows, lay)
    d = torch.from_numpy(data).cuda()
    s = torch.from_numpy(scales).cuda()
    for odt, ocode in ((torch.float32, oracle.FP32), (torch.bfloat16, oracle.BF16)):
        got = mx.dequantize(d, scales=s, layout=lay, fp8="e4m3" if kind == oracle.E4M3 else "e5m2", out_dtype=odt,
                            columnwise=True)
        want = oracle.dequant_mxfp8(np.ascontiguousarray(data.T), cs, oracle.COMPACT, kind, ocode).T
        np.testing.assert_array_equal(host_bits(got), oracle_bits(np.ascontiguousarray(want)))


@pytest.mark.parametrize("K", [224, 288, 416])
@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("kind", [oracle.E4M3, oracle.E5M2])
def test_dequant_columnwise_fast_and_slow_chunks(mx, K, lay, kind):
    """Columnwise dequantize on widths that end in a partial 128-column
    tile (K % 32 == 0, K % 128 != 0), 200 rows (a ragged last band).  Most
    bands hold only codes of the fast path; band 2 has one code 255 in one
    column, band 4 one code below the fp32 fast range, band 6 (the ragged
    one) a code 0; rows 37 and 150 hold NaN / Inf payloads.  bf16 and fp32
    output, every layout (swizzled codes are loaded per warp, compact and
    padded ones per CTA)."""
    rows = 200
    g = np.random.default_rng(K * 7 + kind * 5 + lay)
    special = (lambda b: (b & 0x7F) == 0x7F) if kind == oracle.E4M3 else (lambda b: (b & 0x7C) == 0x7C)
    data = g.integers(0, 256, size=(rows, K), dtype=np.uint8)
    data[special(data)] &= 0x83  # finite payloads everywhere ...
    for r in (37, 150):  # ... but in two rows
        cols = g.choice(K, size=3, replace=False)
        data[r, cols] = 0x7F if kind == oracle.E4M3 else np.array([0x7C, 0xFC, 0x7E], dtype=np.uint8)
    nbr = (rows + 31) // 32
    cs = g.integers(20, 231, size=(K, nbr), dtype=np.uint8)  # K x nbr codes
    cs[5, 2] = 255
    cs[K - 3, 4] = 3
    cs[100, 6] = 0
    scales = cs.reshape(-1) if lay == oracle.COMPACT else oracle.scales_to_layout(cs, K, rows, lay)
    d = torch.from_numpy(data).cuda()
    s = torch.from_numpy(scales).cuda()
    for odt, ocode in ((torch.float32, oracle.FP32), (torch.bfloat16, oracle.BF16)):
        got = mx.dequantize(d, scales=s, layout=lay, fp8="e4m3" if kind == oracle.E4M3 else "e5m2", out_dtype=odt,
                            columnwise=True)
        want = oracle.dequant_mxfp8(np.ascontiguousarray(data.T), cs, oracle.COMPACT, kind, ocode).T
        np.testing.assert_array_equal(host_bits(got), oracle_bits(np.ascontiguousarray(want)))


def test_dequant_block128_arbitrary_scales(mx):
    """Blockwise dequantize with scale_inv that are not powers of two
    (rounded fp32 products, subnormal results, overflow to Inf)."""
    g = np.random.default_rng(3)
    rows, K = 300, 400
    data = g.integers(0, 256, size=(rows, K), dtype=np.uint8)
    tiles = ((rows + 127) // 128, (K + 127) // 128)
    sinv = (g.standard_normal(tiles) * np.ldexp(1.0, g.integers(-140, 120, size=tiles))).astype(np.float32)
    sinv[0, 0] = np.float32(3.4e38)
    sinv[0, 1] = np.float32(1e-44)
    d = torch.from_numpy(data).cuda()
    s = torch.from_numpy(sinv).cuda()
    for odt, ocode in ((torch.float32, oracle.FP32), (torch.bfloat16, oracle.BF16)):
        got = mx.dequantize(d, tile_scale_inv=s, out_dtype=odt)
        np.testing.assert_array_equal(host_bits(got), oracle_bits(oracle.dequant_block128(data, sinv, ocode)))


@pytest.mark.parametrize("K", [256, 272])
def test_dequant_block128_power_of_two_scales(mx, K):
    """Blockwise dequantize of every payload byte with tile scales 2^T over
    the whole range the converter writes -- 2^-127 (the fp32 subnormal), the
    fp32-output boundary 2^-118 / 2^-117, 2^-1, 2^0, 2^7, 2^127 -- and with
    scales just off a power of two, -2^T, +-Inf and NaN beside them (the
    element-wise path).  K = 256 takes the vector path, K = 272 the ragged
    one; rows of a 128-row tile mix NaN payloads (0x7F, 0xFF) with others."""
    scales_t = [-127, -118, -117, -1, 0, 7, 127]
    odd = [np.float32(1.5), np.float32(-1.0), np.float32(np.inf), np.float32(-np.inf), np.float32(np.nan),
           np.float32(np.ldexp(1.0, -120) * 1.25)]
    sinv_list = [np.float32(np.ldexp(1.0, t)) for t in scales_t] + odd
    rows = 128 * len(sinv_list)
    tc = (K + 127) // 128
    data = np.tile(np.arange(256, dtype=np.uint8), rows * K // 256 + 1)[: rows * K].reshape(rows, K)
    data = np.ascontiguousarray(np.roll(data, 5, axis=1))
    sinv = np.empty((len(sinv_list), tc), dtype=np.float32)
    for i, v in enumerate(sinv_list):
        sinv[i, :] = v
    d = torch.from_numpy(data).cuda()
    s = torch.from_numpy(sinv).cuda()
    for odt, ocode in ((torch.float32, oracle.FP32), (torch.bfloat16, oracle.BF16)):
        got = mx.dequantize(d, tile_scale_inv=s, out_dtype=odt)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_bits(got), oracle_bits(oracle.dequant_block128(data, sinv, ocode)))


# ------------------------------------------- full-size workloads, sampled

def _sample_rows(rows, n, seed):
    g = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, size=n)]))


def test_large_bf16_8192_sampled(mx):
    """8192 x 8192 bf16 N(0, 0.02): every conversion at full size in the
    configuration the benchmark times; sampled rows and tile bands against
    the oracle, decode properties over the whole tensor."""
    x_np = syn.normal_bf16(8192, 8192)
    x = dev_bf16(x_np)
    y = mx.fake_quant_mxfp4(x)
    d, s = mx.mxfp8_row_direct(x, "swizzled")
    comp = mx.export_mxfp8(d, s, shape=x.shape, layout="swizzled")
    bd, bs = mx.fp8_block128_direct(x)
    dq = mx.dequantize(d, scales=s, layout="swizzled", out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    # properties over the whole tensor: row decode == projection (bit for bit),
    # blockwise decode == projection when the tile spread allows (N(0, .02) spreads stay small)
    assert torch.equal(dq.view(torch.int16), y.view(torch.int16))
    bq = mx.dequantize(bd, tile_scale_inv=bs, out_dtype=torch.float32)
    assert torch.equal(bq.view(torch.int32), y.float().view(torch.int32))
    rows = _sample_rows(8192, 40, 1)
    ref_y = oracle.fake_quant_mxfp4(x_np[rows])
    np.testing.assert_array_equal(host_bits(y[rows]), ref_y)
    rd, rs = oracle.mxfp8_row_direct(x_np[rows])
    np.testing.assert_array_equal(host_bits(d[rows]), rd)
    np.testing.assert_array_equal(host_bits(comp.scale_inv[rows]), rs)
    for band in (0, 31, 63):
        sl = slice(band * 128, band * 128 + 128)
        rd, rs = oracle.fp8_block128_direct(x_np[sl])
        np.testing.assert_array_equal(host_bits(bd[sl]), rd)
        np.testing.assert_array_equal(host_bits(bs[band]), rs.view(np.uint32)[0])


def test_large_bf16_columnwise_and_packed_sampled(mx):
    """8192 x 8192 bf16: MXFP8 columnwise (swizzled transposed scales) and
    packed MXFP4 at full size; sampled 32-row bands against the oracle, and
    over the whole tensor the packed form decodes to the projection."""
    x_np = syn.normal_bf16(8192, 8192)
    x = dev_bf16(x_np)
    cd, cs = mx.mxfp8_col_direct(x, "compact")
    cd2, cs2 = mx.mxfp8_col_direct(x, "swizzled")
    p, ps = mx.mxfp4_pack(x, "swizzled")
    y = mx.fake_quant_mxfp4(x)
    back = mx.dequantize(p, scales=ps, layout="swizzled", out_dtype=torch.bfloat16, mxfp4_K=8192)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), y.view(torch.int16))
    assert torch.equal(cd, cd2)
    comp = mx.export_mxfp8(torch.empty((8192, 8192), dtype=torch.uint8, device="cuda"), cs2, shape=(8192, 8192),
                           layout="swizzled")
    torch.cuda.synchronize()
    assert torch.equal(comp.scale_inv, cs)
    for band in (0, 101, 255):
        sl = slice(band * 32, band * 32 + 32)
        rd, rs = oracle.mxfp8_col_direct(x_np[sl])
        np.testing.assert_array_equal(host_bits(cd[sl]), rd)
        np.testing.assert_array_equal(host_bits(cs[:, band]), rs[:, 0])


def _tile_spread(x_np):
    """Spread of the 1x32 block exponents (finite, nonzero blocks) per 128x128 tile."""
    rows, K = x_np.shape
    a = np.abs(x_np.astype(np.float64)).reshape(rows, K // 32, 32).max(axis=2)
    with np.errstate(divide="ignore"):
        e = np.ceil(np.log2(a / 6.0))
    e = np.clip(e, -126, 125)
    e[a == 0] = np.nan
    e = e.reshape(rows // 128, 128, K // 128, 4).transpose(0, 2, 1, 3).reshape(rows // 128, K // 128, -1)
    import warnings

    with np.errstate(invalid="ignore"), warnings.catch_warnings():
        warnings.simplefilter("ignore", RuntimeWarning)  # the planted all-zero tiles have no exponent
        return np.nanmax(e, axis=2) - np.nanmin(e, axis=2)


def test_spread_sweep_fp32_8192(mx):
    """128x128 tiles of E2M1 payloads with block exponents spread by d in
    0..16: the blockwise decode equals the projection through spread 14
    (TE PR #3264, "Test results (B200)"); sampled bands against the oracle."""
    x_np, _ = syn.spread_tiles_fp32()
    x = dev_f32(x_np)
    bd, bs = mx.fp8_block128_direct(x)
    y = mx.fake_quant_mxfp4(x)
    bq = mx.dequantize(bd, tile_scale_inv=bs, out_dtype=torch.float32)
    torch.cuda.synchronize()
    eq = (bq.view(torch.int32) == y.view(torch.int32)).view(64, 128, 64, 128).all(dim=3).all(dim=1).cpu().numpy()
    spread = _tile_spread(x_np)
    with np.errstate(invalid="ignore"):
        assert eq[spread <= 14].all()
        assert (~eq[spread >= 15]).any()
    for band in (0, 17, 63):
        sl = slice(band * 128, band * 128 + 128)
        rd, rs = oracle.fp8_block128_direct(x_np[sl])
        np.testing.assert_array_equal(host_bits(bd[sl]), rd)
        np.testing.assert_array_equal(host_bits(bs[band]), rs.view(np.uint32)[0])


@pytest.mark.parametrize("seed", [1004, 77])
def test_spread_tiles_bf16(mx, seed):
    """The spread-sweep tiles in bf16 (1024 x 1024): tiles on both sides of
    every fast-path condition of the blockwise kernel (tile exponent above or
    below 6, block exponents within or beyond 4 of the tile maximum), all
    conversions against the oracle."""
    x32, _ = syn.spread_tiles_fp32(rows=1024, K=1024, seed=seed)
    run_all_and_compare(mx, syn.f32_to_bf16_bits(x32), layouts=(oracle.SWIZZLED,))


def test_moe_expert_stack_export(mx):
    """32 experts x 4096 x 7184 bf16 (K % 32 = 16, 225 scale columns):
    MXFP8 rowwise into the GEMM-swizzled layout, then export; sampled
    experts against the oracle, swizzle invariance over the whole stack."""
    E, R, K = syn.MOE_EXPERTS, syn.MOE_ROWS, syn.MOE_K
    x = torch.empty((E, R, K), dtype=torch.bfloat16, device="cuda")
    host = {}
    for e in range(E):
        xe = syn.moe_expert_bf16(e)
        if e in (0, 13, 31):
            host[e] = xe
        x[e].copy_(dev_bf16(xe))
    d, s = mx.mxfp8_row_direct(x, "swizzled")
    comp = mx.export_mxfp8(d, s, shape=x.shape, layout="swizzled")
    _, s_compact = mx.mxfp8_row_direct(x, "compact")
    torch.cuda.synchronize()
    assert comp.scale_inv.shape == (E, R, 225) and not comp.is_view
    assert torch.equal(comp.scale_inv, s_compact)
    # padding columns 225..227 of the swizzled buffer are zero
    r = torch.arange(E * R, device="cuda", dtype=torch.int64)[:, None]
    j = torch.tensor([225, 226, 227], device="cuda", dtype=torch.int64)[None, :]
    off = ((r // 128) * 57 + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4
    assert int(s.view(-1)[off.view(-1)].max()) == 0
    for e, xe in host.items():
        rows = _sample_rows(R, 12, e)
        rd, rs = oracle.mxfp8_row_direct(xe[rows])
        np.testing.assert_array_equal(host_bits(d[e][rows]), rd)
        np.testing.assert_array_equal(host_bits(comp.scale_inv[e][rows]), rs)


# ---------------------------------------------------------- size limits

def test_grid_loops_past_65535_row_tiles(mx):
    """8,388,736 x 32 bf16: 65,537 tiles of 128 rows and 262,148 bands of 32
    rows, more than one grid dimension holds, so the blockwise, columnwise
    (conversion and dequantize) and export kernels loop over their grid;
    sampled tile bands against the oracle."""
    rows, K = 65537 * 128, 32
    base = syn.normal_bf16(4096, K, seed=61)
    x = dev_bf16(base).repeat(rows // 4096 + 1, 1)[:rows].contiguous()
    bd, bs = mx.fp8_block128_direct(x)
    cd, cs = mx.mxfp8_col_direct(x, "compact")
    cdq = mx.dequantize(cd, scales=cs, layout="compact", out_dtype=torch.bfloat16, columnwise=True)
    d, s = mx.mxfp8_row_direct(x, "swizzled")
    comp = mx.export_mxfp8(d, s, shape=x.shape, layout="swizzled")
    torch.cuda.synchronize()
    for band in (0, 4095, 65536):
        r0 = band * 128
        xb = np.concatenate([base, base])[r0 % 4096:r0 % 4096 + 128]
        rd, rs = oracle.fp8_block128_direct(xb)
        np.testing.assert_array_equal(host_bits(bd[r0:r0 + 128]), rd)
        assert int(host_bits(bs[band])[0]) == int(rs.view(np.uint32)[0, 0])
        cdd, css = oracle.mxfp8_col_direct(xb)
        np.testing.assert_array_equal(host_bits(cd[r0:r0 + 128]), cdd)
        np.testing.assert_array_equal(host_bits(cs[:, 4 * band:4 * band + 4]), css)
        want = oracle.dequant_mxfp8(np.ascontiguousarray(cdd.T), css, oracle.COMPACT, oracle.E4M3, oracle.BF16).T
        np.testing.assert_array_equal(host_bits(cdq[r0:r0 + 128]), oracle_bits(np.ascontiguousarray(want)))
        _, rcs = oracle.mxfp8_row_direct(xb)
        np.testing.assert_array_equal(host_bits(comp.scale_inv[r0:r0 + 128]), rcs)


def test_export_word_store_kernel_loops_over_row_tiles(mx):
    """320,000 x 160 bf16 (5 scale columns): 2500 row tiles, more than the
    word-store export kernel's resident grid, so its CTAs loop; the export
    equals the compact scales over the whole tensor and sampled rows,
    the last 1000 included, match the oracle."""
    rows, K = 2500 * 128, 160
    base = syn.normal_bf16(1000, K, seed=63)
    x = dev_bf16(base).repeat(rows // 1000, 1).contiguous()
    d, s = mx.mxfp8_row_direct(x, "swizzled")
    _, sc = mx.mxfp8_row_direct(x, "compact")
    comp = mx.export_mxfp8(d, s, shape=x.shape, layout="swizzled")
    torch.cuda.synchronize()
    assert torch.equal(comp.scale_inv.reshape(-1), sc.reshape(-1))
    _, ref = oracle.mxfp8_row_direct(base)
    got = host_bits(comp.scale_inv).reshape(rows, -1)
    for r0 in (0, 1000 * 137, rows - 1000):
        np.testing.assert_array_equal(got[r0:r0 + 1000], ref)


def test_tensor_over_4gib_sampled(mx):
    """A 65536 x 40960 bf16 weight (5.4 GB, 2.7e9 elements): projection and
    MXFP8 rowwise, sampled rows against the oracle (64-bit offsets)."""
    rows, K = 65536, 40960
    base = syn.normal_bf16(256, K, seed=62)
    x = dev_bf16(base).repeat(rows // 256, 1)
    y = mx.fake_quant_mxfp4(x)
    d, s = mx.mxfp8_row_direct(x, "compact")
    torch.cuda.synchronize()
    for r in (0, 255, 40000, 65535):
        xr = base[r % 256:r % 256 + 1]
        np.testing.assert_array_equal(host_bits(y[r:r + 1]), oracle.fake_quant_mxfp4(xr))
        rd, rs = oracle.mxfp8_row_direct(xr)
        np.testing.assert_array_equal(host_bits(d[r:r + 1]), rd)
        np.testing.assert_array_equal(host_bits(s[r:r + 1]), rs)
    del x, y, d, s
    torch.cuda.empty_cache()


# ------------------------------------------- grouped export, quantize+export

@pytest.mark.parametrize("K", [32 * 1023, 32 * 1301 - 16])
def test_export_wide_rows(mx, K):
    """Swizzled -> compact export of rows whose scale count is not a
    multiple of 4 and whose 128-row tile is wide: 1023 scale columns stage
    137 KB per tile in shared memory (an opt-in size), 1301 columns exceed
    the 160 KB cap and take the column-group kernel.  Also into a scale_out
    that starts one byte off a word boundary (byte stores)."""
    rows = 130
    g = np.random.default_rng(K)
    w = g.standard_normal((rows, K)).astype(np.float32) * np.float32(0.02)
    w *= np.ldexp(1.0, g.integers(-20, 20, size=(rows, 1))).astype(np.float32)
    x_np = syn.f32_to_bf16_bits(w)
    _, ref_compact = oracle.mxfp8_row_direct(x_np, oracle.COMPACT)
    d, s = mx.mxfp8_row_direct(dev_bf16(x_np), "swizzled")
    nb = (K + 31) // 32
    comp = mx.export_mxfp8(d, s, shape=(rows, K), layout="swizzled")
    raw = torch.full((rows * nb + 8,), 0xA5, dtype=torch.uint8, device="cuda")
    off = mx.export_mxfp8(d, s, shape=(rows, K), layout="swizzled", scale_out=raw[1:1 + rows * nb])
    torch.cuda.synchronize()
    want = ref_compact.reshape(rows, nb)
    np.testing.assert_array_equal(host_bits(comp.scale_inv).reshape(rows, nb), want)
    np.testing.assert_array_equal(host_bits(off.scale_inv).reshape(rows, nb), want)
    r = host_bits(raw)
    assert r[0] == 0xA5 and (r[1 + rows * nb:] == 0xA5).all()


def _random_swizzled(rows, K, seed):
    """A swizzled scale buffer of random bytes, padding included (an export
    must never read the padding into its output)."""
    n = oracle.scale_bytes(rows, K, oracle.SWIZZLED)
    return np.random.default_rng(seed).integers(0, 256, size=n, dtype=np.uint8)


@pytest.mark.parametrize("rows", [1, 31, 127, 128, 129, 300])
def test_export_chunk_path_every_scale_count(mx, rows):
    """Swizzled -> compact export over scale counts 16..70, 100, 225, 256,
    1023 (every nb % 16, nb % 4 and row offset mod 16), ragged last row
    tiles, random bytes in the padding: equal to the oracle's export.  Also
    into outputs 1, 4 and 8 bytes off a 16-byte boundary (the word and byte
    kernels)."""
    for nb in list(range(16, 71)) + [100, 225, 256, 1023]:
        K = 32 * nb - (7 if nb % 3 == 0 else 0)
        sw = _random_swizzled(rows, K, seed=rows * 10000 + nb)
        want = oracle.export_scales(sw, oracle.SWIZZLED, rows, K)
        d = torch.from_numpy(sw).cuda()
        comp = mx.export_mxfp8(torch.empty((rows, K), dtype=torch.uint8, device="cuda"), d, shape=(rows, K),
                               layout="swizzled")
        outs = [comp.scale_inv]
        if nb in (16, 17, 225):
            for off in (1, 4, 8):
                raw = torch.full((rows * nb + 32,), 0xA5, dtype=torch.uint8, device="cuda")
                c = mx.export_mxfp8(torch.empty((rows, K), dtype=torch.uint8, device="cuda"), d, shape=(rows, K),
                                    layout="swizzled", scale_out=raw[off:off + rows * nb])
                outs.append(c.scale_inv)
                torch.cuda.synchronize()
                r = host_bits(raw)
                assert (r[:off] == 0xA5).all() and (r[off + rows * nb:] == 0xA5).all()
        torch.cuda.synchronize()
        for o in outs:
            np.testing.assert_array_equal(host_bits(o).reshape(rows, nb), want, err_msg=f"rows {rows} nb {nb}")


@pytest.mark.parametrize("nb", [16, 17, 63, 64, 128, 225, 240, 256, 257, 300, 512, 600, 1023])
def test_export_bulk_path(mx, nb):
    """Large swizzled exports take the bulk kernel (each row tile staged in
    shared memory by one bulk copy, its compact rows written back by one
    bulk store per 64-row part): 801 row tiles, so widths with the rotated
    chunk order (63, 64, 128, 256, 257, 512; 63 and 257 also take the
    separate row-crossing step) and unrotated widths of 192 columns or more
    (225, 240, 300) go bulk, while 16 and 17 (narrow, unrotated) and 600 and
    1023 (staging too large) stay on the chunk kernel.  The last row tile
    is ragged (77 rows: its second part holds 13 rows, and rows x nb ends
    off a 16-byte boundary for odd nb); random swizzled bytes.  Equal to the
    oracle's export, written at the start of its buffer and 16 bytes into
    one, with the bytes around it untouched; the same weight split into
    three storages through the grouped export likewise."""
    rows = 800 * 128 + 77
    K = 32 * nb - 5
    sw = _random_swizzled(rows, K, seed=nb)
    want = oracle.export_scales(sw, oracle.SWIZZLED, rows, K)
    d = torch.from_numpy(sw).cuda()
    payload = torch.empty((rows, K), dtype=torch.uint8, device="cuda")  # aliased by the export, never read
    comp = mx.export_mxfp8(payload, d, shape=(rows, K), layout="swizzled")
    raw = torch.full((rows * nb + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    c16 = mx.export_mxfp8(payload, d, shape=(rows, K), layout="swizzled", scale_out=raw[16:16 + rows * nb])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(comp.scale_inv).reshape(rows, nb), want)
    np.testing.assert_array_equal(host_bits(c16.scale_inv).reshape(rows, nb), want)
    r = host_bits(raw)
    assert (r[:16] == 0xA5).all() and (r[16 + rows * nb:] == 0xA5).all()
    # the same weight as three storages, split at row tiles (each piece a
    # swizzled buffer of its own): the grouped kernel's bulk path
    ct = (nb + 3) // 4
    cuts = [0, 250 * 128, 600 * 128, rows]
    items = [{"data": payload[a:b], "scales": d[(a // 128) * ct * 512:((b + 127) // 128) * ct * 512],
              "shape": (b - a, K), "layout": "swizzled"} for a, b in zip(cuts, cuts[1:])]
    gout = torch.full((rows * nb + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    mx.export_mxfp8_grouped(items, scale_out=gout[16:16 + rows * nb])
    torch.cuda.synchronize()
    g = host_bits(gout)
    np.testing.assert_array_equal(g[16:16 + rows * nb].reshape(rows, nb), want)
    assert (g[:16] == 0xA5).all() and (g[16 + rows * nb:] == 0xA5).all()


def test_export_chunk_path_past_65535_row_tiles(mx):
    """8,388,736 rows x 16 scale columns (65,537 row tiles of random
    swizzled bytes, 134 MB): the chunk kernel's grid walks the row tiles,
    as does the grouped kernel with the same storage beside two small ones;
    sampled tiles against the oracle, grouped against single over all."""
    rows, K = 65537 * 128, 512
    nb = 16
    sw = _random_swizzled(rows, K, seed=65537)
    d = torch.from_numpy(sw).cuda()
    payload = torch.empty((rows, K), dtype=torch.uint8, device="cuda")  # aliased by the export, never read
    comp = mx.export_mxfp8(payload, d, shape=(rows, K), layout="swizzled")
    small = [(300, 7184), (129, 640)]
    small_sw = [torch.from_numpy(_random_swizzled(r, k, seed=r + k)).cuda() for r, k in small]
    grouped = mx.export_mxfp8_grouped(
        [{"data": torch.empty((r, k), dtype=torch.uint8, device="cuda"), "scales": t, "shape": (r, k),
          "layout": "swizzled"} for (r, k), t in zip(small, small_sw)] +
        [{"data": payload, "scales": d, "shape": (rows, K), "layout": "swizzled"}])
    torch.cuda.synchronize()
    assert torch.equal(grouped[2].scale_inv, comp.scale_inv)
    tile = oracle.scale_bytes(128, K, oracle.SWIZZLED)
    got = host_bits(comp.scale_inv).reshape(rows, nb)
    for t in (0, 1, 40000, 65535, 65536):
        want = oracle.export_scales(sw[t * tile:(t + 1) * tile], oracle.SWIZZLED, 128, K)
        np.testing.assert_array_equal(got[t * 128:(t + 1) * 128], want)
    for (r, k), t, c in zip(small, small_sw, grouped[:2]):
        np.testing.assert_array_equal(host_bits(c.scale_inv).reshape(r, -1),
                                      oracle.export_scales(host_bits(t), oracle.SWIZZLED, r, k))


def test_grouped_export_matches_single_exports(mx):
    """Per-expert export of separate storages in one launch (compact view,
    padded view, padded copy, swizzled copies of different shapes) equals
    the oracle's export of each (TE PR #3790: per-expert export)."""
    cases = [((100, 48), "swizzled"), ((64, 16), "padded"), ((128, 128), "padded"), ((300, 7184 // 4), "swizzled"),
             ((37, 96), "compact"), ((256, 7184), "swizzled")]
    storages, refs = [], []
    for i, (shape, lay) in enumerate(cases):
        x_np = syn.normal_bf16(*shape, seed=500 + i)
        d, s = mx.mxfp8_row_direct(dev_bf16(x_np), lay)
        storages.append({"data": d, "scales": s, "shape": shape, "layout": lay, "fp8": "e4m3" if i % 2 else "e5m2"})
        refs.append(oracle.mxfp8_row_direct(x_np, oracle.COMPACT)[1])
    comps = mx.export_mxfp8_grouped(storages)
    torch.cuda.synchronize()
    for (shape, lay), c, ref, st in zip(cases, comps, refs, storages):
        np.testing.assert_array_equal(host_bits(c.scale_inv).reshape(ref.shape), ref)
        nb = -(-shape[1] // 32)
        assert c.is_view == (lay == "compact" or (lay == "padded" and nb % 4 == 0))
        assert c.data.data_ptr() == st["data"].data_ptr()
    assert mx.export_mxfp8_grouped([]) == []


def test_grouped_bulk_export_many_tiles_per_cta(mx):
    """The grouped kernel's bulk path walks a storage's row tiles with a
    grid stride capped at 64 CTAs per SM, so a storage of more row tiles
    takes several per CTA through one mbarrier's alternating phases:
    1,300,000 rows x 64 scale columns (10,157 row tiles, rotated chunk
    order, random swizzled bytes), beside a storage of 100 scale columns
    (unrotated and narrow: the chunk path) and two small storages the bulk
    path takes because the launch as a whole is large: one row of 225
    columns (a single partial part, its bytes past the last 16-byte boundary
    stored one by one) and 77 rows of 257 (rotated, with the row-crossing
    step).  Equal to the oracle's export."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, K = 1_300_000, 2048
    assert (rows + 127) // 128 > 64 * sms
    sw = _random_swizzled(rows, K, seed=64)
    small = [(300, 3195), (1, 7184), (77, 32 * 257 - 9)]
    small_sw = [_random_swizzled(r, k, seed=7 + i) for i, (r, k) in enumerate(small)]
    items = [{"data": torch.empty((rows, K), dtype=torch.uint8, device="cuda"),  # aliased, never read
              "scales": torch.from_numpy(sw).cuda(), "shape": (rows, K), "layout": "swizzled"}]
    items += [{"data": torch.empty((r, k), dtype=torch.uint8, device="cuda"), "scales": torch.from_numpy(t).cuda(),
               "shape": (r, k), "layout": "swizzled"} for (r, k), t in zip(small, small_sw)]
    comps = mx.export_mxfp8_grouped(items)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(comps[0].scale_inv).reshape(rows, -1),
                                  oracle.export_scales(sw, oracle.SWIZZLED, rows, K))
    for c, (r, k), t in zip(comps[1:], small, small_sw):
        np.testing.assert_array_equal(host_bits(c.scale_inv).reshape(r, -1), oracle.export_scales(t, oracle.SWIZZLED, r, k))


def test_grouped_export_past_one_launch(mx):
    """130 storages -- more than one launch of 128 -- mixing every path of
    the grouped kernel (chunk-path swizzled, other swizzled, padded copies,
    compact and padded views, empty storages), each equal to the oracle's
    export of its random scale bytes, copies packed in order into one
    scale_out."""
    g = np.random.default_rng(130)
    kinds = [(40, 7184, "swizzled"), (129, 160, "swizzled"), (64, 48, "padded"), (33, 96, "compact"),
             (128, 128, "padded"), (0, 64, "swizzled"), (17, 1056, "swizzled"), (1, 16, "padded")]
    storages, wants = [], []
    for i in range(130):
        rows, K, lay = kinds[i % len(kinds)]
        rows = rows + (i // len(kinds)) % 3 if rows else 0
        nbytes = oracle.scale_bytes(rows, K, {"compact": oracle.COMPACT, "padded": oracle.PADDED,
                                              "swizzled": oracle.SWIZZLED}[lay])
        sc = g.integers(0, 256, size=max(nbytes, 1), dtype=np.uint8)
        storages.append({"data": torch.empty((rows, K), dtype=torch.uint8, device="cuda"),
                         "scales": torch.from_numpy(sc).cuda(), "shape": (rows, K), "layout": lay})
        code = {"compact": oracle.COMPACT, "padded": oracle.PADDED, "swizzled": oracle.SWIZZLED}[lay]
        wants.append(oracle.export_scales(sc[:nbytes], code, rows, K) if rows else np.zeros((0, (K + 31) // 32),
                                                                                          np.uint8))
    comps = mx.export_mxfp8_grouped(storages)
    torch.cuda.synchronize()
    assert len(comps) == 130
    for i, (c, w) in enumerate(zip(comps, wants)):
        np.testing.assert_array_equal(host_bits(c.scale_inv).reshape(w.shape), w, err_msg=f"storage {i}")


@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_quantize_export_one_call(mx, dt):
    """Quantize a bf16 or fp32 weight and export it in one call (TE issue
    #3644, workflow 2): values and compact scales equal the oracle's."""
    x_np = syn.moe_expert_bf16(3, rows=512)
    if dt == "fp32":
        x_np = syn.bf16_bits_to_f32(x_np) * np.float32(3.0)  # not bf16-representable everywhere
    comp = mx.quantize_export_mxfp8(dev_input(x_np))
    torch.cuda.synchronize()
    rd, rs = oracle.mxfp8_row_direct(x_np)
    np.testing.assert_array_equal(host_bits(comp.data), rd)
    np.testing.assert_array_equal(host_bits(comp.scale_inv), rs)
    assert comp.is_view and comp.scale_inv.shape == (512, 225)


def test_prepared_exports_replay_in_a_graph(mx):
    """The prepared grouped export and one-call quantize+export capture into
    a CUDA graph; replays after the inputs change give the oracle's bytes."""
    xa, xb = syn.normal_bf16(256, 7184, seed=81), syn.normal_bf16(256, 7184, seed=82)
    x = dev_bf16(xa)
    d, s = mx.mxfp8_row_direct(x, "swizzled")
    out = torch.empty(256 * 225, dtype=torch.uint8, device="cuda")
    qd = torch.empty((256, 7184), dtype=torch.uint8, device="cuda")
    qs = torch.empty((256, 225), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls = [mx.plan_mxfp8_row_direct(x, "swizzled", d, s),
                 mx.plan_export_mxfp8_grouped([{"data": d, "scales": s, "shape": (256, 7184), "layout": "swizzled"}],
                                              scale_out=out)[0],
                 mx.plan_quantize_export_mxfp8(x, qd, qs)[0]]
        for c in calls:
            c()
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for c in calls:
                c()
    torch.cuda.current_stream().wait_stream(side)
    for xn in (xa, xb):
        x.copy_(dev_bf16(xn))
        g.replay()
        torch.cuda.synchronize()
        rd, rs = oracle.mxfp8_row_direct(xn)
        np.testing.assert_array_equal(host_bits(out).reshape(256, 225), rs)
        np.testing.assert_array_equal(host_bits(qd), rd)
        np.testing.assert_array_equal(host_bits(qs), rs)


# ------------------------------------------------------ skip-update flag

@pytest.mark.parametrize("dt", ["bf16", "fp32"])
def test_skip_flag_leaves_every_output_untouched(mx, dt):
    """A nonzero device flag makes the *_update converters write nothing --
    payloads, scales (padding included) and tile scales keep their bytes, for
    every form of the direct workspace: projection, MXFP8 rowwise, MXFP8
    columnwise (transposed swizzled scales), 128x128 blockwise (fp32: the
    pipelined kernel included) and packed MXFP4 (TE PR #3264, review: the
    skip flag gates the whole workspace refresh).  Rows = 200 leave padding
    in both the row and the transposed scale layouts."""
    R, K = 200, 512
    x = dev_bf16(syn.normal_bf16(R, K, seed=31))
    if dt == "fp32":
        x = x.float()
    skip = torch.ones(1, dtype=torch.int32, device="cuda")

    def filled(n, v=0x5A):
        return torch.full((n,), v, dtype=torch.uint8, device="cuda")

    y = torch.full((R, K), 1.0, dtype=x.dtype, device="cuda")
    d, s = filled(R * K).view(R, K), filled(mx.scale_bytes(R, K, "swizzled"))
    cd, cs = filled(R * K).view(R, K), filled(mx.scale_bytes(K, R, "swizzled"))
    pk, ps = filled(R * K // 2).view(R, K // 2), filled(mx.scale_bytes(R, K, "swizzled"))
    bd = filled(R * K).view(R, K)
    bs = torch.full((mx.tile_scale_count(R, K),), 3.0, dtype=torch.float32, device="cuda")

    def run_all():
        mx.fake_quant_mxfp4(x, out=y, skip=skip)
        mx.mxfp8_row_direct(x, "swizzled", data=d, scales=s, skip=skip)
        mx.mxfp8_col_direct(x, "swizzled", data=cd, scales=cs, skip=skip)
        mx.mxfp4_pack(x, "swizzled", packed=pk, scales=ps, skip=skip)
        mx.fp8_block128_direct(x, data=bd, tile_scale_inv=bs, skip=skip)

    run_all()
    torch.cuda.synchronize()
    assert bool((y == 1.0).all())
    for t in (d, s, cd, cs, pk, ps, bd):
        assert bool((t == 0x5A).all())
    assert bool((bs == 3.0).all())
    skip.zero_()
    run_all()
    ry = mx.fake_quant_mxfp4(x)
    rd, rs = mx.mxfp8_row_direct(x, "swizzled")
    rcd, rcs = mx.mxfp8_col_direct(x, "swizzled")
    rpk, rps = mx.mxfp4_pack(x, "swizzled")
    rbd, rbs = mx.fp8_block128_direct(x)
    torch.cuda.synchronize()
    iv = torch.int16 if dt == "bf16" else torch.int32
    assert torch.equal(y.view(iv), ry.view(iv))
    assert torch.equal(d, rd) and torch.equal(s, rs.reshape(-1))
    assert torch.equal(cd, rcd) and torch.equal(cs, rcs.reshape(-1))
    assert torch.equal(pk, rpk) and torch.equal(ps, rps.reshape(-1))
    assert torch.equal(bd, rbd) and torch.equal(bs.view(torch.int32), rbs.reshape(-1).view(torch.int32))
    # and the refreshed bytes are the oracle's (padding of both scale layouts zero)
    x_np = syn.normal_bf16(R, K, seed=31)
    if dt == "fp32":
        x_np = syn.bf16_bits_to_f32(x_np)
    ocd, ocs = oracle.mxfp8_col_direct(x_np, oracle.SWIZZLED)
    opk, ops = oracle.mxfp4_pack(x_np, oracle.SWIZZLED)
    np.testing.assert_array_equal(host_bits(cd), ocd)
    np.testing.assert_array_equal(host_bits(cs), ocs)
    np.testing.assert_array_equal(host_bits(pk), opk)
    np.testing.assert_array_equal(host_bits(ps), ops)


def test_skip_flag_in_a_captured_graph(mx):
    """The flag is read at replay: a graph captured once refreshes the cached
    weight -- MXFP8 rowwise, MXFP8 columnwise, 128x128 blockwise and packed
    MXFP4 -- when the flag is 0 and keeps every byte when it is 1 (TE PR
    #3264, review: skipped cached updates during CUDA-graph replay)."""
    R, K = 384, 1024
    x1 = syn.normal_bf16(R, K, seed=41)
    x2 = syn.normal_bf16(R, K, seed=42)
    x = dev_bf16(x1)
    skip = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = torch.empty((R, K), dtype=torch.uint8, device="cuda")
    s = torch.empty(mx.scale_bytes(R, K, "swizzled"), dtype=torch.uint8, device="cuda")
    cd = torch.empty((R, K), dtype=torch.uint8, device="cuda")
    cs = torch.empty(mx.scale_bytes(K, R, "swizzled"), dtype=torch.uint8, device="cuda")
    bd = torch.empty((R, K), dtype=torch.uint8, device="cuda")
    bs = torch.empty(mx.tile_scale_count(R, K), dtype=torch.float32, device="cuda")
    pk = torch.empty((R, K // 2), dtype=torch.uint8, device="cuda")
    ps = torch.empty(mx.scale_bytes(R, K, "swizzled"), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls = [mx.plan_mxfp8_row_direct(x, "swizzled", d, s, skip=skip),
                 mx.plan_mxfp8_col_direct(x, "swizzled", cd, cs, skip=skip),
                 mx.plan_fp8_block128_direct(x, bd, bs, skip=skip),
                 mx.plan_mxfp4_pack(x, "swizzled", pk, ps, skip=skip)]
        for c in calls:
            c()
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for c in calls:
                c()
    torch.cuda.current_stream().wait_stream(side)
    outs = (d, s, cd, cs, bd, bs, pk, ps)

    def want(xn):
        rd, rs = oracle.mxfp8_row_direct(xn, oracle.SWIZZLED)
        rcd, rcs = oracle.mxfp8_col_direct(xn, oracle.SWIZZLED)
        bdd, bss = oracle.fp8_block128_direct(xn)
        rpk, rps = oracle.mxfp4_pack(xn, oracle.SWIZZLED)
        return rd, rs, rcd, rcs, bdd, bss.view(np.uint32).reshape(-1), rpk, rps

    g.replay()
    torch.cuda.synchronize()
    w1 = want(x1)
    for got, ref in zip(outs, w1):
        np.testing.assert_array_equal(host_bits(got), ref)
    x.copy_(dev_bf16(x2))
    skip.fill_(1)
    g.replay()
    torch.cuda.synchronize()
    for got, ref in zip(outs, w1):  # kept
        np.testing.assert_array_equal(host_bits(got), ref)
    skip.zero_()
    g.replay()
    torch.cuda.synchronize()
    for got, ref in zip(outs, want(x2)):  # refreshed
        np.testing.assert_array_equal(host_bits(got), ref)


def test_packed_mxfp4_moe_expert_sampled(mx):
    """Packed MXFP4 of one 4096 x 7184 expert (K % 32 = 16, 225 scale
    columns) in the swizzled layout; sampled rows against the oracle."""
    xe = syn.moe_expert_bf16(7)
    x = dev_bf16(xe)
    p, s = mx.mxfp4_pack(x, "swizzled")
    pc, sc = mx.mxfp4_pack(x, "compact")
    comp = mx.export_mxfp8(torch.empty(x.shape, dtype=torch.uint8, device="cuda"), s, shape=x.shape, layout="swizzled")
    torch.cuda.synchronize()
    assert torch.equal(p, pc) and torch.equal(comp.scale_inv, sc)
    rows = _sample_rows(4096, 16, 7)
    rp, rs = oracle.mxfp4_pack(xe[rows])
    np.testing.assert_array_equal(host_bits(p[rows]), rp)
    np.testing.assert_array_equal(host_bits(sc[rows]), rs)


# ------------------------------------------------------- fast-math build

def test_concurrent_host_threads(mx):
    """Four host threads, each on its own CUDA stream, converting different
    weights at once through the C ABI (ctypes drops the GIL around the
    calls): the bytes equal those of one-thread runs."""
    import threading

    xs = [dev_bf16(syn.normal_bf16(512, 1024 + 32 * i, seed=70 + i)) for i in range(4)]
    want = []
    for x in xs:
        d, s = mx.mxfp8_row_direct(x, "swizzled")
        bd, bs = mx.fp8_block128_direct(x)
        cd, cs = mx.mxfp8_col_direct(x, "compact")
        want.append([host_bits(t) for t in (mx.fake_quant_mxfp4(x), d, s, bd, bs, cd, cs)])
    torch.cuda.synchronize()
    got = [None] * 4
    errors = []

    def work(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(20):
                    x = xs[i]
                    y = mx.fake_quant_mxfp4(x)
                    d, s = mx.mxfp8_row_direct(x, "swizzled")
                    bd, bs = mx.fp8_block128_direct(x)
                    cd, cs = mx.mxfp8_col_direct(x, "compact")
                st.synchronize()
                got[i] = [host_bits(t) for t in (y, d, s, bd, bs, cd, cs)]
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for i in range(4):
        for a, b in zip(got[i], want[i]):
            np.testing.assert_array_equal(a, b)


def test_fast_math_build_gives_identical_bytes(mx):
    """The same sources built with --use_fast_math give identical bytes
    (TE PR #3264, "Test results (B200)")."""
    fm = mxq.Library(fastmath=True)
    g = np.random.default_rng(8)
    u = g.integers(0, 0x7F800000, size=(256, 128), dtype=np.uint64).astype(np.uint32)
    u[::2] = (u[::2] & 0x807FFFFF) | (np.uint32(3) << np.uint32(23))  # subnormal-scale rows
    inputs = [syn.exhaustive_bf16(), u.view(np.float32), syn.spread_tiles_fp32(rows=256, K=512)[0]]
    for x_np in inputs:
        x = dev_input(x_np)
        for lib_a, lib_b in ((mx, fm),):
            assert torch.equal(lib_a.fake_quant_mxfp4(x).view(torch.uint8), lib_b.fake_quant_mxfp4(x).view(torch.uint8))
            for lay in ("compact", "swizzled"):
                da, sa = lib_a.mxfp8_row_direct(x, lay)
                db, sb = lib_b.mxfp8_row_direct(x, lay)
                assert torch.equal(da, db) and torch.equal(sa, sb)
                for odt in (torch.float32, torch.bfloat16):
                    qa = lib_a.dequantize(da, scales=sa, layout=lay, out_dtype=odt)
                    qb = lib_b.dequantize(db, scales=sb, layout=lay, out_dtype=odt)
                    assert torch.equal(qa.view(torch.uint8), qb.view(torch.uint8))
            da, sa = lib_a.fp8_block128_direct(x)
            db, sb = lib_b.fp8_block128_direct(x)
            assert torch.equal(da, db) and torch.equal(sa.view(torch.int32), sb.view(torch.int32))
            pa, qa = lib_a.mxfp4_pack(x, "swizzled")
            pb, qb = lib_b.mxfp4_pack(x, "swizzled")
            assert torch.equal(pa, pb) and torch.equal(qa, qb)
            K = x.shape[-1]
            assert torch.equal(lib_a.dequantize(pa, scales=qa, layout="swizzled", mxfp4_K=K).view(torch.int16),
                               lib_b.dequantize(pb, scales=qb, layout="swizzled", mxfp4_K=K).view(torch.int16))


def test_binding_rejects_short_buffers(mx):
    """The binding refuses, before any launch, scale buffers shorter than
    their layout, a tile-scale tensor of the wrong dtype or count, and a
    grouped export spread over tensors it cannot address (the C ABI sees
    only pointers, so these would be reads past a buffer's end)."""
    rows, K = 200, 7184
    x = dev_bf16(syn.normal_bf16(rows, K, seed=90))
    d, s = mx.mxfp8_row_direct(x, "swizzled")
    compact = s.reshape(-1)[: rows * 225].clone()
    with pytest.raises(ValueError):
        mx.dequantize(d, scales=compact, layout="swizzled")
    with pytest.raises(ValueError):
        mx.export_mxfp8(d, compact, shape=(rows, K), layout="swizzled")
    with pytest.raises(ValueError):
        mx.export_mxfp8_grouped([{"data": d, "scales": compact, "shape": (rows, K), "layout": "swizzled"}])
    cd, cs = mx.mxfp8_col_direct(x, "swizzled")
    with pytest.raises(ValueError):  # columnwise scales are sized for the transposed matrix
        mx.dequantize(cd, scales=cs.reshape(-1)[: mx.scale_bytes(K, rows, "compact") - 1].clone(), layout="compact",
                      columnwise=True)
    bd, bs = mx.fp8_block128_direct(x)
    with pytest.raises(ValueError):
        mx.dequantize(bd, tile_scale_inv=bs.half())
    with pytest.raises(ValueError):
        mx.dequantize(bd, tile_scale_inv=bs.reshape(-1)[:-1].clone())
    # the valid calls still run and agree
    a = mx.dequantize(d, scales=s, layout="swizzled")
    b = mx.dequantize(d, scales=mx.mxfp8_row_direct(x, "compact")[1], layout="compact")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
