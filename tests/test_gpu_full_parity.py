"""Full-size parity: the three large workloads compared with the CPU oracle
over every output byte (tolerance 0), in the configuration the benchmark
times.

  * 8192 x 8192 bf16, N(0, 0.02): projection, MXFP8 rowwise (swizzled
    scales), export, 128x128 blockwise, both dequantizes, MXFP8 columnwise
    (compact and swizzled transposed scales) and packed MXFP4;
  * the 8192 x 8192 fp32 spread sweep: 128x128 blockwise (payloads and tile
    scales of all 64 x 64 tiles), its dequantize and the projection;
  * the 32 x 4096 x 7184 bf16 MoE expert stack: MXFP8 rowwise payloads,
    GEMM-swizzled scales and the compact export of every expert, and the
    per-expert grouped export.

TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling recipes",
"Test results (B200)": the direct converters' payload and scale bytes are
bitwise equal to the reference path.

The oracle is the plain C of oracle/ unchanged.  It is run on host threads,
one 128-row slab (or 512-row expert slab) per task: its C functions are
called through ctypes, which releases the GIL, so the slabs convert in
parallel on every host core.  Each task compares its slab of every output
and reports the differing bytes; the test fails if any task found one.
"""

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import block_scaled_precision_x32_gb300 as mxq
import oracle
from block_scaled_precision_x32_gb300 import synthetic as syn
from tests.gpu_util import dev_bf16, dev_f32, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    return mxq.library()


def _diff(name, got, want):
    """None when equal, else a one-line description of the first difference."""
    got, want = np.asarray(got), np.asarray(want)
    if got.shape != want.shape:
        return f"{name}: shape {got.shape} != {want.shape}"
    if np.array_equal(got, want):
        return None
    g, w = got.reshape(-1), want.reshape(-1)
    idx = np.flatnonzero(g != w)
    return f"{name}: {idx.size} elements differ, first at flat index {idx[0]} (got {int(g[idx[0]]):#x}, " \
           f"want {int(w[idx[0]]):#x})"


def _run(check, tasks):
    """Run check(task) -> (messages, extra) on every host core; assert that
    no message names a difference; return the extras in task order."""
    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        res = list(ex.map(check, tasks))
    bad = [m for msgs, _ in res for m in msgs if m]
    assert not bad, f"{len(bad)} differences against the oracle:\n" + "\n".join(bad[:20])
    return [extra for _, extra in res]


def test_full_8192_bf16_every_byte(mx):
    """8192 x 8192 bf16 (seed 1003): every conversion of the library against
    the oracle over the whole tensor."""
    R = K = 8192
    x_np = syn.normal_bf16(R, K)
    x = dev_bf16(x_np)
    y = mx.fake_quant_mxfp4(x)
    d, s = mx.mxfp8_row_direct(x, "swizzled")
    comp = mx.export_mxfp8(d, s, shape=x.shape, layout="swizzled")
    dq = mx.dequantize(d, scales=s, layout="swizzled", out_dtype=torch.bfloat16)
    bd, bs = mx.fp8_block128_direct(x)
    bq = mx.dequantize(bd, tile_scale_inv=bs, out_dtype=torch.bfloat16)
    cd, cs = mx.mxfp8_col_direct(x, "compact")
    _, css = mx.mxfp8_col_direct(x, "swizzled")
    p, ps = mx.mxfp4_pack(x, "compact")
    torch.cuda.synchronize()
    g = {k: host_bits(v) for k, v in dict(y=y, d=d, s=s, ex=comp.scale_inv, dq=dq, bd=bd, bs=bs, bq=bq, cd=cd,
                                          cs=cs, css=css, p=p, ps=ps).items()}
    del x, y, d, s, comp, dq, bd, bs, bq, cd, cs, css, p, ps
    torch.cuda.empty_cache()
    seg = mx.scale_bytes(128, K, "swizzled")  # swizzled bytes of one 128-row band

    def check(i):
        sl = slice(128 * i, 128 * i + 128)
        xs = x_np[sl]
        m = [_diff(f"projection rows {sl}", g["y"][sl], oracle.fake_quant_mxfp4(xs))]
        rd, rc = oracle.mxfp8_row_direct(xs)
        m.append(_diff(f"MXFP8 rowwise payload rows {sl}", g["d"][sl], rd))
        m.append(_diff(f"MXFP8 rowwise swizzled scales band {i}", g["s"].reshape(-1)[seg * i:seg * (i + 1)],
                       oracle.scales_to_layout(rc, 128, K, oracle.SWIZZLED)))
        m.append(_diff(f"export compact scales rows {sl}", g["ex"][sl], rc))
        m.append(_diff(f"dequantize (MXFP8 rowwise) -> bf16 rows {sl}", g["dq"][sl],
                       oracle.dequant_mxfp8(rd, rc, oracle.COMPACT, oracle.E4M3, oracle.BF16)))
        bdd, bss = oracle.fp8_block128_direct(xs)
        m.append(_diff(f"128x128 payload rows {sl}", g["bd"][sl], bdd))
        m.append(_diff(f"128x128 tile scales band {i}", g["bs"][i], bss.view(np.uint32)[0]))
        m.append(_diff(f"dequantize (128x128) -> bf16 rows {sl}", g["bq"][sl],
                       oracle.dequant_block128(bdd, bss, oracle.BF16)))
        cdd, ccs = oracle.mxfp8_col_direct(xs)
        m.append(_diff(f"MXFP8 columnwise payload rows {sl}", g["cd"][sl], cdd))
        m.append(_diff(f"MXFP8 columnwise compact scales bands {4 * i}..{4 * i + 3}", g["cs"][:, 4 * i:4 * i + 4],
                       ccs))
        pp, pps = oracle.mxfp4_pack(xs)
        m.append(_diff(f"packed MXFP4 nibbles rows {sl}", g["p"][sl], pp))
        m.append(_diff(f"packed MXFP4 scales rows {sl}", g["ps"][sl], pps))
        return m, ccs

    col_scales = _run(check, range(R // 128))
    full = np.concatenate(col_scales, axis=1)  # the K x 256 transposed scale matrix
    miss = _diff("MXFP8 columnwise swizzled scales", g["css"].reshape(-1),
                 oracle.scales_to_layout(full, K, R, oracle.SWIZZLED))
    assert miss is None, miss


def test_full_spread_sweep_fp32_every_tile(mx):
    """The 8192 x 8192 fp32 spread sweep (seed 1004): the 128x128 blockwise
    payloads and tile scales of all 64 x 64 tiles (spreads 0..16, the planted
    zero, -0 and 2^-127 tiles), their fp32 dequantize and the projection."""
    R = K = 8192
    x_np, _ = syn.spread_tiles_fp32()
    x = dev_f32(x_np)
    bd, bs = mx.fp8_block128_direct(x)
    bq = mx.dequantize(bd, tile_scale_inv=bs, out_dtype=torch.float32)
    y = mx.fake_quant_mxfp4(x)
    torch.cuda.synchronize()
    g = {k: host_bits(v) for k, v in dict(bd=bd, bs=bs, bq=bq, y=y).items()}
    del x, bd, bs, bq, y
    torch.cuda.empty_cache()

    def check(i):
        sl = slice(128 * i, 128 * i + 128)
        xs = x_np[sl]
        bdd, bss = oracle.fp8_block128_direct(xs)
        return [_diff(f"128x128 payload rows {sl}", g["bd"][sl], bdd),
                _diff(f"128x128 tile scales band {i}", g["bs"][i], bss.view(np.uint32)[0]),
                _diff(f"dequantize (128x128) -> fp32 rows {sl}", g["bq"][sl],
                      oracle.dequant_block128(bdd, bss, oracle.FP32).view(np.uint32)),
                _diff(f"projection rows {sl}", g["y"][sl], oracle.fake_quant_mxfp4(xs).view(np.uint32))], None

    _run(check, range(R // 128))


def test_full_moe_expert_stack_every_byte(mx):
    """32 experts x 4096 x 7184 bf16 (K % 32 = 16: 225 scale columns, padded
    to 228): MXFP8 rowwise payloads and GEMM-swizzled scales of the whole
    stack, the compact export, and the grouped export of the 32 experts as
    separate storages, against the oracle on every expert."""
    E, Rw, K = syn.MOE_EXPERTS, syn.MOE_ROWS, syn.MOE_K
    nb = -(-K // 32)
    xh = np.empty((E, Rw, K), dtype=np.uint16)
    with ThreadPoolExecutor(max_workers=max(1, min(E, os.cpu_count() or 1))) as ex:
        for e, h in enumerate(ex.map(syn.moe_expert_bf16, range(E))):
            xh[e] = h
    x = torch.from_numpy(xh.view(np.int16)).view(torch.bfloat16).cuda()
    d, s = mx.mxfp8_row_direct(x, "swizzled")
    comp = mx.export_mxfp8(d, s, shape=x.shape, layout="swizzled")
    tile = mx.scale_bytes(128, K, "swizzled")  # 128 x 228 bytes per 128-row band
    per_expert = Rw // 128 * tile
    grouped = mx.export_mxfp8_grouped([{"data": d[e], "scales": s.reshape(-1)[e * per_expert:(e + 1) * per_expert],
                                        "shape": (Rw, K), "layout": "swizzled"} for e in range(E)])
    torch.cuda.synchronize()
    g_d, g_s, g_ex = host_bits(d), host_bits(s).reshape(-1), host_bits(comp.scale_inv)
    g_grp = np.stack([host_bits(c.scale_inv) for c in grouped])
    del x, d, s, comp, grouped
    torch.cuda.empty_cache()
    miss = _diff("grouped export of the 32 experts vs the single export", g_grp, g_ex)
    assert miss is None, miss
    slab = 512

    def check(task):
        e, r0 = task
        rows = slice(r0, r0 + slab)
        rd, rc = oracle.mxfp8_row_direct(xh[e, rows])
        t0 = (e * Rw + r0) // 128
        return [_diff(f"expert {e} payload rows {rows}", g_d[e, rows], rd),
                _diff(f"expert {e} export scales rows {rows}", g_ex[e, rows], rc),
                _diff(f"expert {e} swizzled scales bands {t0}..", g_s[t0 * tile:(t0 + slab // 128) * tile],
                      oracle.scales_to_layout(rc, slab, K, oracle.SWIZZLED))], None

    _run(check, [(e, r0) for e in range(E) for r0 in range(0, Rw, slab)])
    assert g_ex.shape == (E, Rw, nb)
