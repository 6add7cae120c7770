"""Benchmark of the block-scaled conversion path on one 8192 x 8192 bf16 weight.

One step = the whole hot path once: MXFP4 projection, direct MXFP8 rowwise
(GEMM-swizzled scales), direct FP8 128x128 blockwise, dequantize (MXFP8
rowwise -> bf16) and export_components (swizzled -> compact scales), each a
single libmxq kernel.  Throughput is the algorithmic bytes of the five
conversions over the step time, in GB/s; each conversion is also reported
against the measured HBM copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mxq|reference]

``--impl reference`` times the CPU oracle (the only reference this method
has) on a bounded sample of the same workload.  Under torchrun every rank
converts its own weight (weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GB/s and % of GB300 HBM roofline per conversion, 8192x8192 bf16"
ROWS = COLS = 8192
N = ROWS * COLS
NB = COLS // 32
TILES = (ROWS // 128) * (COLS // 128)
WORKLOAD = ("8192x8192 bf16 weight, N(0,0.02), seed 1003: MXFP4 projection + MXFP8 rowwise direct (swizzled "
            "scales) + FP8 128x128 blockwise direct + dequantize (MXFP8 rowwise -> bf16) + export (swizzled -> "
            "compact scales)")

# Algorithmic bytes of each conversion (read + write, once each).
BYTES = {
    "projection": 2 * N + 2 * N,
    "mxfp8_row": 2 * N + N + N // 32,
    "block128": 2 * N + N + 4 * TILES,
    "dequant_bf16": N + N // 32 + 2 * N,
    "export": 2 * (ROWS * NB),
}
KERNEL_FILES = {
    "projection": "mxq_rowwise.cu",
    "mxfp8_row": "mxq_rowwise.cu",
    "block128": "mxq_block128.cu",
    "dequant_bf16": "mxq_dequant.cu",
    "export": "mxq_export.cu",
    "mxfp8_col": "mxq_colwise.cu",
    "mxfp4_pack": "mxq_rowwise.cu",
    "mxfp4_dequant_bf16": "mxq_dequant.cu",
    "mxfp8_col_dequant_bf16": "mxq_colwise.cu",
}
STEP_BYTES = sum(BYTES.values())
# Conversions beyond the five of the step, timed alone the same way.
EXTRA_BYTES = {
    "mxfp8_col": 2 * N + N + N // 32,
    "mxfp4_pack": 2 * N + N // 2 + N // 32,
    "mxfp4_dequant_bf16": N // 2 + N // 32 + 2 * N,
    "mxfp8_col_dequant_bf16": N + N // 32 + 2 * N,
}
CSRC = os.path.join(ROOT, "block_scaled_precision_x32_gb300", "csrc")


def kernel_source_hash(name: str) -> str:
    h = hashlib.sha256()
    for f in (KERNEL_FILES[name], "mxq_device.cuh", "mxq_internal.h"):
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def load_traffic():
    """Per-kernel DRAM bytes per launch from the committed ncu summary, kept
    only while the kernel's sources are unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return {}
    with open(p) as f:
        d = json.load(f)
    out = {}
    for name, rec in d.get("kernels", {}).items():
        if name in KERNEL_FILES and rec.get("source_hash") == kernel_source_hash(name):
            out[name] = rec.get("dram_bytes_per_launch")
    return out


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            self.result = None
            return
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        self.result = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                       "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, rank, world):
    import torch

    import block_scaled_precision_x32_gb300 as mxq
    from block_scaled_precision_x32_gb300 import synthetic as syn

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    lib = mxq.library()
    stream = torch.cuda.current_stream(dev)

    x_host = syn.normal_bf16(ROWS, COLS, seed=syn.SEED_BASE + 3 + 100 * rank)
    x0 = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).to(dev)
    R = 4  # resident input copies: no kernel reads bytes another touched within the last ~400 MB
    xs = [x0.clone() for _ in range(R)]
    y = torch.empty_like(x0)
    row_d = torch.empty((ROWS, COLS), dtype=torch.uint8, device=dev)
    row_s = torch.empty(lib.scale_bytes(ROWS, COLS, "swizzled"), dtype=torch.uint8, device=dev)
    blk_d = torch.empty_like(row_d)
    blk_s = torch.empty(lib.tile_scale_count(ROWS, COLS), dtype=torch.float32, device=dev)
    dq_in = []
    for i in range(R):
        d, s = lib.mxfp8_row_direct(xs[i], "swizzled")
        dq_in.append((d, s))
    dq_out = torch.empty_like(x0)
    ex_out = torch.empty(ROWS * NB, dtype=torch.uint8, device=dev)
    p4 = torch.empty((ROWS, COLS // 2), dtype=torch.uint8, device=dev)
    p4_s = torch.empty(lib.scale_bytes(ROWS, COLS, "swizzled"), dtype=torch.uint8, device=dev)
    p4_in = [lib.mxfp4_pack(xs[i], "swizzled") for i in range(R)]
    p4_out = torch.empty_like(x0)
    col_in = [lib.mxfp8_col_direct(xs[i], "swizzled") for i in range(R)]
    col_out = torch.empty_like(x0)
    col_d = torch.empty_like(row_d)
    col_s = torch.empty(lib.scale_bytes(COLS, ROWS, "swizzled"), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    names = list(BYTES)
    extra = list(EXTRA_BYTES)
    # Prepared calls (arguments marshalled once), made on a side stream and
    # captured into CUDA graphs: one graph per input rotation holding the
    # step's five launches, and per conversion one graph of R back-to-back
    # launches.  Replays leave the host out of the timed loop.
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        plans = []
        for s in range(R):
            k = 3 * s
            dq_d, dq_s = dq_in[s]
            plans.append([
                lib.plan_fake_quant_mxfp4(xs[k % R], y),
                lib.plan_mxfp8_row_direct(xs[(k + 1) % R], "swizzled", row_d, row_s),
                lib.plan_fp8_block128_direct(xs[(k + 2) % R], blk_d, blk_s),
                lib.plan_dequantize(dq_d, dq_out, scales=dq_s, layout="swizzled"),
                lib.plan_export_mxfp8(dq_d, dq_s, shape=(ROWS, COLS), layout="swizzled", scale_out=ex_out)[0],
            ])
        extra_plans = [[lib.plan_mxfp8_col_direct(xs[s], "swizzled", col_d, col_s),
                        lib.plan_mxfp4_pack(xs[s], "swizzled", p4, p4_s),
                        lib.plan_dequantize(p4_in[s][0], p4_out, scales=p4_in[s][1], layout="swizzled", mxfp4=True),
                        lib.plan_dequantize(col_in[s][0], col_out, scales=col_in[s][1], layout="swizzled",
                                            columnwise=True)]
                       for s in range(R)]
        for s in range(2 * R):  # warm every launch configuration before capture
            for c in plans[s % R] + extra_plans[s % R]:
                c()
        side.synchronize()
        step_graphs, conv_graphs = [], []
        for s in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for c in plans[s]:
                    c()
            step_graphs.append(g)
        for i in range(len(names)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for s in range(R):
                    plans[s][i]()
            conv_graphs.append(g)
        for i in range(len(extra)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for s in range(R):
                    extra_plans[s][i]()
            conv_graphs.append(g)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()

    for s in range(args.warmup):
        step_graphs[s % R].replay()
    torch.cuda.synchronize()

    # timed region 1: exactly `steps` steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(dev.index) as clk:
        t0.record(stream)
        for s in range(args.steps):
            step_graphs[s % R].replay()
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = t0.elapsed_time(t1)
    ms_step = max_over_ranks(elapsed_ms, world) / args.steps

    # timed region 2: each conversion alone, R * ceil(steps / R) launches back to back
    reps = max(1, -(-args.steps // R))
    per = {}
    for i, nm in enumerate(names + extra):
        conv_graphs[i].replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            conv_graphs[i].replay()
        b.record(stream)
        torch.cuda.synchronize()
        per[nm] = max_over_ranks(a.elapsed_time(b), world) / (reps * R)

    # end to end through the public API: pinned host weight in, every result back to pinned host memory
    e2e = None if args.no_e2e else run_e2e(args, lib, dev, x_host, world)

    # the MoE expert stack: MXFP8 rowwise into swizzled scales, then export to compact
    moe = None if args.no_moe else run_moe(args, lib, dev, stream, world)

    # the same conversions of an fp32 weight (fp32 master weights)
    fp32 = None if args.no_fp32 else run_fp32(args, lib, dev, stream, world)

    if rank != 0:
        return None
    peak, peak_src = load_peaks()
    per_conv = {}
    for nm in names + extra:
        nbytes = BYTES.get(nm, EXTRA_BYTES.get(nm))
        us = per[nm] * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        per_conv[nm] = {"us": round(us, 2), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4), "bytes": nbytes,
                        "in_step": nm in BYTES}
    dom = max(names, key=lambda nm: per_conv[nm]["us"])
    traffic = load_traffic()
    value = world * STEP_BYTES / (ms_step * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows": ROWS, "K": COLS, "step_bytes": STEP_BYTES,
                   "l2": "inputs rotate over 4 resident copies of the 134 MB weight and of its MXFP8 form, so no "
                         "kernel reads bytes touched within the previous >400 MB of traffic (L2 is 129 MB)",
                   "parallelism": f"replicas{world}"},
        "per_conversion": per_conv,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": per_conv[dom]["GBps"], "peak": peak,
                     "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured" else peak_src,
                     "unit": "GB/s", "frac": per_conv[dom]["frac"], "traffic": traffic.get(dom),
                     "algorithmic_bytes": BYTES[dom]},
        "clocks": clk.result,
        "e2e": e2e,
        "moe": moe,
        "fp32": fp32,
        "gpu_launches": len(names) * args.steps,
        "timing": "CUDA events on the launch stream; steps replay one CUDA graph per input rotation (5 launches "
                  "each); per_conversion replays per-kernel graphs of back-to-back launches",
    }


def run_moe(args, lib, dev, stream, world):
    """32 experts x 4096 x 7184 bf16 (K % 32 = 16: 225 scale columns, padded
    to 228), each expert N(0, 0.02) * 2^U{-8..8} from its own seed.  Times
    the MXFP8 rowwise conversion of the whole stack into GEMM-swizzled scales
    (one launch, 2.8 GB of traffic, larger than L2) and the export of those
    scales to compact (8 rotating copies of the 29.9 MB swizzled buffer, so
    reads come from HBM)."""
    import concurrent.futures as cf

    import torch

    from block_scaled_precision_x32_gb300 import synthetic as syn

    E, Rw, K = syn.MOE_EXPERTS, syn.MOE_ROWS, syn.MOE_K
    rows, nb = E * Rw, -(-K // 32)
    x = torch.empty((E, Rw, K), dtype=torch.bfloat16, device=dev)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        for e, h in enumerate(ex.map(syn.moe_expert_bf16, range(E))):
            x[e].copy_(torch.from_numpy(h.view(np.int16)).view(torch.bfloat16))
    sbytes = lib.scale_bytes(rows, K, "swizzled")
    data = torch.empty((E, Rw, K), dtype=torch.uint8, device=dev)
    R = 8
    sw = [torch.empty(sbytes, dtype=torch.uint8, device=dev) for _ in range(R)]
    out = torch.empty(rows * nb, dtype=torch.uint8, device=dev)
    # prepared calls captured into CUDA graphs (as for the 8192 x 8192 step), so
    # host launch overhead stays out of the timed loop
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        row = lib.plan_mxfp8_row_direct(x, "swizzled", data, sw[0])
        row()
        for i in range(1, R):
            sw[i].copy_(sw[0])
        exports = [lib.plan_export_mxfp8(data, sw[i], shape=(E, Rw, K), layout="swizzled", scale_out=out)[0]
                   for i in range(R)]
        for c in exports:
            c()
        side.synchronize()
        g_row, g_ex = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_row, stream=side):
            row()
        with torch.cuda.graph(g_ex, stream=side):
            for c in exports:
                c()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    g_row.replay()
    g_ex.replay()
    torch.cuda.synchronize()

    def timed(fn, reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b), world) / reps

    row_reps = max(3, min(50, args.steps // 40))
    ex_reps = max(1, min(200, args.steps // 10))
    row_ms = timed(g_row.replay, row_reps)
    ex_ms = timed(g_ex.replay, ex_reps) / R
    peak, _ = load_peaks()
    row_bytes = 3 * rows * K + sbytes
    ex_bytes = sbytes + rows * nb
    del x, data, sw, g_row, g_ex
    torch.cuda.empty_cache()

    def rec(ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"us": round(ms * 1e3, 2), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4), "bytes": nbytes}

    return {"workload": f"MoE expert stack {E}x{Rw}x{K} bf16, N(0,0.02)*2^U{{-8..8}} per expert (synthetic)",
            "mxfp8_row_swizzled": rec(row_ms, row_bytes), "export_swizzled_to_compact": rec(ex_ms, ex_bytes),
            "reps": {"mxfp8_row": row_reps, "export": ex_reps * R}}


def run_fp32(args, lib, dev, stream, world):
    """The step's conversions and the columnwise / packed forms of an
    8192 x 8192 fp32 weight (N(0, 0.02), seed 1003), three rotating copies
    (800 MB, beyond L2), each conversion a CUDA graph of back-to-back
    launches timed with events."""
    import torch

    from block_scaled_precision_x32_gb300 import synthetic as syn

    R = 3
    w = syn.normal_bf16(ROWS, COLS, seed=syn.SEED_BASE + 3)  # the bf16 weight, widened exactly to fp32
    x0 = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).to(dev).float()
    xs = [x0.clone() for _ in range(R)]
    del x0
    y = torch.empty_like(xs[0])
    rd = torch.empty((ROWS, COLS), dtype=torch.uint8, device=dev)
    rs = torch.empty(lib.scale_bytes(ROWS, COLS, "swizzled"), dtype=torch.uint8, device=dev)
    bd = torch.empty_like(rd)
    bs = torch.empty(lib.tile_scale_count(ROWS, COLS), dtype=torch.float32, device=dev)
    cd = torch.empty_like(rd)
    cs = torch.empty(lib.scale_bytes(COLS, ROWS, "swizzled"), dtype=torch.uint8, device=dev)
    pk = torch.empty((ROWS, COLS // 2), dtype=torch.uint8, device=dev)
    ps = torch.empty_like(rs)
    conv = {
        "projection": (lambda x: lib.plan_fake_quant_mxfp4(x, y), 8 * N),
        "mxfp8_row": (lambda x: lib.plan_mxfp8_row_direct(x, "swizzled", rd, rs), 5 * N + N // 32),
        "block128": (lambda x: lib.plan_fp8_block128_direct(x, bd, bs), 5 * N + 4 * (ROWS // 128) * (COLS // 128)),
        "mxfp8_col": (lambda x: lib.plan_mxfp8_col_direct(x, "swizzled", cd, cs), 5 * N + N // 32),
        "mxfp4_pack": (lambda x: lib.plan_mxfp4_pack(x, "swizzled", pk, ps), 4 * N + N // 2 + N // 32),
    }
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graphs = {}
    with torch.cuda.stream(side):
        for nm, (mk, nbytes) in conv.items():
            calls = [mk(x) for x in xs]
            for c in calls:
                c()
            side.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for c in calls:
                    c()
            graphs[nm] = (g, nbytes)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    peak, _ = load_peaks()
    reps = max(3, min(100, args.steps // 20))
    out = {"workload": "8192x8192 fp32 weight (the bench weight widened), 3 rotating copies"}
    for nm, (g, nbytes) in graphs.items():
        g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(a.elapsed_time(b), world) / (reps * R)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[nm] = {"us": round(ms * 1e3, 2), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4), "bytes": nbytes}
    del xs, graphs
    torch.cuda.empty_cache()
    return out


def run_e2e(args, lib, dev, x_host, world, chunks: int = 2):
    """The same five conversions through the public API with the weight in
    pinned host memory and every result copied back to pinned host memory.
    The weight is cut into row chunks (multiples of 128 rows, so every
    scale layout splits into contiguous slices); chunk c's upload, its five
    conversions and its downloads run on three streams, so copies overlap
    the kernels and copies of the other chunk.  Two chunks measured best:
    each chunk adds eight copies, and 4 / 8 / 16 chunks were slower."""
    import torch

    rows_c = ROWS // chunks
    nbc = NB
    xh = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    host = {
        "y": torch.empty(xh.shape, dtype=torch.bfloat16).pin_memory(),
        "row_d": torch.empty(xh.shape, dtype=torch.uint8).pin_memory(),
        "row_s": torch.empty(lib.scale_bytes(ROWS, COLS, "swizzled"), dtype=torch.uint8).pin_memory(),
        "blk_d": torch.empty(xh.shape, dtype=torch.uint8).pin_memory(),
        "blk_s": torch.empty(lib.tile_scale_count(ROWS, COLS), dtype=torch.float32).pin_memory(),
        "dq": torch.empty(xh.shape, dtype=torch.bfloat16).pin_memory(),
        "ex": torch.empty(ROWS * nbc, dtype=torch.uint8).pin_memory(),
    }
    devb = {k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in host.items()}
    xd = torch.empty(xh.shape, dtype=torch.bfloat16, device=dev)
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def sl(name, c):  # chunk c of a buffer (every layout splits by 128-row bands)
        t = devb[name] if name != "x" else xd
        h = host[name] if name != "x" else xh
        if name in ("row_s",):
            n = lib.scale_bytes(rows_c, COLS, "swizzled")
            return t[c * n:(c + 1) * n], h[c * n:(c + 1) * n]
        if name == "blk_s":
            n = lib.tile_scale_count(rows_c, COLS)
            return t[c * n:(c + 1) * n], h[c * n:(c + 1) * n]
        if name == "ex":
            n = rows_c * nbc
            return t[c * n:(c + 1) * n], h[c * n:(c + 1) * n]
        return t[c * rows_c:(c + 1) * rows_c], h[c * rows_c:(c + 1) * rows_c]

    plans = []
    with torch.cuda.stream(s_cmp):
        for c in range(chunks):
            x_c, _ = sl("x", c)
            y_c, rd_c, rs_c = sl("y", c)[0], sl("row_d", c)[0], sl("row_s", c)[0]
            bd_c, bs_c, dq_c, ex_c = sl("blk_d", c)[0], sl("blk_s", c)[0], sl("dq", c)[0], sl("ex", c)[0]
            plans.append([
                lib.plan_fake_quant_mxfp4(x_c, y_c),
                lib.plan_mxfp8_row_direct(x_c, "swizzled", rd_c, rs_c),
                lib.plan_fp8_block128_direct(x_c, bd_c, bs_c),
                lib.plan_dequantize(rd_c, dq_c, scales=rs_c, layout="swizzled"),
                lib.plan_export_mxfp8(rd_c, rs_c, shape=(rows_c, COLS), layout="swizzled", scale_out=ex_c)[0],
            ])
    ev_in = [torch.cuda.Event() for _ in range(chunks)]
    ev_cmp = [torch.cuda.Event() for _ in range(chunks)]

    def step():
        for c in range(chunks):
            with torch.cuda.stream(s_in):
                d, h = sl("x", c)
                d.copy_(h, non_blocking=True)
                ev_in[c].record(s_in)
            s_cmp.wait_event(ev_in[c])
            for call in plans[c]:
                call()
            ev_cmp[c].record(s_cmp)
            s_out.wait_event(ev_cmp[c])
            with torch.cuda.stream(s_out):
                for name in host:
                    d, h = sl(name, c)
                    h.copy_(d, non_blocking=True)

    main = torch.cuda.current_stream(dev)
    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    n = max(1, min(args.steps, 10))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(main)
    for st in (s_in, s_cmp, s_out):
        st.wait_event(t0)
    for _ in range(n):
        step()
    for st in (s_in, s_cmp, s_out):
        main.wait_stream(st)
    t1.record(main)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world) / n
    d2h = sum(t.numel() * t.element_size() for t in host.values())
    return {"value": round(world * STEP_BYTES / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": int(xh.numel() * 2), "d2h_bytes_per_step": int(d2h), "steps": n,
            "pipeline": f"{chunks} row chunks over 3 streams (upload / convert / download)"}


# --------------------------------------------------- CPU oracle (reference)

def oracle_sample(cols: int, rows: int = 128, seed: int = 1003):
    """One pass of the whole path through the CPU oracle on a rows x cols
    slab (multiples of 128) of the weight.  Returns (seconds, algorithmic
    bytes of the slab)."""
    import oracle
    from block_scaled_precision_x32_gb300 import synthetic as syn

    x = syn.normal_bf16(rows, cols, seed=seed)
    t = time.perf_counter()
    oracle.fake_quant_mxfp4(x)
    d, s = oracle.mxfp8_row_direct(x, oracle.SWIZZLED)
    oracle.fp8_block128_direct(x)
    oracle.dequant_mxfp8(d, s, oracle.SWIZZLED, oracle.E4M3, oracle.BF16)
    oracle.export_scales(s, oracle.SWIZZLED, rows, cols)
    dt = time.perf_counter() - t
    return dt, STEP_BYTES * (rows * cols) / N


def _cols_for(budget_s: float) -> int:
    dt, _ = oracle_sample(512)  # calibrate on a 128 x 512 slab
    cols = int(budget_s / max(dt, 1e-4) * 512) // 128 * 128
    return max(128, min(cols, COLS))


def cpu_baseline(budget_s: float = 15.0):
    cols = _cols_for(budget_s)
    tot_t = tot_b = 0.0
    reps = 0
    while tot_t < budget_s and reps < 64:
        dt, nb = oracle_sample(cols, seed=1003 + reps)
        tot_t += dt
        tot_b += nb
        reps += 1
    return {"value": round(tot_b / tot_t / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} slab(s) of 128 x {cols} of the bf16 weight, whole step (5 conversions) each, "
                      f"single-threaded C oracle, {tot_t:.1f} s"}


def _oracle_slab(task):
    cols, seed = task
    return oracle_sample(cols, seed=seed)


def cpu_baseline_all_cores(budget_s: float = 10.0):
    """The same oracle on every host core at once: one process per core
    (spawned, so no CUDA state is inherited), each converting its own
    128-row slabs.  Throughput = all slabs' bytes / wall time of the pool's
    work (pool start-up and imports excluded by a warm-up task per worker)."""
    import multiprocessing as mp

    n = os.cpu_count() or 1
    cols = _cols_for(budget_s / 2)
    ctx = mp.get_context("spawn")
    with ctx.Pool(n) as pool:
        pool.map(_oracle_slab, [(128, 5000 + i) for i in range(n)])  # start every worker, load the oracle
        tasks = [(cols, 1003 + i) for i in range(2 * n)]
        t = time.perf_counter()
        res = pool.map(_oracle_slab, tasks, chunksize=1)
        wall = time.perf_counter() - t
    nbytes = sum(b for _, b in res)
    return {"value": round(nbytes / wall / 1e9, 5), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{len(tasks)} slabs of 128 x {cols} of the bf16 weight over {n} processes (one per core), "
                      f"whole step (5 conversions) each, the single-threaded C oracle unchanged, {wall:.1f} s wall"}


def _oracle_moe_slab(task):
    """The first `rows` rows of MoE expert `expert` (7184 bf16 columns)
    through the oracle: MXFP8 rowwise into swizzled scales, then the export
    to compact.  Returns (seconds, bytes by the GPU section's definitions of
    both conversions)."""
    import oracle
    from block_scaled_precision_x32_gb300 import synthetic as syn

    expert, rows = task
    x = syn.moe_expert_bf16(expert, rows=rows)  # row-major draws: the expert's first rows
    K = x.shape[1]
    t = time.perf_counter()
    _, s = oracle.mxfp8_row_direct(x, oracle.SWIZZLED)
    oracle.export_scales(s, oracle.SWIZZLED, rows, K)
    dt = time.perf_counter() - t
    return dt, 3 * rows * K + 2 * s.size + rows * (-(-K // 32))


def cpu_baseline_moe(rows: int = 512):
    """The MoE-stack conversions (rowwise into swizzled scales, then export)
    on the oracle, on bounded samples: a `rows`-row slab of one expert on one
    core, and one such slab of a different expert per host core at once."""
    import multiprocessing as mp

    from block_scaled_precision_x32_gb300 import synthetic as syn

    dt1, b1 = _oracle_moe_slab((0, rows))
    n = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(n) as pool:
        pool.map(_oracle_slab, [(128, 6000 + i) for i in range(n)])  # start every worker, load the oracle
        t = time.perf_counter()
        res = pool.map(_oracle_moe_slab, [(e % syn.MOE_EXPERTS, rows) for e in range(n)], chunksize=1)
        wall = time.perf_counter() - t
    nbytes = sum(b for _, b in res)
    return {"one_core": {"value": round(b1 / dt1 / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "seconds": round(dt1, 2)},
            "all_cores": {"value": round(nbytes / wall / 1e9, 5), "unit": "GB/s", "cores": n, "kind": "oracle",
                          "seconds": round(wall, 2)},
            "sample": f"{rows}-row slabs of the {syn.MOE_ROWS} x {syn.MOE_K} bf16 experts (one slab per process), "
                      f"MXFP8 rowwise into swizzled scales + export, the single-threaded C oracle unchanged"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    budget = min(3.0, 150.0 / max(1, args.steps + args.warmup))
    cols = _cols_for(budget)
    for w in range(args.warmup):
        oracle_sample(cols, seed=2000 + w)
    tot_t = tot_b = 0.0
    for s in range(args.steps):
        dt, nb = oracle_sample(cols, seed=1003 + s)
        tot_t += dt
        tot_b += nb
    value = tot_b / tot_t / 1e9
    sample = f"128 x {cols} slab of the bf16 weight per step, whole step (5 conversions), single-threaded C oracle"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / max(1, args.steps) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows": ROWS, "K": COLS, "sample": f"128x{cols}"},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return rank, world


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist

        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["mxq", "reference"], default="mxq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--no-moe", action="store_true", help="skip the MoE expert-stack measurement")
    ap.add_argument("--no-fp32", action="store_true", help="skip the fp32-weight measurement")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, world = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    init_dist(world, "nccl")
    res = run_gpu(args, rank, world)
    if res is not None:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
            res["cpu_baseline_all_cores"] = cpu_baseline_all_cores()
            if not args.no_moe:
                res["cpu_baseline_moe"] = cpu_baseline_moe()
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
