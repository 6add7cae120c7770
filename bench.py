"""Benchmark of the block-scaled conversion path on one 8192 x 8192 bf16 weight.

One step = the whole hot path once: MXFP4 projection, direct MXFP8 rowwise
(GEMM-swizzled scales), direct FP8 128x128 blockwise, dequantize (MXFP8
rowwise -> bf16) and export_components (swizzled -> compact scales), each a
single libmxq kernel.  Throughput is the algorithmic bytes of the five
conversions over the step time, in GB/s; each conversion (and every other
entry point of the library) is also timed alone and reported against the
measured HBM copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mxq|reference]
    python bench.py --profile NAME    # one conversion, 3 launches, small footprint (for ncu)

``--impl reference`` times the CPU oracle (the only reference this method
has) on a bounded sample of the same workload.  Under torchrun every rank
converts its own weight (weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import signal
import statistics
import subprocess
import sys
import threading
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
STEP_BYTES = sum(BYTES.values())
# The library's other entry points on the same weight, timed alone the same way.
EXTRA_BYTES = {
    "mxfp8_col": 2 * N + N + N // 32,
    "mxfp8_col_dequant_bf16": N + N // 32 + 2 * N,
    "mxfp8_col_dequant_fp32": N + N // 32 + 4 * N,
    "mxfp4_pack": 2 * N + N // 2 + N // 32,
    "mxfp4_dequant_bf16": N // 2 + N // 32 + 2 * N,
    "dequant_fp32": N + N // 32 + 4 * N,
    "dequant_block128_bf16": N + 4 * TILES + 2 * N,
    "dequant_block128_fp32": N + 4 * TILES + 4 * N,
    "quantize_export": 2 * N + N + N // 32,
}
KERNEL_FILES = {
    "projection": "mxq_rowwise.cu",
    "mxfp8_row": "mxq_rowwise.cu",
    "block128": "mxq_block128.cu",
    "dequant_bf16": "mxq_dequant.cu",
    "export": "mxq_export.cu",
    "mxfp8_col": "mxq_colwise.cu",
    "mxfp8_col_dequant_bf16": "mxq_colwise.cu",
    "mxfp8_col_dequant_fp32": "mxq_colwise.cu",
    "mxfp4_pack": "mxq_rowwise.cu",
    "mxfp4_dequant_bf16": "mxq_dequant.cu",
    "dequant_fp32": "mxq_dequant.cu",
    "dequant_block128_bf16": "mxq_dequant.cu",
    "dequant_block128_fp32": "mxq_dequant.cu",
    "quantize_export": "mxq_rowwise.cu",
    "moe_export": "mxq_export.cu",
    "moe_grouped_export": "mxq_export.cu",
}
CSRC = os.path.join(ROOT, "block_scaled_precision_x32_gb300", "csrc")
# Launches per timed replay of one conversion: the inputs rotate over their
# resident copies LOOPS times, so the first launch's ramp is a small share.
LOOPS = 4


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
    """Per-kernel traffic per launch from the committed ncu summary, kept
    only while the kernel's sources are unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return {}
    with open(p) as f:
        d = json.load(f)
    out = {}
    for name, rec in d.get("kernels", {}).items():
        if name in KERNEL_FILES and rec.get("source_hash") == kernel_source_hash(name):
            out[name] = rec
    return out


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons every 100 ms
    over the whole GPU section.  Each sample carries nvidia-smi's own
    timestamp, so the samples inside each timed region (host wall times
    taken after synchronizing on both sides) are picked out afterwards."""

    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int, period_ms: int = 100):
        self.index, self.period_ms = index, period_ms
        self.samples = []  # (wall time, sm MHz, max sm MHz, power W, set of active reasons)
        self.regions = {}
        self.proc = self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True,
                bufsize=1)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            arrived = time.time()
            f = [c.strip() for c in line.split(",")]
            if len(f) < 8:
                continue
            try:
                t = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = arrived
            try:
                sm, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            try:
                pw = float(f[3])
            except ValueError:
                pw = None
            self.samples.append((t, sm, mx, pw, {nm for nm, v in zip(self.NAMES, f[4:8]) if v.lower() == "active"}))

    def stop(self):
        if self.proc is None:
            return
        self.proc.send_signal(signal.SIGINT)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait(timeout=5)
        if self.thread is not None:
            self.thread.join(timeout=5)

    def mark(self, name: str, t0: float, t1: float):
        self.regions[name] = (t0, t1)

    def summary(self, names=None):
        """Median SM clock, max clock, throttle reasons of the samples that
        fall inside the named regions (all regions by default)."""
        if self.proc is None:
            return None
        regs = [self.regions[n] for n in (self.regions if names is None else names) if n in self.regions]
        sel = [s for s in self.samples if any(a <= s[0] <= b for a, b in regs)]
        reasons = set()
        for s in sel:
            reasons |= s[4]
        pw = [s[3] for s in sel if s[3] is not None]
        return {"sm_mhz": statistics.median([s[1] for s in sel]) if sel else None,
                "sm_max_mhz": max((s[2] for s in self.samples), default=None),
                "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sel), "samples_total": len(self.samples)}


# ---------------------------------------------------------------- timing

def sync():
    import torch

    torch.cuda.synchronize()


def time_replays(g, per_replay: int, stream, world, clocks=None, name=None, min_reps: int = 50,
                 min_s: float = 0.3, max_reps: int = 20000):
    """Event-time each replay of CUDA graph g (per_replay launches of one
    conversion) on its own: at least min_reps replays and about min_s
    seconds of them.  Returns (median ms per launch, mean ms per launch,
    replays) -- the max over ranks of each."""
    import torch

    g.replay()
    sync()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(5):
        g.replay()
    b.record(stream)
    sync()
    est = max(a.elapsed_time(b) / 5, 1e-4)
    n = int(min(max_reps, max(min_reps, math.ceil(min_s * 1e3 / est))))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    barrier(world)
    sync()
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(2_000_000)  # ~1 ms of GPU time: the host gets ahead before the first event
    t0 = time.time()
    for ea, eb in evs:
        ea.record(stream)
        g.replay()
        eb.record(stream)
    sync()
    t1 = time.time()
    if clocks is not None and name is not None:
        clocks.mark(name, t0, t1)
    ts = [ea.elapsed_time(eb) / per_replay for ea, eb in evs]
    return max_over_ranks(statistics.median(ts), world), max_over_ranks(statistics.fmean(ts), world), n


class RawGraph:
    """A CUDA graph of prepared libmxq calls, captured and launched through
    the CUDA runtime API itself.  (torch's CUDAGraph.replay() also refills its
    random-generator seed and offset tensors -- two small kernels per replay
    -- which would sit inside the timed regions.)  replay() launches on the
    current torch stream."""

    _rt = None

    @classmethod
    def runtime(cls):
        if cls._rt is None:
            import ctypes
            import glob

            import torch

            cands = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcudart.so")]
            cands += sorted(glob.glob(os.path.join(os.path.dirname(os.path.dirname(torch.__file__)), "nvidia", "*",
                                                   "lib", "libcudart.so*")))
            cands += ["libcudart.so", "libcudart.so.13"]
            err = None
            for c in cands:
                try:
                    rt = ctypes.CDLL(c)
                    break
                except OSError as e:
                    err = e
            else:
                raise RuntimeError(f"libcudart not found: {err}")
            vp = ctypes.c_void_p
            rt.cudaStreamBeginCapture.argtypes = [vp, ctypes.c_int]
            rt.cudaStreamEndCapture.argtypes = [vp, ctypes.POINTER(vp)]
            rt.cudaGraphInstantiate.argtypes = [ctypes.POINTER(vp), vp, ctypes.c_ulonglong]
            rt.cudaGraphLaunch.argtypes = [vp, vp]
            rt.cudaGraphExecDestroy.argtypes = [vp]
            rt.cudaGraphDestroy.argtypes = [vp]
            cls._rt = rt
        return cls._rt

    def __init__(self, calls, stream):
        import ctypes

        rt = self.runtime()
        h = ctypes.c_void_p(stream.cuda_stream)

        def ok(code, what):
            if code != 0:
                raise RuntimeError(f"{what} failed with CUDA error {code}")

        ok(rt.cudaStreamBeginCapture(h, 0), "cudaStreamBeginCapture")  # global capture mode
        try:
            for c in calls:
                c()
        finally:
            self.graph = ctypes.c_void_p()
            ok(rt.cudaStreamEndCapture(h, ctypes.byref(self.graph)), "cudaStreamEndCapture")
        self.exe = ctypes.c_void_p()
        ok(rt.cudaGraphInstantiate(ctypes.byref(self.exe), self.graph, 0), "cudaGraphInstantiate")
        self._ok = ok

    def replay(self):
        import ctypes

        import torch

        self._ok(self.runtime().cudaGraphLaunch(self.exe, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)),
                 "cudaGraphLaunch")

    def __del__(self):
        rt = self._rt
        if rt is not None and getattr(self, "exe", None):
            rt.cudaGraphExecDestroy(self.exe)
            rt.cudaGraphDestroy(self.graph)


def capture(calls, stream):
    """One CUDA graph holding the given prepared calls, in order."""
    return RawGraph(calls, stream)


def capture_parallel(branches, streams, fork):
    """One CUDA graph whose branches run concurrently: branch i (a list of
    prepared calls planned on streams[i]) forks from streams[0] and joins it
    again.  The graph holds no other work than the calls."""
    import torch

    events = [torch.cuda.Event() for _ in streams]

    def body():
        fork.record(streams[0])
        for st in streams[1:]:
            st.wait_event(fork)
        for calls in branches:
            for c in calls:
                c()
        for ev, st in zip(events[1:], streams[1:]):
            ev.record(st)
            streams[0].wait_event(ev)

    return RawGraph([body], streams[0])


def record(name, nbytes, med_ms, mean_ms, reps, peak, clocks, in_step=None):
    us = med_ms * 1e3
    gbs = nbytes / (us * 1e-6) / 1e9
    rec = {"us": round(us, 2), "us_mean": round(mean_ms * 1e3, 2), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
           "bytes": nbytes, "replays": reps}
    if in_step is not None:
        rec["in_step"] = in_step
    c = clocks.summary([name]) if clocks is not None else None
    if c and c["sm_mhz"]:
        rec["sm_mhz"] = c["sm_mhz"]
        rec["clock_samples"] = c["samples"]
        rec["sm_kcycles"] = round(us * c["sm_mhz"] / 1e3, 2)  # us x MHz / 1000: thousands of SM cycles
    return rec


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, rank, world):
    import torch

    import block_scaled_precision_x32_gb300 as mxq
    from block_scaled_precision_x32_gb300 import synthetic as syn

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    lib = mxq.library()
    stream = torch.cuda.current_stream(dev)
    peak, peak_src = load_peaks()

    x_host = syn.normal_bf16(ROWS, COLS, seed=syn.SEED_BASE + 3 + 100 * rank)
    x0 = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).to(dev)
    R = 4  # resident input copies: no kernel reads bytes another touched within the last ~400 MB
    xs = [x0.clone() for _ in range(R)]
    y = torch.empty_like(x0)
    row_d = torch.empty((ROWS, COLS), dtype=torch.uint8, device=dev)
    row_s = torch.empty(lib.scale_bytes(ROWS, COLS, "swizzled"), dtype=torch.uint8, device=dev)
    blk_d = torch.empty_like(row_d)
    blk_s = torch.empty(lib.tile_scale_count(ROWS, COLS), dtype=torch.float32, device=dev)
    dq_in = [lib.mxfp8_row_direct(xs[i], "swizzled") for i in range(R)]
    blk_in = [lib.fp8_block128_direct(xs[i]) for i in range(R)]
    dq_out = torch.empty_like(x0)
    dq_out32 = torch.empty((ROWS, COLS), dtype=torch.float32, device=dev)
    ex_out = torch.empty(ROWS * NB, dtype=torch.uint8, device=dev)
    p4 = torch.empty((ROWS, COLS // 2), dtype=torch.uint8, device=dev)
    p4_s = torch.empty(lib.scale_bytes(ROWS, COLS, "swizzled"), dtype=torch.uint8, device=dev)
    p4_in = [lib.mxfp4_pack(xs[i], "swizzled") for i in range(R)]
    col_in = [lib.mxfp8_col_direct(xs[i], "swizzled") for i in range(R)]
    col_d = torch.empty_like(row_d)
    col_s = torch.empty(lib.scale_bytes(COLS, ROWS, "swizzled"), dtype=torch.uint8, device=dev)
    qe_s = torch.empty((ROWS, NB), dtype=torch.uint8, device=dev)
    sync()

    names = list(BYTES)
    extra = list(EXTRA_BYTES)
    # Prepared calls (arguments marshalled once), made on a side stream and
    # captured into CUDA graphs: one graph per input rotation holding the
    # step's five launches, and per conversion one graph of R back-to-back
    # launches over the R input copies.  Replays keep the host out of the
    # timed loop.
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    # the step's five conversions read independent inputs (dequantize and
    # export take an earlier rotation's MXFP8 form), so the step graph runs
    # them as concurrent branches, each planned on its own stream
    branch = [side] + [torch.cuda.Stream(dev) for _ in range(len(BYTES) - 1)]
    for b in branch[1:]:
        b.wait_stream(torch.cuda.current_stream(dev))
    step_plans = []
    for s in range(R):
        k = 3 * s
        dq_d, dq_s = dq_in[s]
        makers = [
            lambda: lib.plan_fake_quant_mxfp4(xs[k % R], y),
            lambda: lib.plan_mxfp8_row_direct(xs[(k + 1) % R], "swizzled", row_d, row_s),
            lambda: lib.plan_fp8_block128_direct(xs[(k + 2) % R], blk_d, blk_s),
            lambda: lib.plan_dequantize(dq_d, dq_out, scales=dq_s, layout="swizzled"),
            lambda: lib.plan_export_mxfp8(dq_d, dq_s, shape=(ROWS, COLS), layout="swizzled", scale_out=ex_out)[0],
        ]
        row = []
        for mk, st in zip(makers, branch):
            with torch.cuda.stream(st):
                row.append(mk())
        step_plans.append(row)
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
        extra_plans = [{
            "mxfp8_col": lib.plan_mxfp8_col_direct(xs[s], "swizzled", col_d, col_s),
            "mxfp8_col_dequant_bf16": lib.plan_dequantize(col_in[s][0], dq_out, scales=col_in[s][1],
                                                          layout="swizzled", columnwise=True),
            "mxfp8_col_dequant_fp32": lib.plan_dequantize(col_in[s][0], dq_out32, scales=col_in[s][1],
                                                          layout="swizzled", columnwise=True),
            "mxfp4_pack": lib.plan_mxfp4_pack(xs[s], "swizzled", p4, p4_s),
            "mxfp4_dequant_bf16": lib.plan_dequantize(p4_in[s][0], dq_out, scales=p4_in[s][1], layout="swizzled",
                                                      mxfp4=True),
            "dequant_fp32": lib.plan_dequantize(dq_in[s][0], dq_out32, scales=dq_in[s][1], layout="swizzled"),
            "dequant_block128_bf16": lib.plan_dequantize(blk_in[s][0], dq_out, tile_scale_inv=blk_in[s][1]),
            "dequant_block128_fp32": lib.plan_dequantize(blk_in[s][0], dq_out32, tile_scale_inv=blk_in[s][1]),
            "quantize_export": lib.plan_quantize_export_mxfp8(xs[s], row_d, qe_s)[0],
        } for s in range(R)]
        for s in range(2 * R):  # warm every launch configuration before capture
            for c in plans[s % R] + step_plans[s % R] + list(extra_plans[s % R].values()):
                c()
        for b in branch:
            b.synchronize()
        fork = torch.cuda.Event()
        step_graphs = [capture_parallel([[c] for c in step_plans[s]], branch, fork) for s in range(R)]
        conv_graphs = {nm: capture([plans[s][i] for s in range(R)] * LOOPS, side) for i, nm in enumerate(names)}
        for nm in extra:
            conv_graphs[nm] = capture([extra_plans[s][nm] for s in range(R)] * LOOPS, side)
    torch.cuda.current_stream(dev).wait_stream(side)
    sync()

    clocks = ClockSampler(dev.index).start()
    time.sleep(0.3)  # the sampler's first lines
    for s in range(args.warmup):
        step_graphs[s % R].replay()
    sync()

    # timed region 1: exactly `steps` steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    sync()
    w0 = time.time()
    t0.record(stream)
    for s in range(args.steps):
        step_graphs[s % R].replay()
    t1.record(stream)
    sync()
    clocks.mark("step", w0, time.time())
    barrier(world)
    elapsed_ms = t0.elapsed_time(t1)
    ms_step = max_over_ranks(elapsed_ms, world) / args.steps

    # timed region 2: each conversion alone, >= 50 individually timed replays
    # of R * LOOPS back-to-back launches and >= 0.3 s of them; the median is reported
    per_conv = {}
    for nm in names + extra:
        med, mean, n = time_replays(conv_graphs[nm], R * LOOPS, stream, world, clocks, nm)
        per_conv[nm] = record(nm, BYTES.get(nm, EXTRA_BYTES.get(nm)), med, mean, n, peak, clocks, nm in BYTES)
    del conv_graphs, step_graphs

    # the MoE expert stack: MXFP8 rowwise into swizzled scales, then export to compact
    moe = None if args.no_moe else run_moe(args, lib, dev, stream, world, clocks, peak)

    # the same conversions of an fp32 weight (fp32 master weights)
    fp32 = None if args.no_fp32 else run_fp32(args, lib, dev, stream, world, clocks, peak)
    clocks.stop()

    # end to end through the public API: pinned host weight in, every result back to pinned host memory
    e2e = None if args.no_e2e else run_e2e(args, lib, dev, x_host, world)

    if rank != 0:
        return None
    dom = max(names, key=lambda nm: per_conv[nm]["us"])
    traffic = load_traffic().get(dom, {})
    value = world * STEP_BYTES / (ms_step * 1e-3) / 1e9
    clk = clocks.summary()
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
                     "unit": "GB/s", "frac": per_conv[dom]["frac"], "traffic": traffic.get("traffic"),
                     "traffic_def": traffic.get("traffic_def"),
                     "dram_read": traffic.get("dram_read"), "dram_write": traffic.get("dram_write"),
                     "l2_write": traffic.get("l2_write"), "algorithmic_bytes": BYTES[dom]},
        "clocks": clk,
        "e2e": e2e,
        "moe": moe,
        "fp32": fp32,
        "gpu_launches": len(names) * args.steps,
        "timing": "CUDA events on the launch stream; steps replay one CUDA graph per input rotation (the 5 "
                  "launches as concurrent branches: the conversions read independent inputs); per_conversion: median over >= 50 individually event-timed replays (>= 0.3 s) of a graph "
                  "of 16 back-to-back launches over 4 rotating inputs (MoE: 16 over 8, fp32: 12 over 3); clocks: "
                  "nvidia-smi samples inside the timed regions",
    }


def run_moe(args, lib, dev, stream, world, clocks, peak):
    """32 experts x 4096 x 7184 bf16 (K % 32 = 16: 225 scale columns, padded
    to 228), each expert N(0, 0.02) * 2^U{-8..8} from its own seed.  Times
    the MXFP8 rowwise conversion of the whole stack into GEMM-swizzled scales
    (one launch, 2.8 GB of traffic, larger than L2), the export of those
    scales to compact (8 rotating copies of the 29.9 MB swizzled buffer, so
    reads come from HBM), and the same export with the 32 experts as
    separate storages (the grouped export, one launch per copy)."""
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
    per_expert = lib.scale_bytes(Rw, K, "swizzled")
    data = torch.empty((E, Rw, K), dtype=torch.uint8, device=dev)
    R = 8
    sw = [torch.empty(sbytes, dtype=torch.uint8, device=dev) for _ in range(R)]
    out = torch.empty(rows * nb, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        row = lib.plan_mxfp8_row_direct(x, "swizzled", data, sw[0])
        row()
        for i in range(1, R):
            sw[i].copy_(sw[0])
        exports = [lib.plan_export_mxfp8(data, sw[i], shape=(E, Rw, K), layout="swizzled", scale_out=out)[0]
                   for i in range(R)]
        grouped = [lib.plan_export_mxfp8_grouped(
            [{"data": data[e], "scales": sw[i][e * per_expert:(e + 1) * per_expert], "shape": (Rw, K),
              "layout": "swizzled"} for e in range(E)], scale_out=out)[0] for i in range(R)]
        for c in exports + grouped:
            c()
        side.synchronize()
        g_row, g_ex, g_grp = capture([row], side), capture(exports * 2, side), capture(grouped * 2, side)
    torch.cuda.current_stream(dev).wait_stream(side)
    sync()
    row_bytes = 3 * rows * K + sbytes
    ex_bytes = sbytes + rows * nb
    res = {"workload": f"MoE expert stack {E}x{Rw}x{K} bf16, N(0,0.02)*2^U{{-8..8}} per expert (synthetic)"}
    for nm, g, per, nbytes in (("moe_mxfp8_row", g_row, 1, row_bytes), ("moe_export", g_ex, 2 * R, ex_bytes),
                               ("moe_grouped_export", g_grp, 2 * R, ex_bytes)):
        med, mean, n = time_replays(g, per, stream, world, clocks, nm)
        res[{"moe_mxfp8_row": "mxfp8_row_swizzled", "moe_export": "export_swizzled_to_compact",
             "moe_grouped_export": "grouped_export_32_storages"}[nm]] = record(nm, nbytes, med, mean, n, peak, clocks)
    del x, data, sw, g_row, g_ex, g_grp
    torch.cuda.empty_cache()
    return res


def run_fp32(args, lib, dev, stream, world, clocks, peak):
    """The step's conversions and the columnwise / packed forms of an
    8192 x 8192 fp32 weight (N(0, 0.02), seed 1003), three rotating copies
    (800 MB, beyond L2), each conversion a CUDA graph of back-to-back
    launches timed as the bf16 conversions are."""
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
        "block128": (lambda x: lib.plan_fp8_block128_direct(x, bd, bs), 5 * N + 4 * TILES),
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
            graphs[nm] = (capture(calls * LOOPS, side), nbytes)
    torch.cuda.current_stream(dev).wait_stream(side)
    sync()
    out = {"workload": "8192x8192 fp32 weight (the bench weight widened), 3 rotating copies"}
    for nm, (g, nbytes) in graphs.items():
        med, mean, n = time_replays(g, R * LOOPS, stream, world, clocks, "fp32_" + nm)
        out[nm] = record("fp32_" + nm, nbytes, med, mean, n, peak, clocks)
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
    sync()
    n = max(1, min(args.steps, 10))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    sync()
    t0.record(main)
    for st in (s_in, s_cmp, s_out):
        st.wait_event(t0)
    for _ in range(n):
        step()
    for st in (s_in, s_cmp, s_out):
        main.wait_stream(st)
    t1.record(main)
    sync()
    ms = max_over_ranks(t0.elapsed_time(t1), world) / n
    d2h = sum(t.numel() * t.element_size() for t in host.values())
    return {"value": round(world * STEP_BYTES / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": int(xh.numel() * 2), "d2h_bytes_per_step": int(d2h), "steps": n,
            "pipeline": f"{chunks} row chunks over 3 streams (upload / convert / download)"}


# ------------------------------------------------- small driver for ncu

PROFILE_NAMES = ("projection", "mxfp8_row", "block128", "dequant_bf16", "export", "mxfp8_col",
                 "mxfp8_col_dequant_bf16", "mxfp8_col_dequant_fp32", "mxfp4_pack", "mxfp4_dequant_bf16", "dequant_fp32",
                 "dequant_block128_bf16", "dequant_block128_fp32", "quantize_export", "fp32_block128", "fp32_mxfp8_col",
                 "moe_export", "moe_grouped_export")


def run_profile(name: str, reps: int = 3):
    """One conversion of the benchmark, `reps` launches, with only the
    buffers it needs (at most about 1 GB on the device), for ncu captures of
    a single kernel.  The 8192 x 8192 weight (134 MB bf16, 268 MB fp32) is
    larger than L2.  The MoE exports take a 29.9 MB swizzled scale buffer
    of the expert stack's shape filled with random bytes (the copy moves
    bytes; their values do not change its work) and an uninitialised
    payload for the export to alias, without the 1.9 GB bf16 stack.
    Inputs of the timed kernel are produced first by other kernels."""
    import torch

    import block_scaled_precision_x32_gb300 as mxq
    from block_scaled_precision_x32_gb300 import synthetic as syn

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = mxq.library()
    if name.startswith("moe_"):
        E, Rw, K = syn.MOE_EXPERTS, syn.MOE_ROWS, syn.MOE_K
        rows, nb = E * Rw, -(-K // 32)
        g = torch.Generator(device=dev)
        g.manual_seed(1005)
        sw = torch.randint(0, 256, (lib.scale_bytes(rows, K, "swizzled"),), dtype=torch.uint8, device=dev,
                           generator=g)
        # the payload an export aliases (its bytes are never read: left uninitialised)
        data = torch.empty((E, Rw, K), dtype=torch.uint8, device=dev)
        out = torch.empty(rows * nb, dtype=torch.uint8, device=dev)
        if name == "moe_export":
            call = lib.plan_export_mxfp8(data, sw, shape=(E, Rw, K), layout="swizzled", scale_out=out)[0]
        else:
            pe = lib.scale_bytes(Rw, K, "swizzled")
            call = lib.plan_export_mxfp8_grouped(
                [{"data": data[e], "scales": sw[e * pe:(e + 1) * pe], "shape": (Rw, K), "layout": "swizzled"}
                 for e in range(E)], scale_out=out)[0]
    else:
        x = torch.from_numpy(syn.normal_bf16(ROWS, COLS).view(np.int16)).view(torch.bfloat16).to(dev)
        if name.startswith("fp32_"):
            x = x.float()
        u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device=dev)  # noqa: E731
        if name == "projection":
            call = lib.plan_fake_quant_mxfp4(x, torch.empty_like(x))
        elif name == "mxfp8_row":
            call = lib.plan_mxfp8_row_direct(x, "swizzled", u8(ROWS, COLS), u8(lib.scale_bytes(ROWS, COLS, 2)))
        elif name in ("block128", "fp32_block128"):
            call = lib.plan_fp8_block128_direct(x, u8(ROWS, COLS), torch.empty(TILES, dtype=torch.float32,
                                                                               device=dev))
        elif name in ("mxfp8_col", "fp32_mxfp8_col"):
            call = lib.plan_mxfp8_col_direct(x, "swizzled", u8(ROWS, COLS), u8(lib.scale_bytes(COLS, ROWS, 2)))
        elif name == "mxfp4_pack":
            call = lib.plan_mxfp4_pack(x, "swizzled", u8(ROWS, COLS // 2), u8(lib.scale_bytes(ROWS, COLS, 2)))
        elif name == "quantize_export":
            call = lib.plan_quantize_export_mxfp8(x, u8(ROWS, COLS), u8(ROWS, NB))[0]
        elif name in ("dequant_bf16", "dequant_fp32", "export"):
            d, s = lib.mxfp8_row_direct(x, "swizzled")
            del x
            if name == "export":
                call = lib.plan_export_mxfp8(d, s, shape=(ROWS, COLS), layout="swizzled", scale_out=u8(ROWS * NB))[0]
            else:
                out = torch.empty((ROWS, COLS), dtype=torch.bfloat16 if name == "dequant_bf16" else torch.float32,
                                  device=dev)
                call = lib.plan_dequantize(d, out, scales=s, layout="swizzled")
        elif name in ("dequant_block128_bf16", "dequant_block128_fp32"):
            d, s = lib.fp8_block128_direct(x)
            del x
            odt = torch.bfloat16 if name == "dequant_block128_bf16" else torch.float32
            call = lib.plan_dequantize(d, torch.empty((ROWS, COLS), dtype=odt, device=dev), tile_scale_inv=s)
        elif name in ("mxfp8_col_dequant_bf16", "mxfp8_col_dequant_fp32"):
            d, s = lib.mxfp8_col_direct(x, "swizzled")
            del x
            odt = torch.bfloat16 if name == "mxfp8_col_dequant_bf16" else torch.float32
            call = lib.plan_dequantize(d, torch.empty((ROWS, COLS), dtype=odt, device=dev), scales=s,
                                       layout="swizzled", columnwise=True)
        elif name == "mxfp4_dequant_bf16":
            p, s = lib.mxfp4_pack(x, "swizzled")
            del x
            call = lib.plan_dequantize(p, torch.empty((ROWS, COLS), dtype=torch.bfloat16, device=dev), scales=s,
                                       layout="swizzled", mxfp4=True)
        else:
            raise SystemExit(f"unknown --profile {name}; one of {', '.join(PROFILE_NAMES)}")
    sync()
    for _ in range(reps):
        call()
    sync()
    print(json.dumps({"profile": name, "launches": reps,
                      "device_bytes": torch.cuda.max_memory_allocated(dev)}), flush=True)


# --------------------------------------------------- CPU oracle (reference)

def oracle_sample(cols: int, rows: int = 128, seed: int = 1003, x=None):
    """One pass of the whole path through the CPU oracle on a rows x cols
    slab (multiples of 128) of the weight, or on the given slab x.  Returns
    (seconds, algorithmic bytes of the slab)."""
    import oracle
    from block_scaled_precision_x32_gb300 import synthetic as syn

    if x is None:
        x = syn.normal_bf16(rows, cols, seed=seed)
    rows, cols = x.shape
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


def cpu_baseline_one_core(budget_s: float = 12.0):
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


def cpu_baseline_full():
    """The whole 8192 x 8192 step (config: the bench weight, seed 1003)
    through the unchanged oracle on every host core: 64 slabs of 128 rows
    over one thread per core (the oracle's C functions run outside the GIL
    through ctypes).  Throughput = the step's algorithmic bytes / wall time
    of the conversions (generating the weight is not timed)."""
    import concurrent.futures as cf

    from block_scaled_precision_x32_gb300 import synthetic as syn

    x = syn.normal_bf16(ROWS, COLS)
    n = os.cpu_count() or 1
    oracle_sample(128, x=x[:128, :256])  # load the oracle library before the clock starts
    t = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        res = list(ex.map(lambda i: oracle_sample(COLS, x=x[128 * i:128 * i + 128]), range(ROWS // 128)))
    wall = time.perf_counter() - t
    nbytes = sum(b for _, b in res)
    return {"value": round(nbytes / wall / 1e9, 5), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"the whole 8192 x 8192 bf16 step (5 conversions, {nbytes / 1e6:.1f} MB) as 64 slabs of 128 "
                      f"rows over {n} threads (one per host core), the single-threaded C oracle unchanged, "
                      f"{wall:.1f} s wall"}


def _oracle_slab(task):
    cols, seed = task
    return oracle_sample(cols, seed=seed)


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
    ap.add_argument("--profile", choices=PROFILE_NAMES, help="run one conversion 3 times on a small footprint "
                                                               "(for ncu) and exit")
    args = ap.parse_args(argv)
    if args.profile:
        run_profile(args.profile)
        return 0
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
            res["cpu_baseline"] = cpu_baseline_full()
            res["cpu_baseline_one_core"] = cpu_baseline_one_core()
            if not args.no_moe:
                res["cpu_baseline_moe"] = cpu_baseline_moe()
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
