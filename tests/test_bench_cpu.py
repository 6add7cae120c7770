"""bench.py's host-side helpers without a GPU: the nvidia-smi sample parser,
the selection of samples inside timed regions, the algorithmic byte counts
and the traffic record the roofline reads."""

import json
import os

import bench


class _FakeSmi:
    def __init__(self, lines):
        self.stdout = iter(lines)


def test_clock_samples_are_parsed_with_their_own_timestamps():
    c = bench.ClockSampler(0)
    c.proc = _FakeSmi([
        "2026/12/03 05:29:32.000, 2070, 2070, 900.10, Not Active, Not Active, Not Active, Not Active\n",
        "2026/12/03 05:29:32.100, 1995, 2070, 1300.00, Not Active, Not Active, Not Active, Active\n",
        "2026/12/03 05:29:33.500, 1400, 2070, 1390.00, Active, Not Active, Not Active, Active\n",
        "not a sample\n",
        "2026/12/03 05:29:34.000, [N/A], 2070, 100.00, Not Active, Not Active, Not Active, Not Active\n",
    ])
    c._read()
    assert len(c.samples) == 3
    t0 = c.samples[0][0]
    assert abs(c.samples[1][0] - t0 - 0.1) < 1e-6
    c.mark("a", t0 - 0.01, t0 + 0.15)  # the first two samples
    c.mark("b", t0 + 1.4, t0 + 1.6)    # the third
    sa = c.summary(["a"])
    assert sa["samples"] == 2 and sa["sm_mhz"] == (2070.0 + 1995.0) / 2 and sa["reasons"] == ["sw_power_cap"]
    sb = c.summary(["b"])
    assert sb["samples"] == 1 and sb["sm_mhz"] == 1400.0 and sb["reasons"] == ["hw_slowdown", "sw_power_cap"]
    sall = c.summary()
    assert sall["samples"] == 3 and sall["samples_total"] == 3 and sall["sm_max_mhz"] == 2070.0
    assert sall["power_w_max"] == 1390.0


def test_algorithmic_bytes():
    n = 8192 * 8192
    assert bench.BYTES["projection"] == 4 * n
    assert bench.BYTES["mxfp8_row"] == 3 * n + n // 32 == 203_423_744
    assert bench.BYTES["block128"] == 3 * n + 4 * 64 * 64
    assert bench.BYTES["dequant_bf16"] == 3 * n + n // 32
    assert bench.BYTES["export"] == 2 * 8192 * 256
    assert bench.STEP_BYTES == 880_820_224
    assert bench.EXTRA_BYTES["dequant_fp32"] == 5 * n + n // 32
    assert bench.EXTRA_BYTES["mxfp8_col_dequant_fp32"] == 5 * n + n // 32
    assert bench.EXTRA_BYTES["dequant_block128_fp32"] == 5 * n + 4 * 64 * 64
    # every timed conversion names the source its kernel is built from and has a --profile driver
    for name in list(bench.BYTES) + list(bench.EXTRA_BYTES):
        assert name in bench.KERNEL_FILES and name in bench.PROFILE_NAMES, name


def test_traffic_record_matches_the_kernel_sources():
    """The committed ncu traffic is used only while the kernel's sources are
    unchanged; for the roofline kernel it must be on record and cover the
    algorithmic bytes (no write undercount)."""
    rec = bench.load_traffic()
    p = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    allk = json.load(open(p))["kernels"]
    for name, r in rec.items():
        assert r["source_hash"] == bench.kernel_source_hash(name)
        assert r["traffic"] == r["dram_read"] + r["l2_write"]
    assert "projection" in allk
    if "projection" in rec:
        assert rec["projection"]["traffic"] >= bench.BYTES["projection"]
