"""The C ABI without a GPU: the library builds, loads, exports every symbol
that include/mxq.h declares, and rejects bad arguments on the host before
touching CUDA (no kernel is launched by any call here)."""

import ctypes
import os
import re

import pytest

from block_scaled_precision_x32_gb300 import build as mxbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxq.h")

OK, INVALID, UNSUPPORTED, NO_ROWWISE, TOO_SMALL = 0, 1, 2, 3, 4


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MXQ_API\s+[\w\s\*]+?\b(mxq_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def libs():
    paths = mxbuild.build()
    return {name: ctypes.CDLL(p) for name, p in paths.items()}


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for s in ("mxq_fake_quant_mxfp4", "mxq_mxfp8_row_direct", "mxq_fp8_block128_direct", "mxq_export_mxfp8",
              "mxq_dequantize", "mxq_scale_bytes", "mxq_status_string"):
        assert s in syms


def test_every_declared_symbol_is_exported(libs):
    syms = declared_symbols()
    for name, lib in libs.items():
        for s in syms:
            assert hasattr(lib, s), f"{name} lacks {s}"


def test_library_is_for_sm103a_only():
    assert mxbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


class _Q(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("data", ctypes.c_void_p), ("rows", ctypes.c_int64), ("K", ctypes.c_int64),
                ("fp8", ctypes.c_int), ("scales", ctypes.c_void_p), ("lay", ctypes.c_int),
                ("tile_scale_inv", ctypes.c_void_p)]


class _S(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("fp8", ctypes.c_int), ("lay", ctypes.c_int),
                ("rows", ctypes.c_int64), ("K", ctypes.c_int64)]


class _C(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("fp8", ctypes.c_int), ("scales", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("K", ctypes.c_int64), ("scale_cols", ctypes.c_int64),
                ("is_view", ctypes.c_int)]


def _setup(L):
    i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    L.mxq_fake_quant_mxfp4.argtypes = [vp, vp, ci, i64, i64, i64, i64, vp]
    L.mxq_mxfp8_row_direct.argtypes = [vp, ci, i64, i64, i64, vp, vp, ci, vp]
    L.mxq_fp8_block128_direct.argtypes = [vp, ci, i64, i64, i64, vp, vp, vp]
    L.mxq_dequantize.argtypes = [ctypes.POINTER(_Q), vp, ci, vp]
    L.mxq_export_mxfp8.argtypes = [ctypes.POINTER(_S), vp, ctypes.c_size_t, ctypes.POINTER(_C), vp]
    L.mxq_scale_bytes.argtypes = [i64, i64, ci]
    L.mxq_scale_bytes.restype = ctypes.c_size_t
    L.mxq_tile_scale_count.argtypes = [i64, i64]
    L.mxq_tile_scale_count.restype = ctypes.c_size_t
    L.mxq_status_string.restype = ctypes.c_char_p
    return L


def test_sizes_and_strings(libs):
    L = _setup(libs["libmxq.so"])
    assert L.mxq_version() == 1
    assert L.mxq_scale_bytes(100, 48, 0) == 200          # compact (100, ceil(48/32) = 2)
    assert L.mxq_scale_bytes(100, 48, 1) == 128 * 4      # padded to (128, 4)
    assert L.mxq_scale_bytes(100, 48, 2) == 128 * 4      # swizzled: same bytes
    assert L.mxq_scale_bytes(32 * 4096, 7184, 2) == 32 * 4096 * 228
    assert L.mxq_scale_bytes(8192, 8192, 0) == 8192 * 256
    assert L.mxq_scale_bytes(0, 48, 1) == 0
    assert L.mxq_tile_scale_count(8192, 8192) == 64 * 64
    assert L.mxq_tile_scale_count(129, 130) == 4
    assert b"fp16" in L.mxq_status_string(UNSUPPORTED)
    assert L.mxq_status_string(99) == b"unknown status"


FAKE = 0x10000000  # never dereferenced: every call below fails or returns before any launch


def test_host_side_rejections(libs):
    L = _setup(libs["libmxq.so"])
    # fp16 is rejected (TE PR #3264: "fp16 is rejected")
    assert L.mxq_fake_quant_mxfp4(FAKE, FAKE, 2, 4, 32, 32, 32, None) == UNSUPPORTED
    assert L.mxq_mxfp8_row_direct(FAKE, 2, 4, 32, 32, FAKE, FAKE, 0, None) == UNSUPPORTED
    assert L.mxq_fp8_block128_direct(FAKE, 2, 4, 32, 32, FAKE, FAKE, None) == UNSUPPORTED
    assert L.mxq_fake_quant_mxfp4(FAKE, FAKE, 7, 4, 32, 32, 32, None) == INVALID
    # shapes and pointers
    assert L.mxq_fake_quant_mxfp4(FAKE, FAKE, 0, -1, 32, 32, 32, None) == INVALID
    assert L.mxq_fake_quant_mxfp4(FAKE, FAKE, 0, 4, 32, 16, 32, None) == INVALID  # ld < K
    assert L.mxq_fake_quant_mxfp4(None, FAKE, 0, 4, 32, 32, 32, None) == INVALID
    assert L.mxq_fake_quant_mxfp4(FAKE + 1, FAKE, 0, 4, 32, 32, 32, None) == INVALID  # bf16 at odd address
    assert L.mxq_fake_quant_mxfp4(FAKE, FAKE, 0, 4, 32, 32, 64, None) == INVALID  # in place needs equal ld
    assert L.mxq_mxfp8_row_direct(FAKE, 0, 4, 32, 32, FAKE, FAKE, 3, None) == INVALID  # layout
    assert L.mxq_mxfp8_row_direct(FAKE, 0, 4, 32, 32, None, FAKE, 0, None) == INVALID
    assert L.mxq_fp8_block128_direct(FAKE, 1, 4, 32, 32, FAKE, FAKE + 2, None) == INVALID
    # empty tensors are a no-op (TE PR #3790 tests: empty tensor)
    assert L.mxq_fake_quant_mxfp4(None, None, 0, 0, 32, 32, 32, None) == OK
    assert L.mxq_mxfp8_row_direct(None, 1, 5, 0, 0, None, None, 2, None) == OK
    assert L.mxq_fp8_block128_direct(None, 0, 0, 0, 0, None, None, None) == OK
    q = _Q(kind=0, data=FAKE, rows=4, K=32, fp8=0, scales=FAKE, lay=0, tile_scale_inv=None)
    assert L.mxq_dequantize(ctypes.byref(q), FAKE, 2, None) == UNSUPPORTED
    q.kind = 1
    q.fp8 = 1
    assert L.mxq_dequantize(ctypes.byref(q), FAKE, 0, None) == INVALID  # blockwise is E4M3 only
    assert L.mxq_dequantize(None, FAKE, 0, None) == INVALID
    # skip flags must be int32-aligned device pointers; packed MXFP4 validates like MXFP8
    L.mxq_mxfp8_row_direct_update.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_void_p]
    assert L.mxq_mxfp8_row_direct_update(FAKE, 0, 4, 32, 32, FAKE, FAKE, 0, FAKE + 2, None) == INVALID
    assert L.mxq_mxfp8_row_direct_update(FAKE, 2, 4, 32, 32, FAKE, FAKE, 0, FAKE, None) == UNSUPPORTED
    L.mxq_mxfp4_pack.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert L.mxq_mxfp4_pack(FAKE, 2, 4, 32, 32, FAKE, FAKE, 0, None) == UNSUPPORTED
    assert L.mxq_mxfp4_pack(FAKE, 0, 4, 32, 32, FAKE, FAKE, 7, None) == INVALID
    assert L.mxq_mxfp4_pack(None, 0, 0, 32, 32, None, None, 0, None) == OK
    q = _Q(kind=2, data=FAKE, rows=4, K=32, fp8=9, scales=None, lay=0, tile_scale_inv=None)
    assert L.mxq_dequantize(ctypes.byref(q), FAKE, 0, None) == INVALID  # MXFP4 needs scales


def test_export_host_logic(libs):
    L = _setup(libs["libmxq.so"])
    c = _C()
    # no row-scaled data -> the ValueError analogue (TE PR #3790)
    st = _S(data=None, scales=FAKE, fp8=0, lay=0, rows=100, K=48)
    assert L.mxq_export_mxfp8(ctypes.byref(st), None, 0, ctypes.byref(c), None) == NO_ROWWISE
    # compact -> view, no launch
    st = _S(data=FAKE, scales=FAKE + 4096, fp8=1, lay=0, rows=100, K=48)
    assert L.mxq_export_mxfp8(ctypes.byref(st), None, 0, ctypes.byref(c), None) == OK
    assert c.is_view == 1 and c.scales == FAKE + 4096 and c.data == FAKE and c.scale_cols == 2 and c.fp8 == 1
    # padded with ceil(K/32) % 4 == 0 -> view of the prefix
    st = _S(data=FAKE, scales=FAKE + 4096, fp8=0, lay=1, rows=100, K=128)
    assert L.mxq_export_mxfp8(ctypes.byref(st), None, 0, ctypes.byref(c), None) == OK
    assert c.is_view == 1 and c.scale_cols == 4
    # padded with nb = 2, or swizzled -> copy needed, buffer checked first
    for lay in (1, 2):
        st = _S(data=FAKE, scales=FAKE + 4096, fp8=0, lay=lay, rows=100, K=48)
        assert L.mxq_export_mxfp8(ctypes.byref(st), None, 0, ctypes.byref(c), None) == TOO_SMALL
        assert L.mxq_export_mxfp8(ctypes.byref(st), FAKE, 199, ctypes.byref(c), None) == TOO_SMALL
    # grouped: every storage is checked before anything launches
    L.mxq_export_mxfp8_grouped.argtypes = [ctypes.POINTER(_S), ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.POINTER(_C), ctypes.c_void_p]
    arr = (_S * 3)(_S(data=FAKE, scales=FAKE, fp8=0, lay=0, rows=4, K=32),
                   _S(data=FAKE, scales=FAKE, fp8=0, lay=2, rows=100, K=48),
                   _S(data=None, scales=FAKE, fp8=0, lay=0, rows=4, K=32))
    comps = (_C * 3)()
    assert L.mxq_export_mxfp8_grouped(arr, 3, FAKE, 1 << 20, comps, None) == NO_ROWWISE
    assert L.mxq_export_mxfp8_grouped(arr, 2, FAKE, 199, comps, None) == TOO_SMALL
    assert L.mxq_export_mxfp8_grouped(arr, 1, None, 0, comps, None) == OK  # a view: nothing to copy
    assert comps[0].is_view == 1 and comps[0].scales == FAKE
    assert L.mxq_export_mxfp8_grouped(arr, 0, None, 0, comps, None) == OK
    assert L.mxq_export_mxfp8_grouped(arr, -1, None, 0, comps, None) == INVALID
    # empty storage exports as an empty view even without data
    st = _S(data=None, scales=None, fp8=0, lay=2, rows=0, K=48)
    assert L.mxq_export_mxfp8(ctypes.byref(st), None, 0, ctypes.byref(c), None) == OK
    assert c.is_view == 1
