"""CPU oracle for block-scaled weight conversion (MXFP4 projection, direct
MXFP8 rowwise, direct FP8 128x128 blockwise, dequantize, export).

TEST INFRASTRUCTURE ONLY.  The product library never imports, links or runs
anything here: only ``tests/``, the package smoke check in
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may.  The arithmetic lives in ``mxq_oracle.c`` (plain
C, exact doubles decoded from the IEEE fields); this module only builds it
with gcc and marshals numpy arrays through ctypes.

Every function cites the passage it follows in ``mxq_oracle.c``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmxq_oracle.so")

BF16, FP32 = 0, 1
E4M3, E5M2 = 0, 1
COMPACT, PADDED, SWIZZLED = 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE doubles are required)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            # MXQ_ORACLE_LIB: load another build of the oracle source instead
            # (the mutation tests point it at copies with planted mistakes)
            lib = ctypes.CDLL(os.environ.get("MXQ_ORACLE_LIB") or build())
            i64, ip, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_fake_quant_mxfp4.argtypes = [vp, vp, ip, i64, i64, i64, i64]
            lib.oracle_mxfp8_row_direct.argtypes = [vp, ip, i64, i64, i64, vp, vp]
            lib.oracle_fp8_block128_direct.argtypes = [vp, ip, i64, i64, i64, vp, vp]
            lib.oracle_dequant_mxfp8.argtypes = [vp, vp, ip, ip, i64, i64, vp, ip]
            lib.oracle_dequant_block128.argtypes = [vp, vp, i64, i64, vp, ip]
            lib.oracle_export_scales.argtypes = [vp, ip, i64, i64, vp]
            lib.oracle_scales_to_layout.argtypes = [vp, i64, i64, ip, vp]
            lib.oracle_scale_bytes.argtypes = [i64, i64, ip]
            lib.oracle_scale_bytes.restype = i64
            lib.oracle_scale_offset.argtypes = [i64, i64, i64, ip]
            lib.oracle_scale_offset.restype = i64
            lib.oracle_block_exponent.argtypes = [ctypes.c_uint32, ip]
            lib.oracle_block_exponent.restype = ip
            lib.oracle_e2m1_rtne_code.argtypes = [ctypes.c_double]
            lib.oracle_e2m1_rtne_code.restype = ip
            lib.oracle_fp8_value.argtypes = [ctypes.c_uint8, ip]
            lib.oracle_fp8_value.restype = ctypes.c_double
            lib.oracle_e4m3_rtne.argtypes = [ctypes.c_double]
            lib.oracle_e4m3_rtne.restype = ctypes.c_uint8
            lib.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_value.restype = ctypes.c_double
            lib.oracle_mxfp4_pack.argtypes = [vp, ip, i64, i64, i64, vp, vp]
            lib.oracle_mxfp8_col_direct.argtypes = [vp, ip, i64, i64, i64, vp, vp]
            lib.oracle_mxfp8_host_exponent.argtypes = [ctypes.c_double]
            lib.oracle_mxfp8_host_exponent.restype = ip
            lib.oracle_dequant_mxfp4.argtypes = [vp, vp, ip, i64, i64, vp, ip]
            lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_value.restype = ctypes.c_double
            lib.oracle_f32_to_bf16.argtypes = [ctypes.c_uint32]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            _lib = lib
    return _lib


def _dt_of(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return BF16
    if x.dtype in (np.uint32, np.float32):
        return FP32
    raise TypeError("oracle inputs are bf16 bit patterns (uint16) or fp32 (float32/uint32)")


def _rows_k_ld(x: np.ndarray):
    if x.ndim < 1:
        raise ValueError("need at least one dimension")
    K = x.shape[-1]
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    if x.ndim == 1:
        return rows, K, K
    x2 = x.reshape(rows, K) if x.ndim > 2 else x
    if x2.strides[-1] != x.itemsize:
        raise ValueError("last dimension must be contiguous")
    return rows, K, x2.strides[0] // x.itemsize


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def scale_cols(K: int) -> int:
    return (K + 31) // 32


def scale_bytes(rows: int, K: int, lay: int) -> int:
    return int(_L().oracle_scale_bytes(rows, K, lay))


def scale_offset(r: int, j: int, nb: int, lay: int) -> int:
    return int(_L().oracle_scale_offset(r, j, nb, lay))


def fake_quant_mxfp4(x: np.ndarray) -> np.ndarray:
    """MXFP4 projection of bf16 (uint16 patterns) or fp32 ``x``; same shape and dtype."""
    dt = _dt_of(x)
    rows, K, ldx = _rows_k_ld(x)
    y = np.empty(x.shape, dtype=x.dtype)
    if x.size:
        _L().oracle_fake_quant_mxfp4(_ptr(x), _ptr(y), dt, rows, K, ldx, K)
    return y


def mxfp8_row_direct(x: np.ndarray, lay: int = COMPACT):
    """Direct MXFP8 rowwise: (E4M3 payload bytes [*shape], scales in ``lay``)."""
    dt = _dt_of(x)
    rows, K, ldx = _rows_k_ld(x)
    data = np.empty(x.shape, dtype=np.uint8)
    nb = scale_cols(K)
    compact = np.empty((rows, nb), dtype=np.uint8)
    if x.size:
        _L().oracle_mxfp8_row_direct(_ptr(x), dt, rows, K, ldx, _ptr(data), _ptr(compact))
    if lay == COMPACT:
        return data, compact.reshape(tuple(x.shape[:-1]) + (nb,))
    out = np.empty(scale_bytes(rows, K, lay), dtype=np.uint8)
    _L().oracle_scales_to_layout(_ptr(compact), rows, K, lay, _ptr(out))
    return data, out


def scales_to_layout(compact: np.ndarray, rows: int, K: int, lay: int) -> np.ndarray:
    compact = np.ascontiguousarray(compact, dtype=np.uint8)
    out = np.empty(scale_bytes(rows, K, lay), dtype=np.uint8)
    _L().oracle_scales_to_layout(_ptr(compact), rows, K, lay, _ptr(out))
    return out


def fp8_block128_direct(x: np.ndarray):
    """Direct FP8 128x128 blockwise: (E4M3 bytes [rows, K], fp32 2^T [ceil(rows/128), ceil(K/128)])."""
    dt = _dt_of(x)
    rows, K, ldx = _rows_k_ld(x)
    data = np.empty(x.shape, dtype=np.uint8)
    sinv = np.empty(((rows + 127) // 128, (K + 127) // 128), dtype=np.float32)
    if x.size:
        _L().oracle_fp8_block128_direct(_ptr(x), dt, rows, K, ldx, _ptr(data), _ptr(sinv))
    return data, sinv


def dequant_mxfp8(data: np.ndarray, scales: np.ndarray, lay: int, kind: int, out_dt: int) -> np.ndarray:
    """payload * 2^(code-127) as fp32 (float32) or bf16 (uint16 patterns)."""
    data = np.ascontiguousarray(data, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    K = data.shape[-1]
    rows = data.size // K if K else 0
    out = np.empty(data.shape, dtype=np.float32 if out_dt == FP32 else np.uint16)
    if data.size:
        _L().oracle_dequant_mxfp8(_ptr(data), _ptr(scales), lay, kind, rows, K, _ptr(out), out_dt)
    return out


def dequant_block128(data: np.ndarray, tile_scale_inv: np.ndarray, out_dt: int) -> np.ndarray:
    data = np.ascontiguousarray(data, dtype=np.uint8)
    sinv = np.ascontiguousarray(tile_scale_inv, dtype=np.float32)
    K = data.shape[-1]
    rows = data.size // K if K else 0
    out = np.empty(data.shape, dtype=np.float32 if out_dt == FP32 else np.uint16)
    if data.size:
        _L().oracle_dequant_block128(_ptr(data), _ptr(sinv), rows, K, _ptr(out), out_dt)
    return out


def mxfp4_pack(x: np.ndarray, lay: int = COMPACT):
    """Packed MXFP4: (nibbles uint8 [rows, ceil(K/2)], scales in ``lay``)."""
    dt = _dt_of(x)
    rows, K, ldx = _rows_k_ld(x)
    packed = np.zeros((rows, (K + 1) // 2), dtype=np.uint8)
    nb = scale_cols(K)
    compact = np.empty((rows, nb), dtype=np.uint8)
    if x.size:
        _L().oracle_mxfp4_pack(_ptr(x), dt, rows, K, ldx, _ptr(packed), _ptr(compact))
    if lay == COMPACT:
        return packed, compact
    return packed, scales_to_layout(compact, rows, K, lay)


def mxfp8_col_direct(x: np.ndarray, lay: int = COMPACT):
    """Direct MXFP8 columnwise: (E4M3 bytes [rows, K], scales of the K x
    ceil(rows/32) transposed scale matrix in ``lay``)."""
    dt = _dt_of(x)
    rows, K, ldx = _rows_k_ld(x)
    data = np.empty((rows, K), dtype=np.uint8)
    nbr = (rows + 31) // 32
    compact = np.empty((K, nbr), dtype=np.uint8)
    if x.size:
        _L().oracle_mxfp8_col_direct(_ptr(x), dt, rows, K, ldx, _ptr(data), _ptr(compact))
    if lay == COMPACT:
        return data, compact
    return data, scales_to_layout(compact, K, rows, lay)


def mxfp8_host_exponent(amax: float) -> int:
    return int(_L().oracle_mxfp8_host_exponent(amax))


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray, lay: int, K: int, out_dt: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows = packed.shape[0] if packed.ndim > 1 else 1
    out = np.empty((rows, K), dtype=np.float32 if out_dt == FP32 else np.uint16)
    if rows and K:
        _L().oracle_dequant_mxfp4(_ptr(packed), _ptr(scales), lay, rows, K, _ptr(out), out_dt)
    return out


def e2m1_value(nibble: int) -> float:
    return float(_L().oracle_e2m1_value(nibble))


def export_scales(scales: np.ndarray, lay: int, rows: int, K: int) -> np.ndarray:
    """Compact (rows, ceil(K/32)) uint8 scales from a layout."""
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty((rows, scale_cols(K)), dtype=np.uint8)
    if rows and K:
        _L().oracle_export_scales(_ptr(scales), lay, rows, K, _ptr(out))
    return out


def block_exponent(amax_mag_bits: int, dt: int) -> int:
    return int(_L().oracle_block_exponent(amax_mag_bits, dt))


def e2m1_rtne_code(v: float) -> int:
    return int(_L().oracle_e2m1_rtne_code(v))


def fp8_value(b: int, kind: int) -> float:
    return float(_L().oracle_fp8_value(b, kind))


def e4m3_rtne(u: float) -> int:
    return int(_L().oracle_e4m3_rtne(u))


def e8m0_value(c: int) -> float:
    return float(_L().oracle_e8m0_value(c))


def f32_to_bf16(bits: int) -> int:
    return int(_L().oracle_f32_to_bf16(bits))
