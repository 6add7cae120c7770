"""Block-scaled weight conversion on GB300: Python binding of libmxq.

Argument marshalling only.  Every conversion runs in the CUDA kernels of
``libmxq.so`` (built from ``csrc/`` by ``build.py``) through its C ABI
(``include/mxq.h``); PyTorch supplies device memory and the current stream.
There is no CPU path: if the library is missing the call raises.

Functions carry the C names:

* ``mxq_fake_quant_mxfp4``     MXFP4 projection (TE PR #3264, mode 1)
* ``mxq_mxfp8_row_direct``     direct MXFP8 rowwise (TE PR #3264, mode 2)
* ``mxq_fp8_block128_direct``  direct FP8 128x128 blockwise (TE PR #3264, mode 2)
* ``mxq_mxfp4_pack``           packed MXFP4 deployment form (TE PR #3264)
* ``mxq_mxfp8_col_direct``     direct MXFP8 columnwise, 32x1 blocks (TE PR #3264, mode 2)
* ``mxq_dequantize``           MXFP8 rowwise / 128x128 blockwise / packed MXFP4 -> bf16 / fp32
* ``mxq_export_mxfp8``         export_components (TE PR #3790)
* ``mxq_export_mxfp8_grouped`` export of many storages (per expert) in one launch
* ``mxq_quantize_export_mxfp8`` quantize a bf16/fp32 weight and export it in one call

The ``skip=`` argument of the converters selects the ``*_update`` entry
points: a device int32 tensor, read when the kernel runs; nonzero means the
call writes nothing (for cached weights inside captured CUDA graphs).
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import NamedTuple, Optional

import torch

from . import build as _build

__all__ = [
    "MXQError", "MXFP8Components", "Library", "Call", "library",
    "mxq_fake_quant_mxfp4", "mxq_mxfp8_row_direct", "mxq_fp8_block128_direct",
    "mxq_dequantize", "mxq_export_mxfp8", "mxq_mxfp4_pack", "mxq_mxfp8_col_direct", "mxq_scale_bytes",
    "mxq_tile_scale_count", "mxq_export_mxfp8_grouped", "mxq_quantize_export_mxfp8",
    "COMPACT", "PADDED", "SWIZZLED", "scale_cols",
]

COMPACT, PADDED, SWIZZLED = 0, 1, 2
_LAYOUTS = {"compact": COMPACT, "padded": PADDED, "swizzled": SWIZZLED, COMPACT: COMPACT, PADDED: PADDED,
            SWIZZLED: SWIZZLED}
_BF16, _FP32, _FP16 = 0, 1, 2
_E4M3, _E5M2 = 0, 1
_MXFP8_ROW, _BLOCK128, _MXFP4, _MXFP8_COL = 0, 1, 2, 3


class MXQError(RuntimeError):
    def __init__(self, status: int, msg: str, where: str):
        super().__init__(f"{where}: {msg} (mxq status {status})")
        self.status = status


class MXFP8Components(NamedTuple):
    """Exported MXFP8 values and compact E8M0 scales (TE PR #3790)."""
    data: torch.Tensor       # float8_e4m3fn / float8_e5m2 view of the payload
    scale_inv: torch.Tensor  # uint8 (*shape[:-1], ceil(K/32))
    is_view: bool            # True if scale_inv aliases the storage's scales


class _Quantized(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("data", ctypes.c_void_p), ("rows", ctypes.c_int64), ("K", ctypes.c_int64),
                ("fp8", ctypes.c_int), ("scales", ctypes.c_void_p), ("lay", ctypes.c_int),
                ("tile_scale_inv", ctypes.c_void_p)]


class _Storage(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("fp8", ctypes.c_int), ("lay", ctypes.c_int),
                ("rows", ctypes.c_int64), ("K", ctypes.c_int64)]


class _Components(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("fp8", ctypes.c_int), ("scales", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("K", ctypes.c_int64), ("scale_cols", ctypes.c_int64),
                ("is_view", ctypes.c_int)]


def scale_cols(K: int) -> int:
    return (K + 31) // 32


def _dt_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _BF16
    if t.dtype == torch.float32:
        return _FP32
    if t.dtype == torch.float16:
        return _FP16
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32 expected")


def _fp8_code(fp8) -> int:
    if fp8 in ("e4m3", torch.float8_e4m3fn, _E4M3):
        return _E4M3
    if fp8 in ("e5m2", torch.float8_e5m2, _E5M2):
        return _E5M2
    raise ValueError(f"unknown fp8 kind {fp8!r}")


def _rows_view(x: torch.Tensor):
    """(rows, K, ld) of x seen as rows of its last dimension, without a copy."""
    if x.dim() == 0:
        raise ValueError("need at least one dimension")
    K = x.shape[-1]
    if x.dim() == 1:
        if K > 1 and x.stride(0) != 1:
            raise ValueError("last dimension must be contiguous")
        return 1, K, K
    if x.numel() == 0:
        rows = 1
        for d in x.shape[:-1]:
            rows *= d
        return rows, K, K
    if K > 1 and x.stride(-1) != 1:
        raise ValueError("last dimension must be contiguous")
    try:
        v = x.view(-1, K)
    except RuntimeError as exc:
        raise ValueError("leading dimensions must flatten to one row stride (no copy is made)") from exc
    ld = v.stride(0) if v.shape[0] > 1 else K
    return v.shape[0], K, max(ld, K)


def _stream(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _skip_ptr(skip: torch.Tensor) -> ctypes.c_void_p:
    if skip.dtype != torch.int32 or skip.numel() < 1:
        raise ValueError("skip must be a device int32 tensor (nonzero = write nothing)")
    return ctypes.c_void_p(skip.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libmxq works on CUDA tensors only")


def _check_bytes(t: torch.Tensor, need: int, name: str, what: str):
    """The C ABI sees only a pointer: a buffer shorter than the layout would
    be read (or written) past its end, so the binding checks it here."""
    if t.dtype != torch.uint8 or not t.is_contiguous() or t.numel() < need:
        raise ValueError(f"{name} must be a contiguous uint8 buffer of at least {what} = {need} bytes")


def _check_storage(lib, data, scales, rows: int, K: int, layout):
    """Sizes of an MXFP8 storage handed to an export: rows*K payload bytes
    and the scale bytes of its layout."""
    _check_bytes(scales, lib.scale_bytes(rows, K, _LAYOUTS[layout]), "scales", "mxq_scale_bytes(rows, K, layout)")
    if data is not None and (not data.is_contiguous() or data.numel() != rows * K or data.element_size() != 1):
        raise ValueError("data must be the contiguous rows*K payload bytes of the storage")


class Library:
    """One loaded libmxq variant (``fastmath=True`` loads the --use_fast_math build)."""

    def __init__(self, fastmath: bool = False, build: bool = True):
        name = "libmxq_fastmath.so" if fastmath else "libmxq.so"
        path = _build.lib_path(name)
        if build:
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with python -m block_scaled_precision_x32_gb300.build")
        self.path = path
        L = ctypes.CDLL(path)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        L.mxq_fake_quant_mxfp4.argtypes = [vp, vp, ci, i64, i64, i64, i64, vp]
        L.mxq_mxfp8_row_direct.argtypes = [vp, ci, i64, i64, i64, vp, vp, ci, vp]
        L.mxq_fp8_block128_direct.argtypes = [vp, ci, i64, i64, i64, vp, vp, vp]
        L.mxq_fake_quant_mxfp4_update.argtypes = [vp, vp, ci, i64, i64, i64, i64, vp, vp]
        L.mxq_mxfp8_row_direct_update.argtypes = [vp, ci, i64, i64, i64, vp, vp, ci, vp, vp]
        L.mxq_fp8_block128_direct_update.argtypes = [vp, ci, i64, i64, i64, vp, vp, vp, vp]
        L.mxq_mxfp4_pack.argtypes = [vp, ci, i64, i64, i64, vp, vp, ci, vp]
        L.mxq_mxfp8_col_direct.argtypes = [vp, ci, i64, i64, i64, vp, vp, ci, vp]
        L.mxq_mxfp4_pack_update.argtypes = [vp, ci, i64, i64, i64, vp, vp, ci, vp, vp]
        L.mxq_mxfp8_col_direct_update.argtypes = [vp, ci, i64, i64, i64, vp, vp, ci, vp, vp]
        L.mxq_export_mxfp8_grouped.argtypes = [ctypes.POINTER(_Storage), i64, vp, ctypes.c_size_t,
                                               ctypes.POINTER(_Components), vp]
        L.mxq_quantize_export_mxfp8.argtypes = [vp, ci, i64, i64, i64, vp, vp, ctypes.POINTER(_Components), vp]
        L.mxq_dequantize.argtypes = [ctypes.POINTER(_Quantized), vp, ci, vp]
        L.mxq_export_mxfp8.argtypes = [ctypes.POINTER(_Storage), vp, ctypes.c_size_t, ctypes.POINTER(_Components), vp]
        L.mxq_scale_bytes.argtypes = [i64, i64, ci]
        L.mxq_scale_bytes.restype = ctypes.c_size_t
        L.mxq_tile_scale_count.argtypes = [i64, i64]
        L.mxq_tile_scale_count.restype = ctypes.c_size_t
        L.mxq_status_string.argtypes = [ci]
        L.mxq_status_string.restype = ctypes.c_char_p
        for fn in ("mxq_fake_quant_mxfp4", "mxq_mxfp8_row_direct", "mxq_fp8_block128_direct", "mxq_dequantize",
                   "mxq_export_mxfp8", "mxq_fake_quant_mxfp4_update", "mxq_mxfp8_row_direct_update",
                   "mxq_fp8_block128_direct_update", "mxq_mxfp4_pack", "mxq_mxfp8_col_direct",
                   "mxq_mxfp4_pack_update", "mxq_mxfp8_col_direct_update", "mxq_export_mxfp8_grouped",
                   "mxq_quantize_export_mxfp8"):
            getattr(L, fn).restype = ci
        self.L = L

    def _check(self, status: int, where: str):
        if status != 0:
            raise MXQError(status, self.L.mxq_status_string(status).decode(), where)

    # -- sizes ----------------------------------------------------------
    def scale_bytes(self, rows: int, K: int, layout="compact") -> int:
        return int(self.L.mxq_scale_bytes(rows, K, _LAYOUTS[layout]))

    def tile_scale_count(self, rows: int, K: int) -> int:
        return int(self.L.mxq_tile_scale_count(rows, K))

    # -- prepared calls -------------------------------------------------
    # Each plan_* validates and marshals its arguments once and returns a
    # Call: invoking it enqueues the one kernel on the stream that was
    # current when the plan was made.  The Call keeps its tensors alive.
    # The eager methods below are plan_*(...)() with freshly allocated
    # outputs.

    def plan_fake_quant_mxfp4(self, x: torch.Tensor, out: torch.Tensor, skip: Optional[torch.Tensor] = None) -> "Call":
        _need_cuda(x, out, skip)
        dt = _dt_code(x)
        rows, K, ldx = _rows_view(x)
        if out.shape != x.shape or out.dtype != x.dtype:
            raise ValueError("out must match x in shape and dtype")
        _, _, ldy = _rows_view(out)
        args = (ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(out.data_ptr()), dt, rows, K, ldx, ldy)
        if skip is not None:
            args += (_skip_ptr(skip), _stream(x))
            return Call(self, self.L.mxq_fake_quant_mxfp4_update, args, "mxq_fake_quant_mxfp4_update", (x, out, skip),
                        x.device)
        return Call(self, self.L.mxq_fake_quant_mxfp4, args + (_stream(x),), "mxq_fake_quant_mxfp4", (x, out), x.device)

    def _plan_rowwise_quant(self, name, x, layout, data, scales, data_bytes, skip):
        _need_cuda(x, data, scales, skip)
        dt = _dt_code(x)
        lay = _LAYOUTS[layout]
        rows, K, ldx = _rows_view(x)
        if not data.is_contiguous() or data.numel() != data_bytes(rows, K) or data.dtype != torch.uint8:
            raise ValueError("data must be a contiguous uint8 tensor of the payload size")
        if not scales.is_contiguous() or scales.dtype != torch.uint8 or scales.numel() < self.scale_bytes(rows, K, lay):
            raise ValueError("scales must be a contiguous uint8 buffer of mxq_scale_bytes() bytes")
        args = (ctypes.c_void_p(x.data_ptr()), dt, rows, K, ldx, ctypes.c_void_p(data.data_ptr()),
                ctypes.c_void_p(scales.data_ptr()), lay)
        if skip is not None:
            name += "_update"
            args += (_skip_ptr(skip),)
        return Call(self, getattr(self.L, name), args + (_stream(x),), name, (x, data, scales, skip), x.device)

    def plan_mxfp8_row_direct(self, x: torch.Tensor, layout, data: torch.Tensor, scales: torch.Tensor,
                              skip: Optional[torch.Tensor] = None) -> "Call":
        return self._plan_rowwise_quant("mxq_mxfp8_row_direct", x, layout, data, scales, lambda r, k: r * k, skip)

    def plan_mxfp4_pack(self, x: torch.Tensor, layout, packed: torch.Tensor, scales: torch.Tensor,
                        skip: Optional[torch.Tensor] = None) -> "Call":
        return self._plan_rowwise_quant("mxq_mxfp4_pack", x, layout, packed, scales, lambda r, k: r * ((k + 1) // 2),
                                        skip)

    def plan_mxfp8_col_direct(self, x: torch.Tensor, layout, data: torch.Tensor, scales: torch.Tensor,
                              skip: Optional[torch.Tensor] = None) -> "Call":
        """Columnwise MXFP8: data [rows, K]; scales hold the K x ceil(rows/32)
        scale matrix of the transposed tensor in ``layout``."""
        _need_cuda(x, data, scales, skip)
        dt = _dt_code(x)
        lay = _LAYOUTS[layout]
        rows, K, ldx = _rows_view(x)
        if not data.is_contiguous() or data.numel() != rows * K or data.dtype != torch.uint8:
            raise ValueError("data must be a contiguous uint8 tensor of rows*K bytes")
        if not scales.is_contiguous() or scales.dtype != torch.uint8 or scales.numel() < self.scale_bytes(K, rows, lay):
            raise ValueError("scales must be a contiguous uint8 buffer of mxq_scale_bytes(K, rows) bytes")
        args = (ctypes.c_void_p(x.data_ptr()), dt, rows, K, ldx, ctypes.c_void_p(data.data_ptr()),
                ctypes.c_void_p(scales.data_ptr()), lay)
        if skip is not None:
            return Call(self, self.L.mxq_mxfp8_col_direct_update, args + (_skip_ptr(skip), _stream(x)),
                        "mxq_mxfp8_col_direct_update", (x, data, scales, skip), x.device)
        return Call(self, self.L.mxq_mxfp8_col_direct, args + (_stream(x),), "mxq_mxfp8_col_direct",
                    (x, data, scales), x.device)

    def plan_fp8_block128_direct(self, x: torch.Tensor, data: torch.Tensor, tile_scale_inv: torch.Tensor,
                                 skip: Optional[torch.Tensor] = None) -> "Call":
        _need_cuda(x, data, tile_scale_inv, skip)
        dt = _dt_code(x)
        rows, K, ldx = _rows_view(x)
        if not data.is_contiguous() or data.numel() != rows * K or data.dtype != torch.uint8:
            raise ValueError("data must be a contiguous uint8 tensor of rows*K bytes")
        if tile_scale_inv.dtype != torch.float32 or tile_scale_inv.numel() < self.tile_scale_count(rows, K):
            raise ValueError("tile_scale_inv must be fp32 with ceil(rows/128)*ceil(K/128) entries")
        args = (ctypes.c_void_p(x.data_ptr()), dt, rows, K, ldx, ctypes.c_void_p(data.data_ptr()),
                ctypes.c_void_p(tile_scale_inv.data_ptr()))
        if skip is not None:
            return Call(self, self.L.mxq_fp8_block128_direct_update, args + (_skip_ptr(skip), _stream(x)),
                        "mxq_fp8_block128_direct_update", (x, data, tile_scale_inv, skip), x.device)
        return Call(self, self.L.mxq_fp8_block128_direct, args + (_stream(x),), "mxq_fp8_block128_direct",
                    (x, data, tile_scale_inv), x.device)

    def plan_dequantize(self, data: torch.Tensor, out: torch.Tensor, *, scales: Optional[torch.Tensor] = None,
                        layout="compact", fp8="e4m3", tile_scale_inv: Optional[torch.Tensor] = None,
                        mxfp4: bool = False, columnwise: bool = False) -> "Call":
        """MXFP8 rowwise (``scales``), 128x128 (``tile_scale_inv``) or packed
        MXFP4 (``mxfp4=True`` with ``scales``; ``data`` holds ceil(K/2) bytes
        per row and K is taken from ``out``)."""
        _need_cuda(data, scales, tile_scale_inv, out)
        if (scales is None) == (tile_scale_inv is None) or (mxfp4 and scales is None):
            raise ValueError("pass exactly one of scales (MXFP8 rowwise, MXFP4) or tile_scale_inv (128x128)")
        if not data.is_contiguous():
            raise ValueError("data must be contiguous")
        if not out.is_contiguous():
            raise ValueError("out must be contiguous")
        if mxfp4:
            K = out.shape[-1] if out.dim() else 1
            rows = out.numel() // K if K else 0
            if data.numel() != rows * ((K + 1) // 2):
                raise ValueError("packed data must hold ceil(K/2) bytes per row of out")
        else:
            if out.shape != data.shape:
                raise ValueError("out must have data's shape")
            K = data.shape[-1] if data.dim() else 1
            rows = data.numel() // K if K else 0
        if data.dtype not in (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2):
            raise ValueError("data must hold payload bytes (uint8 or an fp8 view)")
        lay = _LAYOUTS[layout]
        if scales is not None:
            # the kernels read every scale of the layout: a short buffer would be read past its end
            need = self.scale_bytes(K, rows, lay) if columnwise else self.scale_bytes(rows, K, lay)
            _check_bytes(scales, need, "scales", "mxq_scale_bytes(K, rows, layout)" if columnwise
                         else "mxq_scale_bytes(rows, K, layout)")
        else:
            if (not tile_scale_inv.is_contiguous() or tile_scale_inv.dtype != torch.float32
                    or tile_scale_inv.numel() < self.tile_scale_count(rows, K)):
                raise ValueError("tile_scale_inv must be a contiguous fp32 tensor of "
                                 "ceil(rows/128)*ceil(K/128) values")
        q = _Quantized()
        q.kind = _MXFP4 if mxfp4 else (_MXFP8_COL if columnwise else (_MXFP8_ROW if scales is not None else _BLOCK128))
        q.data = data.data_ptr()
        q.rows, q.K = rows, K
        q.fp8 = _fp8_code(fp8)
        q.lay = lay
        q.scales = scales.data_ptr() if scales is not None else None
        q.tile_scale_inv = tile_scale_inv.data_ptr() if tile_scale_inv is not None else None
        odt = _FP16 if out.dtype == torch.float16 else _dt_code(out)
        args = (ctypes.byref(q), ctypes.c_void_p(out.data_ptr()), odt, _stream(data))
        return Call(self, self.L.mxq_dequantize, args, "mxq_dequantize", (data, out, scales, tile_scale_inv, q),
                    data.device)

    def plan_export_mxfp8(self, data: Optional[torch.Tensor], scales: torch.Tensor, *, shape, layout="compact",
                          fp8="e4m3", scale_out: Optional[torch.Tensor] = None):
        """Returns (Call, MXFP8Components).  The components are views whose
        scale bytes are valid once the Call has run (a view of the storage
        needs no kernel; the Call then launches nothing)."""
        shape = tuple(shape)
        K = shape[-1] if shape else 0
        rows = 1
        for d in shape[:-1]:
            rows *= d
        nb = scale_cols(K)
        _need_cuda(scales, data, scale_out)
        _check_storage(self, data, scales, rows, K, layout)
        if scale_out is not None and (scale_out.dtype != torch.uint8 or not scale_out.is_contiguous()):
            raise ValueError("scale_out must be a contiguous uint8 tensor")
        st = _Storage()
        st.data = data.data_ptr() if data is not None else None
        st.scales = scales.data_ptr()
        st.fp8 = _fp8_code(fp8)
        st.lay = _LAYOUTS[layout]
        st.rows, st.K = rows, K
        view = st.lay == COMPACT or (st.lay == PADDED and nb % 4 == 0) or rows * K == 0
        if scale_out is None and not view:
            scale_out = torch.empty(rows * nb, dtype=torch.uint8, device=scales.device)
        comp = _Components()
        args = (ctypes.byref(st), ctypes.c_void_p(scale_out.data_ptr()) if scale_out is not None else None,
                scale_out.numel() if scale_out is not None else 0, ctypes.byref(comp), _stream(scales))
        call = Call(self, self.L.mxq_export_mxfp8, args, "mxq_export_mxfp8", (data, scales, scale_out, st, comp),
                    scales.device)
        fp8_dtype = torch.float8_e4m3fn if st.fp8 == _E4M3 else torch.float8_e5m2
        values = data.view(fp8_dtype).view(shape) if data is not None else None
        src = scales if view else scale_out
        s = src.reshape(-1)[: rows * nb].view(shape[:-1] + (nb,))
        return call, MXFP8Components(values, s, view)

    # -- eager conversions ----------------------------------------------

    def fake_quant_mxfp4(self, x: torch.Tensor, out: Optional[torch.Tensor] = None,
                         skip: Optional[torch.Tensor] = None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(x, memory_format=torch.contiguous_format)
        self.plan_fake_quant_mxfp4(x, out, skip)()
        return out

    def mxfp8_row_direct(self, x: torch.Tensor, layout="compact", data: Optional[torch.Tensor] = None,
                         scales: Optional[torch.Tensor] = None, skip: Optional[torch.Tensor] = None):
        """Returns (payload uint8 of x's shape, scales).  Compact scales are
        shaped (*shape[:-1], nb); padded and swizzled ones (Rp, Cp)."""
        rows, K, _ = _rows_view(x)
        if data is None:
            data = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        if scales is None:
            scales = self._scale_buffer(x, rows, K, layout)
        self.plan_mxfp8_row_direct(x, layout, data, scales, skip)()
        return data, scales

    def fp8_block128_direct(self, x: torch.Tensor, data: Optional[torch.Tensor] = None,
                            tile_scale_inv: Optional[torch.Tensor] = None, skip: Optional[torch.Tensor] = None):
        """Returns (E4M3 payload uint8 of x's shape, fp32 2^T per 128x128 tile)."""
        rows, K, _ = _rows_view(x)
        if data is None:
            data = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        if tile_scale_inv is None:
            tile_scale_inv = torch.empty(((rows + 127) // 128, (K + 127) // 128), dtype=torch.float32,
                                         device=x.device)
        self.plan_fp8_block128_direct(x, data, tile_scale_inv, skip)()
        return data, tile_scale_inv

    def mxfp8_col_direct(self, x: torch.Tensor, layout="compact", data: Optional[torch.Tensor] = None,
                         scales: Optional[torch.Tensor] = None, skip: Optional[torch.Tensor] = None):
        """Returns (payload uint8 [rows, K], scales of the K x ceil(rows/32)
        transposed scale matrix: compact (K, nbr), padded/swizzled (Kp, Cp))."""
        rows, K, _ = _rows_view(x)
        nbr = (rows + 31) // 32
        if data is None:
            data = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
        if scales is None:
            if _LAYOUTS[layout] == COMPACT:
                scales = torch.empty((K, nbr), dtype=torch.uint8, device=x.device)
            else:
                scales = torch.empty(((K + 127) // 128 * 128, (nbr + 3) // 4 * 4), dtype=torch.uint8, device=x.device)
        self.plan_mxfp8_col_direct(x, layout, data, scales, skip)()
        return data, scales

    def mxfp4_pack(self, x: torch.Tensor, layout="compact", packed: Optional[torch.Tensor] = None,
                   scales: Optional[torch.Tensor] = None, skip: Optional[torch.Tensor] = None):
        """Returns (nibbles uint8 (*shape[:-1], ceil(K/2)), scales) of the
        packed MXFP4 form; scales shaped as in mxfp8_row_direct."""
        rows, K, _ = _rows_view(x)
        if packed is None:
            packed = torch.empty(tuple(x.shape[:-1]) + ((K + 1) // 2,), dtype=torch.uint8, device=x.device)
        if scales is None:
            scales = self._scale_buffer(x, rows, K, layout)
        self.plan_mxfp4_pack(x, layout, packed, scales, skip)()
        return packed, scales

    def _scale_buffer(self, x, rows, K, layout):
        nb = scale_cols(K)
        if _LAYOUTS[layout] == COMPACT:
            return torch.empty(tuple(x.shape[:-1]) + (nb,), dtype=torch.uint8, device=x.device)
        return torch.empty(((rows + 127) // 128 * 128, (nb + 3) // 4 * 4), dtype=torch.uint8, device=x.device)

    def dequantize(self, data: torch.Tensor, *, scales: Optional[torch.Tensor] = None, layout="compact",
                   fp8="e4m3", tile_scale_inv: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                   out: Optional[torch.Tensor] = None, mxfp4_K: Optional[int] = None,
                   columnwise: bool = False) -> torch.Tensor:
        """MXFP8 rowwise (pass ``scales``), 128x128 blockwise (pass
        ``tile_scale_inv``) or packed MXFP4 (pass ``scales`` and ``mxfp4_K``,
        the unpacked row length) -> bf16 / fp32."""
        if out is None:
            shape = data.shape if mxfp4_K is None else tuple(data.shape[:-1]) + (mxfp4_K,)
            out = torch.empty(shape, dtype=out_dtype, device=data.device)
        self.plan_dequantize(data, out, scales=scales, layout=layout, fp8=fp8, tile_scale_inv=tile_scale_inv,
                             mxfp4=mxfp4_K is not None, columnwise=columnwise)()
        return out

    def export_mxfp8(self, data: Optional[torch.Tensor], scales: torch.Tensor, *, shape, layout="compact",
                     fp8="e4m3", scale_out: Optional[torch.Tensor] = None) -> MXFP8Components:
        """export_components of an MXFP8 storage whose rowwise payload is
        ``data`` (None = no row-scaled data) and whose scales are held in
        ``layout``."""
        call, comp = self.plan_export_mxfp8(data, scales, shape=shape, layout=layout, fp8=fp8, scale_out=scale_out)
        call()
        return comp

    def plan_export_mxfp8_grouped(self, storages, scale_out: Optional[torch.Tensor] = None):
        """Export many MXFP8 storages at once.  ``storages`` is a list of
        dicts with keys data, scales, shape, layout (default compact) and fp8
        (default e4m3).  The copies share ``scale_out`` (allocated when None)
        and run in one launch per 128 storages.  Returns (Call, list of
        MXFP8Components); the components' scales are valid once the Call has
        run."""
        n = len(storages)
        st = (_Storage * max(n, 1))()
        sizes, keep = [], []
        dev = None
        for g, d in enumerate(storages):
            shape = tuple(d["shape"])
            K = shape[-1] if shape else 0
            rows = 1
            for v in shape[:-1]:
                rows *= v
            data, scales = d.get("data"), d["scales"]
            _need_cuda(data, scales)
            _check_storage(self, data, scales, rows, K, d.get("layout", "compact"))
            for t in (data, scales):
                if t is not None and dev is not None and t.device != dev:
                    raise ValueError("every storage of a grouped export must sit on one device")
                if t is not None:
                    dev = t.device
            st[g].data = data.data_ptr() if data is not None else None
            st[g].scales = scales.data_ptr()
            st[g].fp8 = _fp8_code(d.get("fp8", "e4m3"))
            st[g].lay = _LAYOUTS[d.get("layout", "compact")]
            st[g].rows, st[g].K = rows, K
            nb = scale_cols(K)
            view = st[g].lay == COMPACT or (st[g].lay == PADDED and nb % 4 == 0) or rows * K == 0
            sizes.append((shape, rows, nb, view))
            keep.append((data, scales))
        need = sum(rows * nb for _, rows, nb, view in sizes if not view)
        if scale_out is not None:
            _need_cuda(scale_out)
            if dev is not None and scale_out.device != dev:
                raise ValueError("scale_out must sit on the storages' device")
            if scale_out.dtype != torch.uint8 or not scale_out.is_contiguous():
                raise ValueError("scale_out must be a contiguous uint8 tensor")
        if scale_out is None and need:
            scale_out = torch.empty(need, dtype=torch.uint8, device=dev)
        comps = (_Components * max(n, 1))()
        out, off = [], 0
        for g, (shape, rows, nb, view) in enumerate(sizes):
            data, scales = keep[g]
            fp8_dtype = torch.float8_e4m3fn if st[g].fp8 == _E4M3 else torch.float8_e5m2
            values = data.view(fp8_dtype).view(shape) if data is not None else None
            if view:
                sc = scales.reshape(-1)[: rows * nb].view(shape[:-1] + (nb,))
            else:
                sc = scale_out[off: off + rows * nb].view(shape[:-1] + (nb,))
                off += rows * nb
            out.append(MXFP8Components(values, sc, view))
        if not n:
            return Call(self, None, (), "mxq_export_mxfp8_grouped", (), None), out
        args = (st, n, ctypes.c_void_p(scale_out.data_ptr()) if scale_out is not None else None,
                scale_out.numel() if scale_out is not None else 0, comps, _stream(keep[0][1]))
        return Call(self, self.L.mxq_export_mxfp8_grouped, args, "mxq_export_mxfp8_grouped",
                    (keep, scale_out, st, comps), dev), out

    def export_mxfp8_grouped(self, storages, scale_out: Optional[torch.Tensor] = None):
        """Eager form of plan_export_mxfp8_grouped: runs the copies and
        returns the list of MXFP8Components."""
        call, out = self.plan_export_mxfp8_grouped(storages, scale_out)
        call()
        return out

    def plan_quantize_export_mxfp8(self, x: torch.Tensor, data: Optional[torch.Tensor] = None,
                                   scales: Optional[torch.Tensor] = None):
        """Quantize x (bf16/fp32) to MXFP8 rowwise (direct lift) and export it
        in one call.  Returns (Call, MXFP8Components): the values and compact
        scales are views of ``data`` and ``scales``, valid once the Call has
        run."""
        _need_cuda(x, data, scales)
        dt = _dt_code(x)
        rows, K, ldx = _rows_view(x)
        nb = scale_cols(K)
        if data is None:
            data = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        if scales is None:
            scales = torch.empty(tuple(x.shape[:-1]) + (nb,), dtype=torch.uint8, device=x.device)
        if not data.is_contiguous() or data.numel() != rows * K or data.dtype != torch.uint8:
            raise ValueError("data must be a contiguous uint8 tensor of rows*K bytes")
        _check_bytes(scales, rows * nb, "scales", "rows*ceil(K/32)")
        comp = _Components()
        args = (ctypes.c_void_p(x.data_ptr()), dt, rows, K, ldx, ctypes.c_void_p(data.data_ptr()),
                ctypes.c_void_p(scales.data_ptr()), ctypes.byref(comp), _stream(x))
        call = Call(self, self.L.mxq_quantize_export_mxfp8, args, "mxq_quantize_export_mxfp8",
                    (x, data, scales, comp), x.device)
        return call, MXFP8Components(data.view(torch.float8_e4m3fn).view(x.shape),
                                     scales.reshape(-1)[: rows * nb].view(tuple(x.shape[:-1]) + (nb,)), True)

    def quantize_export_mxfp8(self, x: torch.Tensor, data: Optional[torch.Tensor] = None,
                              scales: Optional[torch.Tensor] = None) -> MXFP8Components:
        """Eager form of plan_quantize_export_mxfp8."""
        call, comp = self.plan_quantize_export_mxfp8(x, data, scales)
        call()
        return comp


class Call:
    """A prepared libmxq call (see Library.plan_*)."""

    __slots__ = ("lib", "fn", "args", "name", "keep", "device")

    def __init__(self, lib: "Library", fn, args, name: str, keep, device):
        self.lib, self.fn, self.args, self.name, self.keep, self.device = lib, fn, args, name, keep, device

    def __call__(self) -> None:
        if self.fn is None:  # nothing to launch (an empty grouped export)
            return
        if torch.cuda.current_device() != self.device.index:
            with torch.cuda.device(self.device):
                status = self.fn(*self.args)
        else:
            status = self.fn(*self.args)
        if status != 0:
            self.lib._check(status, self.name)


_default: Optional[Library] = None
_lock = threading.Lock()


def library() -> Library:
    """The default libmxq, built in-tree on first use."""
    global _default
    with _lock:
        if _default is None:
            _default = Library()
    return _default


def mxq_fake_quant_mxfp4(x, out=None, skip=None):
    return library().fake_quant_mxfp4(x, out, skip)


def mxq_mxfp8_row_direct(x, layout="compact", data=None, scales=None, skip=None):
    return library().mxfp8_row_direct(x, layout, data, scales, skip)


def mxq_fp8_block128_direct(x, data=None, tile_scale_inv=None, skip=None):
    return library().fp8_block128_direct(x, data, tile_scale_inv, skip)


def mxq_mxfp8_col_direct(x, layout="compact", data=None, scales=None, skip=None):
    return library().mxfp8_col_direct(x, layout, data, scales, skip)


def mxq_mxfp4_pack(x, layout="compact", packed=None, scales=None, skip=None):
    return library().mxfp4_pack(x, layout, packed, scales, skip)


def mxq_dequantize(data, **kw):
    return library().dequantize(data, **kw)


def mxq_export_mxfp8(data, scales, **kw):
    return library().export_mxfp8(data, scales, **kw)


def mxq_export_mxfp8_grouped(storages, scale_out=None):
    return library().export_mxfp8_grouped(storages, scale_out)


def mxq_quantize_export_mxfp8(x, data=None, scales=None):
    return library().quantize_export_mxfp8(x, data, scales)


def mxq_scale_bytes(rows, K, layout="compact"):
    return library().scale_bytes(rows, K, layout)


def mxq_tile_scale_count(rows, K):
    return library().tile_scale_count(rows, K)
