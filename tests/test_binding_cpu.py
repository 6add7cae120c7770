"""Host-side checks of the Python binding, without a GPU.

The C ABI receives raw pointers and cannot see how long a buffer is, so the
binding checks every scale buffer, tile-scale tensor and payload tensor
against the size its layout needs before anything is launched.  These tests
drive those checks directly on CPU tensors."""

import pytest
import torch

import block_scaled_precision_x32_gb300 as mxq


@pytest.fixture(scope="module")
def lib():
    return mxq.Library()


def test_scale_buffer_sizes_are_checked(lib):
    need = lib.scale_bytes(256, 7184, "swizzled")  # 256 rows x 228 padded columns
    assert need == 256 * 228
    mxq._check_bytes(torch.zeros(need, dtype=torch.uint8), need, "scales", "layout")
    with pytest.raises(ValueError):
        mxq._check_bytes(torch.zeros(need - 1, dtype=torch.uint8), need, "scales", "layout")
    with pytest.raises(ValueError):  # right size, wrong dtype
        mxq._check_bytes(torch.zeros(need, dtype=torch.int8), need, "scales", "layout")
    with pytest.raises(ValueError):  # right size, not contiguous
        mxq._check_bytes(torch.zeros(2 * need, dtype=torch.uint8)[::2], need, "scales", "layout")


def test_storage_checks_cover_layout_and_payload(lib):
    rows, K = 200, 7184  # 225 scale columns: the compact, padded and swizzled sizes all differ
    compact, padded = lib.scale_bytes(rows, K, "compact"), lib.scale_bytes(rows, K, "padded")
    assert compact == 200 * 225 and padded == 256 * 228
    data = torch.zeros(rows * K, dtype=torch.uint8)
    mxq._check_storage(lib, data, torch.zeros(compact, dtype=torch.uint8), rows, K, "compact")
    mxq._check_storage(lib, None, torch.zeros(padded, dtype=torch.uint8), rows, K, "swizzled")
    with pytest.raises(ValueError):  # a compact-sized buffer handed in as swizzled
        mxq._check_storage(lib, data, torch.zeros(compact, dtype=torch.uint8), rows, K, "swizzled")
    with pytest.raises(ValueError):  # payload one row short
        mxq._check_storage(lib, data[: (rows - 1) * K], torch.zeros(compact, dtype=torch.uint8), rows, K, "compact")
    with pytest.raises(ValueError):  # payload as bf16, not bytes
        mxq._check_storage(lib, torch.zeros(rows * K, dtype=torch.bfloat16), torch.zeros(compact, dtype=torch.uint8),
                           rows, K, "compact")


def test_cpu_tensors_are_refused_before_any_call(lib):
    x = torch.zeros(64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lib.plan_mxfp8_col_direct(x, "compact", torch.zeros(64, 64, dtype=torch.uint8),
                                  torch.zeros(128, dtype=torch.uint8))
    with pytest.raises(ValueError):
        lib.plan_dequantize(torch.zeros(64, 64, dtype=torch.uint8), torch.zeros(64, 64, dtype=torch.bfloat16),
                            scales=torch.zeros(128, dtype=torch.uint8))
    with pytest.raises(ValueError):
        lib.export_mxfp8_grouped([{"data": None, "scales": torch.zeros(128, dtype=torch.uint8), "shape": (64, 64)}])
