// mxq_api.cu -- the C entry points of libmxq: host-side argument checks,
// then one kernel launch on the caller's stream.  Declared and documented
// in include/mxq.h.
#include <cuda_runtime.h>

#include <atomic>

#include <cstdint>

#include "../../include/mxq.h"
#include "mxq_internal.h"

namespace mxq {

int sm_count() {
    static std::atomic<int> cached[64];  // zero-initialised; one SM count per device, written once
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
    const int slot = dev < 64 ? dev : 63;
    if (cached[slot].load(std::memory_order_relaxed) == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        cached[slot].store(n, std::memory_order_relaxed);
    }
    return cached[slot];
}

}  // namespace mxq

namespace {

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

mxq_status check_dtype(mxq_dtype dt) {
    if (dt == MXQ_BF16 || dt == MXQ_FP32) return MXQ_OK;
    if (dt == MXQ_FP16) return MXQ_ERR_UNSUPPORTED_DTYPE;
    return MXQ_ERR_INVALID_ARG;
}

size_t elt_size(mxq_dtype dt) { return dt == MXQ_BF16 ? 2 : 4; }

bool valid_layout(mxq_scale_layout lay) {
    return lay == MXQ_SCALES_COMPACT || lay == MXQ_SCALES_PADDED || lay == MXQ_SCALES_SWIZZLED;
}

// rows, K >= 0; ld >= K; the byte span of the view fits in int64.
bool valid_shape(int64_t rows, int64_t K, int64_t ld) {
    if (rows < 0 || K < 0 || ld < K) return false;
    if (rows > 0 && ld > (INT64_C(1) << 40)) return false;
    if (rows > (INT64_C(1) << 40) || K > (INT64_C(1) << 40)) return false;
    return true;
}

mxq_status launch_status(cudaError_t e) { return e == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA; }

mxq::Elt elt_of(mxq_dtype dt) { return dt == MXQ_BF16 ? mxq::Elt::BF16 : mxq::Elt::FP32; }

}  // namespace

extern "C" {

size_t mxq_scale_bytes(int64_t rows, int64_t K, mxq_scale_layout lay) {
    if (rows <= 0 || K <= 0) return 0;
    const int64_t nb = (K + 31) / 32;
    if (lay == MXQ_SCALES_COMPACT) return (size_t)(rows * nb);
    return (size_t)(((rows + 127) / 128 * 128) * ((nb + 3) / 4 * 4));
}

size_t mxq_tile_scale_count(int64_t rows, int64_t K) {
    if (rows <= 0 || K <= 0) return 0;
    return (size_t)(((rows + 127) / 128) * ((K + 127) / 128));
}

mxq_status mxq_fake_quant_mxfp4_update(const void* x, void* y, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                       int64_t ldy, const int32_t* skip, cudaStream_t stream) {
    mxq_status st = check_dtype(dt);
    if (st != MXQ_OK) return st;
    if (!valid_shape(rows, K, ldx) || !valid_shape(rows, K, ldy)) return MXQ_ERR_INVALID_ARG;
    if (rows == 0 || K == 0) return MXQ_OK;
    if (!x || !y || !aligned(x, elt_size(dt)) || !aligned(y, elt_size(dt))) return MXQ_ERR_INVALID_ARG;
    if (x == y && ldx != ldy) return MXQ_ERR_INVALID_ARG;
    if (skip && !aligned(skip, 4)) return MXQ_ERR_INVALID_ARG;
    mxq::RowwiseArgs a{};
    a.x = x;
    a.y = y;
    a.rows = rows;
    a.K = K;
    a.ldx = ldx;
    a.ldy = ldy;
    a.skip = skip;
    return launch_status(mxq::launch_rowwise(mxq::RowMode::PROJECT, elt_of(dt), a, stream));
}

mxq_status mxq_fake_quant_mxfp4(const void* x, void* y, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                int64_t ldy, cudaStream_t stream) {
    return mxq_fake_quant_mxfp4_update(x, y, dt, rows, K, ldx, ldy, nullptr, stream);
}

static mxq_status rowwise_quant(mxq::RowMode mode, const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                uint8_t* data, uint8_t* scales, mxq_scale_layout lay, const int32_t* skip,
                                cudaStream_t stream) {
    mxq_status st = check_dtype(dt);
    if (st != MXQ_OK) return st;
    if (!valid_shape(rows, K, ldx) || !valid_layout(lay)) return MXQ_ERR_INVALID_ARG;
    if (rows == 0 || K == 0) return MXQ_OK;
    if (!x || !data || !scales || !aligned(x, elt_size(dt))) return MXQ_ERR_INVALID_ARG;
    if (skip && !aligned(skip, 4)) return MXQ_ERR_INVALID_ARG;
    mxq::RowwiseArgs a{};
    a.x = x;
    a.data = data;
    a.scales = scales;
    a.rows = rows;
    a.K = K;
    a.ldx = ldx;
    a.ldy = K;
    a.lay = (int)lay;
    a.skip = skip;
    return launch_status(mxq::launch_rowwise(mode, elt_of(dt), a, stream));
}

mxq_status mxq_mxfp8_row_direct_update(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                       uint8_t* data, uint8_t* scales, mxq_scale_layout lay, const int32_t* skip,
                                       cudaStream_t stream) {
    return rowwise_quant(mxq::RowMode::MXFP8, x, dt, rows, K, ldx, data, scales, lay, skip, stream);
}

mxq_status mxq_mxfp8_row_direct(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* data,
                                uint8_t* scales, mxq_scale_layout lay, cudaStream_t stream) {
    return rowwise_quant(mxq::RowMode::MXFP8, x, dt, rows, K, ldx, data, scales, lay, nullptr, stream);
}

mxq_status mxq_mxfp4_pack_update(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* packed,
                                 uint8_t* scales, mxq_scale_layout lay, const int32_t* skip, cudaStream_t stream) {
    return rowwise_quant(mxq::RowMode::MXFP4, x, dt, rows, K, ldx, packed, scales, lay, skip, stream);
}

mxq_status mxq_mxfp4_pack(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* packed,
                          uint8_t* scales, mxq_scale_layout lay, cudaStream_t stream) {
    return rowwise_quant(mxq::RowMode::MXFP4, x, dt, rows, K, ldx, packed, scales, lay, nullptr, stream);
}

mxq_status mxq_mxfp8_col_direct_update(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                       uint8_t* data, uint8_t* scales, mxq_scale_layout lay, const int32_t* skip,
                                       cudaStream_t stream) {
    mxq_status st = check_dtype(dt);
    if (st != MXQ_OK) return st;
    if (!valid_shape(rows, K, ldx) || !valid_layout(lay)) return MXQ_ERR_INVALID_ARG;
    if (rows == 0 || K == 0) return MXQ_OK;
    if (!x || !data || !scales || !aligned(x, elt_size(dt))) return MXQ_ERR_INVALID_ARG;
    if (skip && !aligned(skip, 4)) return MXQ_ERR_INVALID_ARG;
    mxq::ColwiseArgs a{};
    a.x = x;
    a.data = data;
    a.scales = scales;
    a.rows = rows;
    a.K = K;
    a.ldx = ldx;
    a.lay = (int)lay;
    a.skip = skip;
    return launch_status(mxq::launch_colwise(elt_of(dt), a, stream));
}

mxq_status mxq_mxfp8_col_direct(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* data,
                                uint8_t* scales, mxq_scale_layout lay, cudaStream_t stream) {
    return mxq_mxfp8_col_direct_update(x, dt, rows, K, ldx, data, scales, lay, nullptr, stream);
}

mxq_status mxq_fp8_block128_direct_update(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                          uint8_t* data, float* tile_scale_inv, const int32_t* skip,
                                          cudaStream_t stream) {
    mxq_status st = check_dtype(dt);
    if (st != MXQ_OK) return st;
    if (!valid_shape(rows, K, ldx)) return MXQ_ERR_INVALID_ARG;
    if (rows == 0 || K == 0) return MXQ_OK;
    if (!x || !data || !tile_scale_inv || !aligned(x, elt_size(dt)) || !aligned(tile_scale_inv, 4))
        return MXQ_ERR_INVALID_ARG;
    if (skip && !aligned(skip, 4)) return MXQ_ERR_INVALID_ARG;
    mxq::Block128Args a{};
    a.x = x;
    a.data = data;
    a.tile_scale_inv = tile_scale_inv;
    a.rows = rows;
    a.K = K;
    a.ldx = ldx;
    a.skip = skip;
    return launch_status(mxq::launch_block128(elt_of(dt), a, stream));
}

mxq_status mxq_fp8_block128_direct(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* data,
                                   float* tile_scale_inv, cudaStream_t stream) {
    return mxq_fp8_block128_direct_update(x, dt, rows, K, ldx, data, tile_scale_inv, nullptr, stream);
}

mxq_status mxq_dequantize(const mxq_quantized* q, void* out, mxq_dtype out_dt, cudaStream_t stream) {
    if (!q) return MXQ_ERR_INVALID_ARG;
    mxq_status st = check_dtype(out_dt);
    if (st != MXQ_OK) return st;
    if (!valid_shape(q->rows, q->K, q->K)) return MXQ_ERR_INVALID_ARG;
    if (q->kind != MXQ_QUANT_MXFP8_ROW && q->kind != MXQ_QUANT_FP8_BLOCK128 && q->kind != MXQ_QUANT_MXFP4 &&
        q->kind != MXQ_QUANT_MXFP8_COL)
        return MXQ_ERR_INVALID_ARG;
    if (q->kind != MXQ_QUANT_MXFP4 && q->fp8 != MXQ_E4M3 && q->fp8 != MXQ_E5M2) return MXQ_ERR_INVALID_ARG;
    if (q->kind == MXQ_QUANT_FP8_BLOCK128 && q->fp8 != MXQ_E4M3) return MXQ_ERR_INVALID_ARG;
    if (q->kind != MXQ_QUANT_FP8_BLOCK128 && !valid_layout(q->lay)) return MXQ_ERR_INVALID_ARG;
    if (q->rows == 0 || q->K == 0) return MXQ_OK;
    if (!q->data || !out || !aligned(out, elt_size(out_dt))) return MXQ_ERR_INVALID_ARG;
    if (q->kind != MXQ_QUANT_FP8_BLOCK128 && !q->scales) return MXQ_ERR_INVALID_ARG;
    if (q->kind == MXQ_QUANT_FP8_BLOCK128 && (!q->tile_scale_inv || !aligned(q->tile_scale_inv, 4)))
        return MXQ_ERR_INVALID_ARG;
    mxq::DequantArgs a{};
    a.kind = (int)q->kind;
    a.data = q->data;
    a.rows = q->rows;
    a.K = q->K;
    a.fp8 = (int)q->fp8;
    a.scales = q->scales;
    a.lay = (int)q->lay;
    a.tile_scale_inv = q->tile_scale_inv;
    a.out = out;
    a.out_bf16 = out_dt == MXQ_BF16;
    if (q->kind == MXQ_QUANT_MXFP8_COL) return launch_status(mxq::launch_colwise_dequant(a, stream));
    return launch_status(mxq::launch_dequant(a, stream));
}

// Validation and view logic shared by the single and grouped exports: fills
// `c` and reports whether a copy is needed (rows * nb bytes).
static mxq_status export_plan(const mxq_mxfp8_storage* st, mxq_mxfp8_components* c, bool* copy) {
    if (!st) return MXQ_ERR_INVALID_ARG;
    if (!valid_shape(st->rows, st->K, st->K) || !valid_layout(st->lay)) return MXQ_ERR_INVALID_ARG;
    if (st->fp8 != MXQ_E4M3 && st->fp8 != MXQ_E5M2) return MXQ_ERR_INVALID_ARG;
    const int64_t nb = (st->K + 31) / 32;
    const bool empty = st->rows == 0 || st->K == 0;
    if (!st->data && !empty) return MXQ_ERR_NO_ROWWISE_DATA;
    if (!st->scales && !empty) return MXQ_ERR_INVALID_ARG;
    *c = mxq_mxfp8_components{};
    c->data = st->data;
    c->fp8 = st->fp8;
    c->rows = st->rows;
    c->K = st->K;
    c->scale_cols = nb;
    const bool view = st->lay == MXQ_SCALES_COMPACT || (st->lay == MXQ_SCALES_PADDED && nb % 4 == 0);
    *copy = !(empty || view);
    if (!*copy) {
        c->scales = st->scales;
        c->is_view = 1;
    }
    return MXQ_OK;
}

mxq_status mxq_export_mxfp8(const mxq_mxfp8_storage* st, uint8_t* scale_out, size_t scale_out_bytes,
                            mxq_mxfp8_components* out, cudaStream_t stream) {
    if (!st || !out) return MXQ_ERR_INVALID_ARG;
    mxq_mxfp8_components c;
    bool copy = false;
    mxq_status s = export_plan(st, &c, &copy);
    if (s != MXQ_OK) return s;
    if (!copy) {
        *out = c;
        return MXQ_OK;
    }
    if (!scale_out || scale_out_bytes < (size_t)(st->rows * c.scale_cols)) return MXQ_ERR_BUFFER_TOO_SMALL;
    mxq::ExportArgs a{};
    a.scales = st->scales;
    a.lay = (int)st->lay;
    a.rows = st->rows;
    a.K = st->K;
    a.out = scale_out;
    const mxq_status ls = launch_status(mxq::launch_export(a, stream));
    if (ls != MXQ_OK) return ls;
    c.scales = scale_out;
    c.is_view = 0;
    *out = c;
    return MXQ_OK;
}

mxq_status mxq_export_mxfp8_grouped(const mxq_mxfp8_storage* st, int64_t count, uint8_t* scale_out,
                                    size_t scale_out_bytes, mxq_mxfp8_components* out, cudaStream_t stream) {
    if (count < 0 || (count > 0 && (!st || !out))) return MXQ_ERR_INVALID_ARG;
    // check everything and size the copies before launching anything
    size_t need = 0;
    for (int64_t g = 0; g < count; ++g) {
        mxq_mxfp8_components c;
        bool copy = false;
        mxq_status s = export_plan(&st[g], &c, &copy);
        if (s != MXQ_OK) return s;
        if (copy) need += (size_t)(st[g].rows * c.scale_cols);
    }
    if (need > 0 && (!scale_out || scale_out_bytes < need)) return MXQ_ERR_BUFFER_TOO_SMALL;
    mxq::GroupedExport batch{};
    size_t off = 0;
    for (int64_t g = 0; g < count; ++g) {
        mxq_mxfp8_components c;
        bool copy = false;
        export_plan(&st[g], &c, &copy);
        if (copy) {
            mxq::ExportArgs& a = batch.item[batch.count++];
            a.scales = st[g].scales;
            a.lay = (int)st[g].lay;
            a.rows = st[g].rows;
            a.K = st[g].K;
            a.out = scale_out + off;
            c.scales = scale_out + off;
            c.is_view = 0;
            off += (size_t)(st[g].rows * c.scale_cols);
            if (batch.count == mxq::kGroupedMax) {
                const mxq_status ls = launch_status(mxq::launch_export_grouped(batch, stream));
                if (ls != MXQ_OK) return ls;
                batch.count = 0;
            }
        }
        out[g] = c;
    }
    return launch_status(mxq::launch_export_grouped(batch, stream));
}

mxq_status mxq_quantize_export_mxfp8(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                     uint8_t* data, uint8_t* scales, mxq_mxfp8_components* out, cudaStream_t stream) {
    if (!out) return MXQ_ERR_INVALID_ARG;
    const mxq_status s = rowwise_quant(mxq::RowMode::MXFP8, x, dt, rows, K, ldx, data, scales, MXQ_SCALES_COMPACT,
                                       nullptr, stream);
    if (s != MXQ_OK) return s;
    mxq_mxfp8_components c{};
    c.data = data;
    c.fp8 = MXQ_E4M3;
    c.scales = scales;
    c.rows = rows;
    c.K = K;
    c.scale_cols = (K + 31) / 32;
    c.is_view = 1;
    *out = c;
    return MXQ_OK;
}

const char* mxq_status_string(mxq_status s) {
    switch (s) {
        case MXQ_OK: return "ok";
        case MXQ_ERR_INVALID_ARG: return "invalid argument";
        case MXQ_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype (fp16 is rejected)";
        case MXQ_ERR_NO_ROWWISE_DATA: return "tensor has no row-scaled data";
        case MXQ_ERR_BUFFER_TOO_SMALL: return "scale output buffer too small";
        case MXQ_ERR_CUDA: return "CUDA launch failed";
    }
    return "unknown status";
}

int mxq_version(void) { return MXQ_VERSION; }

}  // extern "C"
