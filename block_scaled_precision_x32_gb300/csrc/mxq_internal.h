// mxq_internal.h -- host-side launchers shared between the C entry points
// (mxq_api.cu) and the kernel translation units.  Not part of the ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime_api.h>

namespace mxq {

enum class Elt { BF16, FP32 };
enum class RowMode { PROJECT, MXFP8, MXFP4 };

struct RowwiseArgs {
    const void* x;
    void* y;          // PROJECT output
    uint8_t* data;    // MXFP8 payload [rows, K]; MXFP4 nibbles [rows, ceil(K/2)]
    uint8_t* scales;  // UE8M0 scale bytes in `lay`
    int64_t rows, K, ldx, ldy;
    int lay;          // mxq_scale_layout
    const int32_t* skip;  // optional device flag: nonzero = write nothing
};

struct Block128Args {
    const void* x;
    uint8_t* data;
    float* tile_scale_inv;
    int64_t rows, K, ldx;
    const int32_t* skip;  // optional device flag: nonzero = write nothing
};

struct ColwiseArgs {
    const void* x;
    uint8_t* data;    // [rows, K] E4M3
    uint8_t* scales;  // transposed scale matrix (K x ceil(rows/32)) in `lay`
    int64_t rows, K, ldx;
    int lay;
    const int32_t* skip;  // optional device flag: nonzero = write nothing
};

struct DequantArgs {
    int kind;  // mxq_quant_kind (0 MXFP8 row, 1 128x128, 2 packed MXFP4, 3 MXFP8 columnwise)
    const uint8_t* data;
    int64_t rows, K;
    int fp8;   // mxq_fp8
    const uint8_t* scales;
    int lay;
    const float* tile_scale_inv;
    void* out;
    bool out_bf16;
};

struct ExportArgs {
    const uint8_t* scales;
    int lay;
    int path;  // grouped export only: 1 = the chunk kernel's path (set by the launcher)
    int64_t rows, K;
    uint8_t* out;  // compact [rows, nb]
};

// Descriptors of a grouped export, passed by value as kernel parameters.
constexpr int kGroupedMax = 128;
struct GroupedExport {
    ExportArgs item[kGroupedMax];
    int count;
};

// Each returns cudaSuccess or the launch error.
cudaError_t launch_rowwise(RowMode mode, Elt elt, const RowwiseArgs& a, cudaStream_t s);
cudaError_t launch_block128(Elt elt, const Block128Args& a, cudaStream_t s);
cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t s);
cudaError_t launch_export(const ExportArgs& a, cudaStream_t s);
cudaError_t launch_export_grouped(const GroupedExport& b, cudaStream_t s);
cudaError_t launch_colwise(Elt elt, const ColwiseArgs& a, cudaStream_t s);
cudaError_t launch_colwise_dequant(const DequantArgs& a, cudaStream_t s);

// Resident-grid sizing: number of SMs of the current device (cached).
int sm_count();

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace mxq
