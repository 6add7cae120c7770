// mxq_export.cu -- the copy behind export_components(): compact
// (rows, ceil(K/32)) UE8M0 scales out of a padded or GEMM-swizzled buffer.
//
// TE PR #3790 "MXFP8TensorStorage.export_components()", Description:
// scales are copied only when padded in the last dimension or swizzled for
// GEMM, padding dropped and the swizzle undone.
//
// Swizzled input: one CTA per (128-row tile, group of 32 column tiles).
// The group's bytes are contiguous in the swizzled buffer (32 x 512), so
// they are staged in shared memory with 16-byte loads and written out row
// by row, consecutive threads on consecutive output bytes.
// Padded input: one warp per row, lanes on consecutive bytes.
#include <cuda_runtime.h>

#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kGroup = 32;  // column tiles (4 scale columns each) per CTA

template <bool VEC>
__global__ void __launch_bounds__(kThreads) unswizzle_kernel(ExportArgs a, int64_t tiles_r) {
    __shared__ __align__(16) uint8_t tile[kGroup * 512];
    const int64_t nb = (a.K + 31) >> 5;
    const int64_t Cp = (nb + 3) & ~int64_t(3);
    const int64_t ct = Cp >> 2;  // column tiles per row tile
    const int64_t jt0 = (int64_t)blockIdx.x * kGroup;
    const int64_t g = min((int64_t)kGroup, ct - jt0);
    const int64_t W = min(4 * g, nb - 4 * jt0);  // output columns of this group
    for (int64_t rt = blockIdx.y; rt < tiles_r; rt += gridDim.y) {
        const uint8_t* src = a.scales + (rt * ct + jt0) * 512;
        if (VEC) {
            for (int64_t i = threadIdx.x; i < g * 32; i += kThreads)
                reinterpret_cast<uint4*>(tile)[i] = reinterpret_cast<const uint4*>(src)[i];
        } else {
            for (int64_t i = threadIdx.x; i < g * 512; i += kThreads) tile[i] = src[i];
        }
        __syncthreads();
        const int64_t r0 = rt * 128;
        const int64_t nrows = min((int64_t)128, a.rows - r0);
        for (int64_t idx = threadIdx.x; idx < nrows * W; idx += kThreads) {
            const int64_t rr = idx / W, j = idx - rr * W;
            const int64_t off = (j >> 2) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (j & 3);
            a.out[(r0 + rr) * nb + 4 * jt0 + j] = tile[off];
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreads) unpad_kernel(ExportArgs a) {
    const int64_t nb = (a.K + 31) >> 5;
    const int64_t Cp = (nb + 3) & ~int64_t(3);
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    for (int64_t r = warp; r < a.rows; r += nwarps)
        for (int64_t j = lane; j < nb; j += 32) a.out[r * nb + j] = a.scales[r * Cp + j];
}

}  // namespace

cudaError_t launch_export(const ExportArgs& a, cudaStream_t s) {
    const int64_t nb = ceil_div(a.K, 32);
    if (a.lay == 2) {
        const int64_t ct = ceil_div(nb, 4);
        const int64_t tr = ceil_div(a.rows, 128);
        const int64_t gx = ceil_div(ct, kGroup);
        const unsigned gy = (unsigned)(tr < 65535 ? tr : 65535);
        const bool vec = (reinterpret_cast<uintptr_t>(a.scales) & 15) == 0;
        if (vec)
            unswizzle_kernel<true><<<dim3((unsigned)gx, gy), kThreads, 0, s>>>(a, tr);
        else
            unswizzle_kernel<false><<<dim3((unsigned)gx, gy), kThreads, 0, s>>>(a, tr);
    } else {
        int64_t grid = ceil_div(a.rows, kThreads / 32);
        const int64_t cap = (int64_t)sm_count() * 8;
        if (grid > cap) grid = cap;
        unpad_kernel<<<(unsigned)grid, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace mxq
