// mxq_export.cu -- the copy behind export_components(): compact
// (rows, ceil(K/32)) UE8M0 scales out of a padded or GEMM-swizzled buffer.
//
// TE PR #3790 "MXFP8TensorStorage.export_components()", Description:
// scales are copied only when padded in the last dimension or swizzled for
// GEMM, padding dropped and the swizzle undone.
//
// Swizzled input: one CTA per (128-row tile, group of 32 column tiles).
// The group's bytes are contiguous in the swizzled buffer (32 x 512), so
// they are staged in shared memory with 16-byte loads -- each 512-byte tile
// padded by one word so that lanes reading the same word of consecutive
// tiles hit distinct banks -- and written out row by row, consecutive lanes
// on consecutive output words (4 scales) or bytes.
// Padded input: one warp per row, lanes on consecutive bytes.
// Grouped export: up to kGroupedMax storages per launch, their descriptors
// passed by value in the kernel parameters.
#include <cuda_runtime.h>

#include <algorithm>

#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kGroup = 32;        // column tiles (4 scale columns each) per CTA
constexpr int kTileWords = 129;   // 128 words of a 512-byte tile + 1 pad word

// One (128-row tile rt, group of column tiles starting at jt0) of a
// swizzled scale buffer -> compact rows.  `tile` is the CTA's staging area.
template <bool VEC_IN, bool WORD_OUT>
__device__ __forceinline__ void unswizzle_group(const ExportArgs& a, int64_t rt, int64_t jt0, uint32_t* tile) {
    const int64_t nb = (a.K + 31) >> 5;
    const int64_t Cp = (nb + 3) & ~int64_t(3);
    const int64_t ct = Cp >> 2;  // column tiles per row tile
    const int g = (int)min((int64_t)kGroup, ct - jt0);
    const int W = (int)min((int64_t)4 * g, nb - 4 * jt0);  // output columns of this group
    const uint8_t* src = a.scales + (rt * ct + jt0) * 512;
    if constexpr (VEC_IN) {
        for (int i = threadIdx.x; i < g * 32; i += kThreads) {
            const uint4 q = reinterpret_cast<const uint4*>(src)[i];
            uint32_t* d = tile + (i >> 5) * kTileWords + (i & 31) * 4;
            d[0] = q.x;
            d[1] = q.y;
            d[2] = q.z;
            d[3] = q.w;
        }
    } else {
        for (int i = threadIdx.x; i < g * 128; i += kThreads) {
            const uint8_t* b = src + 4 * i;
            tile[(i >> 7) * kTileWords + (i & 127)] =
                b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) | ((uint32_t)b[3] << 24);
        }
    }
    __syncthreads();
    const int64_t r0 = rt * 128;
    const int nrows = (int)min((int64_t)128, a.rows - r0);
    if constexpr (WORD_OUT) {
        // nb % 4 == 0: the 4 scales of a (row, column tile) are one aligned word
        uint32_t* out = reinterpret_cast<uint32_t*>(a.out);
        for (int idx = threadIdx.x; idx < nrows * g; idx += kThreads) {
            const int rr = idx / g, jt = idx - rr * g;
            out[(r0 + rr) * (nb >> 2) + jt0 + jt] = tile[jt * kTileWords + (rr & 31) * 4 + (rr >> 5)];
        }
    } else {
        for (int idx = threadIdx.x; idx < nrows * W; idx += kThreads) {
            const int rr = idx / W, j = idx - rr * W;
            const uint32_t word = tile[(j >> 2) * kTileWords + (rr & 31) * 4 + (rr >> 5)];
            a.out[(r0 + rr) * nb + 4 * jt0 + j] = (uint8_t)(word >> ((j & 3) * 8));
        }
    }
    __syncthreads();
}

template <bool VEC_IN, bool WORD_OUT>
__global__ void __launch_bounds__(kThreads) unswizzle_kernel(ExportArgs a, int64_t tiles_r) {
    __shared__ uint32_t tile[kGroup * kTileWords];
    const int64_t jt0 = (int64_t)blockIdx.x * kGroup;
    for (int64_t rt = blockIdx.y; rt < tiles_r; rt += gridDim.y) unswizzle_group<VEC_IN, WORD_OUT>(a, rt, jt0, tile);
}

// Rows [r0, r1) of a padded buffer -> compact; one warp per row.
__device__ __forceinline__ void unpad_rows(const ExportArgs& a, int64_t r0, int64_t r1, int64_t warp, int64_t nwarps) {
    const int64_t nb = (a.K + 31) >> 5;
    const int64_t Cp = (nb + 3) & ~int64_t(3);
    const int lane = threadIdx.x & 31;
    for (int64_t r = r0 + warp; r < r1; r += nwarps)
        for (int64_t j = lane; j < nb; j += 32) a.out[r * nb + j] = a.scales[r * Cp + j];
}

__global__ void __launch_bounds__(kThreads) unpad_kernel(ExportArgs a) {
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    unpad_rows(a, 0, a.rows, warp, nwarps);
}

// Many storages in one launch: blockIdx.z picks the storage, (x, y) its
// column group and 128-row tile; CTAs outside a storage's extent return.
__global__ void __launch_bounds__(kThreads) grouped_export_kernel(GroupedExport b) {
    __shared__ uint32_t tile[kGroup * kTileWords];
    const ExportArgs& a = b.item[blockIdx.z];
    const int64_t nb = (a.K + 31) >> 5;
    const int64_t rt = blockIdx.y, tr = (a.rows + 127) >> 7;
    if (rt >= tr) return;
    if (a.lay == 2) {
        const int64_t ct = ((nb + 3) >> 2), jt0 = (int64_t)blockIdx.x * kGroup;
        if (jt0 >= ct) return;
        unswizzle_group<false, false>(a, rt, jt0, tile);
    } else if (blockIdx.x == 0) {
        unpad_rows(a, rt * 128, min(a.rows, rt * 128 + 128), threadIdx.x >> 5, kThreads / 32);
    }
}

}  // namespace

cudaError_t launch_export(const ExportArgs& a, cudaStream_t s) {
    const int64_t nb = ceil_div(a.K, 32);
    if (a.lay == 2) {
        const int64_t ct = ceil_div(nb, 4);
        const int64_t tr = ceil_div(a.rows, 128);
        const int64_t gx = ceil_div(ct, kGroup);
        const unsigned gy = (unsigned)(tr < 65535 ? tr : 65535);
        const dim3 grid((unsigned)gx, gy);
        const bool vin = (reinterpret_cast<uintptr_t>(a.scales) & 15) == 0;
        const bool wout = nb % 4 == 0 && (reinterpret_cast<uintptr_t>(a.out) & 3) == 0;
        if (vin && wout)
            unswizzle_kernel<true, true><<<grid, kThreads, 0, s>>>(a, tr);
        else if (vin)
            unswizzle_kernel<true, false><<<grid, kThreads, 0, s>>>(a, tr);
        else if (wout)
            unswizzle_kernel<false, true><<<grid, kThreads, 0, s>>>(a, tr);
        else
            unswizzle_kernel<false, false><<<grid, kThreads, 0, s>>>(a, tr);
    } else {
        int64_t grid = ceil_div(a.rows, kThreads / 32);
        const int64_t cap = (int64_t)sm_count() * 8;
        if (grid > cap) grid = cap;
        unpad_kernel<<<(unsigned)grid, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_export_grouped(const GroupedExport& b, cudaStream_t s) {
    if (b.count <= 0) return cudaSuccess;
    int64_t gx = 1, gy = 1;
    for (int i = 0; i < b.count; ++i) {
        const int64_t nb = ceil_div(b.item[i].K, 32);
        gx = std::max(gx, ceil_div(ceil_div(nb, 4), kGroup));
        gy = std::max(gy, ceil_div(b.item[i].rows, 128));
    }
    if (gy > 65535) return cudaErrorInvalidValue;
    grouped_export_kernel<<<dim3((unsigned)gx, (unsigned)gy, (unsigned)b.count), kThreads, 0, s>>>(b);
    return cudaGetLastError();
}

}  // namespace mxq
