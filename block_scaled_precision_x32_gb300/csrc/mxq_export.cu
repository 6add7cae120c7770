// mxq_export.cu -- the copy behind export_components(): compact
// (rows, ceil(K/32)) UE8M0 scales out of a padded or GEMM-swizzled buffer.
//
// TE PR #3790 "MXFP8TensorStorage.export_components()", Description:
// scales are copied only when padded in the last dimension or swizzled for
// GEMM, padding dropped and the swizzle undone.
//
// Swizzled input: one CTA per (128-row tile, group of 16 column tiles).
// The group's bytes are contiguous in the swizzled buffer (16 x 512), so
// they are staged in shared memory with 16-byte loads -- each 512-byte tile
// padded by one word so that lanes reading the same word of consecutive
// tiles hit distinct banks -- and written out row by row, consecutive lanes
// on consecutive output words (4 scales) or bytes.
// Swizzled input with nb % 4 != 0 (compact rows are not whole words): one CTA
// per 128-row tile stages all of the tile's column tiles, and writes the
// tile's compact output -- one contiguous range -- as aligned words.
// Padded input: one warp per row, lanes on consecutive bytes.
// Grouped export: up to kGroupedMax storages per launch, their descriptors
// passed by value in the kernel parameters.
#include <cuda_runtime.h>

#include <algorithm>

#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kGroup = 16;        // column tiles (4 scale columns each) per CTA: 3.6 us at 8192^2 against 4.1 for 32
constexpr int kTileWords = 129;   // 128 words of a 512-byte tile + 1 pad word

// Stage `ntiles` consecutive 512-byte swizzled tiles from `src` into `tile`
// (kTileWords words per tile).  Each thread issues up to kStageBatch loads
// before its first shared-memory store, so the loads of a thread overlap
// instead of paying one memory latency each.
constexpr int kStageBatch = 8;

template <bool VEC_IN, int BATCH = kStageBatch, int NT = kThreads>
__device__ __forceinline__ void stage_tiles(const uint8_t* src, int ntiles, uint32_t* tile) {
    if constexpr (VEC_IN) {
        const int n = ntiles * 32;  // 16-byte chunks
        for (int base = 0; base < n; base += BATCH * NT) {
            uint4 q[BATCH];
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int i = base + u * NT + (int)threadIdx.x;
                if (i < n) q[u] = reinterpret_cast<const uint4*>(src)[i];
            }
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int i = base + u * NT + (int)threadIdx.x;
                if (i < n) {
                    uint32_t* d = tile + (i >> 5) * kTileWords + (i & 31) * 4;
                    d[0] = q[u].x;
                    d[1] = q[u].y;
                    d[2] = q[u].z;
                    d[3] = q[u].w;
                }
            }
        }
    } else {
        const int n = ntiles * 128;  // words
        for (int base = 0; base < n; base += BATCH * NT) {
            uint32_t wv[BATCH];
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int i = base + u * NT + (int)threadIdx.x;
                if (i < n) {
                    const uint8_t* b = src + 4 * i;
                    wv[u] = b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) | ((uint32_t)b[3] << 24);
                }
            }
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int i = base + u * NT + (int)threadIdx.x;
                if (i < n) tile[(i >> 7) * kTileWords + (i & 127)] = wv[u];
            }
        }
    }
}

// One (128-row tile rt, group of column tiles starting at jt0) of a
// swizzled scale buffer -> compact rows.  `tile` is the CTA's staging area.
template <bool VEC_IN, bool WORD_OUT>
__device__ __forceinline__ void unswizzle_group(const ExportArgs& a, int64_t rt, int64_t jt0, uint32_t* tile) {
    const int64_t nb = (a.K + 31) >> 5;
    const int64_t Cp = (nb + 3) & ~int64_t(3);
    const int64_t ct = Cp >> 2;  // column tiles per row tile
    const int g = (int)min((int64_t)kGroup, ct - jt0);
    const int W = (int)min((int64_t)4 * g, nb - 4 * jt0);  // output columns of this group
    stage_tiles<VEC_IN>(a.scales + (rt * ct + jt0) * 512, g, tile);
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

// Swizzled input, compact rows that are not whole words (nb % 4 != 0).
// One CTA per 128-row tile stages the tile's ct * 512 contiguous swizzled
// bytes.  Four consecutive compact rows starting at a multiple of 4 are
// 4 * nb bytes = nb whole aligned words (the tile's output starts on a
// 16-byte boundary), and every such group has the same layout, so a table
// of nb entries -- built once per CTA, one division per entry -- says for
// group word k which row (0..3) and row byte j its first byte is.  Word k
// is then a funnel shift of the staged words of column tiles j/4 and
// j/4 + 1 of that row, or, where it runs into the next row (three words
// per group), the row's last bytes (which may also straddle two column
// tiles) merged with the next row's first word.
// Consecutive lanes take consecutive words: consecutive column tiles of
// one row (distinct banks with the one-word pad), consecutive addresses.
// (gbase[e >> 20] is the next row's column tile 0.)
// Rows past the last whole group (only in the last tile) are byte stores;
// so is everything when the output is not word aligned (VW == 1).
constexpr int kFlatThreads = 256;

template <int VW>
__global__ void __launch_bounds__(kFlatThreads) unswizzle_flat_kernel(ExportArgs a, int64_t tiles_r) {
    constexpr int NW = kFlatThreads / 32;  // warps
    static_assert(NW % 8 == 0, "the group walk below steps by NW / 8 slot words: NW must be a multiple of 8");
    // nb table entries, then ct + 1 staged tiles of kTileWords words (the
    // spare tile lets a word read column tile j/4 + 1 unconditionally; what
    // it holds is shifted or masked away)
    extern __shared__ uint32_t smem[];
    const int nb = (int)((a.K + 31) >> 5);
    const int ct = (nb + 3) >> 2;
    uint32_t* table = smem;
    uint32_t* stile = smem + ((nb + 3) & ~3);
    // Entry k: offset of the first byte's staged word from the group's row-0
    // slot (4 r + (j/4) * kTileWords: rows 4G + r share the slot base of row
    // 4G, as 4G + r never carries past bit 4), the byte shift j % 4, and for
    // a word that crosses into the next row its c bytes left in the row and
    // the next row's slot offset 4 (r + 1).
    for (int k = threadIdx.x; k < nb; k += kFlatThreads) {
        const int p = 4 * k, r = p / nb, j = p - r * nb;
        const int c = j + 4 > nb ? nb - j : 0;
        table[k] = (uint32_t)(4 * r + (j >> 2) * kTileWords) | ((uint32_t)(j & 3) << 16) | ((uint32_t)c << 18) |
                   ((uint32_t)(4 * (r + 1)) << 20);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t rt = blockIdx.x; rt < tiles_r; rt += gridDim.x) {
        stage_tiles<true, 4, kFlatThreads>(a.scales + rt * ct * 512, ct, stile);
        __syncthreads();
        const int64_t r0 = rt * 128;
        const int nrows = (int)min((int64_t)128, a.rows - r0);
        uint8_t* out = a.out + r0 * nb;
        const int groups = VW == 1 ? 0 : nrows >> 2;
        // lane: words k = lane, lane + 32, ... of every group G = warp + NW i of this
        // warp; group G's row-0 slot is 16 (G % 8) + G / 8 = 16 (warp % 8) + warp / 8
        // + (NW / 8) i, so the inner loop steps NW / 8 words in shared memory and
        // NW nb words in the output.
        uint32_t* const o0 = reinterpret_cast<uint32_t*>(out) + (int64_t)warp * nb;
        const int ng = groups > warp ? (groups - warp + NW - 1) / NW : 0;  // this warp's groups
        const uint32_t* const wbase = stile + 16 * (warp & 7) + (warp >> 3);
        constexpr int ds = NW / 8;
        for (int k = lane; k < nb; k += 32) {
            const uint32_t e = table[k];
            const uint32_t* pa = wbase + (e & 0xFFFFu);
            const int sh = 8 * (int)((e >> 16) & 3u), c = (int)((e >> 18) & 3u);
            uint32_t* ow = o0 + k;
            if (c == 0) {
                for (int i = 0; i < ng; ++i)
                    ow[(int64_t)i * NW * nb] = __funnelshift_r(pa[ds * i], pa[ds * i + kTileWords], sh);
            } else {
                const uint32_t* pb = wbase + (e >> 20);
                const uint32_t m = (1u << (8 * c)) - 1u;
                for (int i = 0; i < ng; ++i)
                    ow[(int64_t)i * NW * nb] =
                        (__funnelshift_r(pa[ds * i], pa[ds * i + kTileWords], sh) & m) | (pb[ds * i] << (8 * c));
            }
        }
        // rows past the last whole group: byte stores
        for (int f = 4 * groups * nb + (int)threadIdx.x; f < nrows * nb; f += kFlatThreads) {
            const int rr = f / nb, j = f - rr * nb;
            out[f] = (uint8_t)(stile[(rr & 31) * 4 + (rr >> 5) + (j >> 2) * kTileWords] >> ((j & 3) * 8));
        }
        __syncthreads();  // the staged tile is rewritten by the next row tile
    }
}

// Largest staging area of the flat kernel (bytes of dynamic shared memory).
constexpr int kFlatSmemMax = 160 * 1024;

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

namespace {
template <int VW>
cudaError_t launch_flat(const ExportArgs& a, int64_t tr, int64_t grid, int64_t smem, cudaStream_t s) {
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(unswizzle_flat_kernel<VW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // the kernel keeps nothing in L1: let shared memory take the whole carveout
    const cudaError_t e = cudaFuncSetAttribute(unswizzle_flat_kernel<VW>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    unswizzle_flat_kernel<VW><<<(unsigned)grid, kFlatThreads, (size_t)smem, s>>>(a, tr);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_export(const ExportArgs& a, cudaStream_t s) {
    const int64_t nb = ceil_div(a.K, 32);
    if (a.lay == 2) {
        const int64_t ct = ceil_div(nb, 4);
        const int64_t tr = ceil_div(a.rows, 128);
        const bool vin = (reinterpret_cast<uintptr_t>(a.scales) & 15) == 0;
        const int64_t smem = (ct + 1) * kTileWords * 4 + ((nb + 3) & ~int64_t(3)) * 4;
        // nb > 4: a word of compact output then meets at most one row boundary
        if (nb % 4 != 0 && nb > 4 && vin && smem <= kFlatSmemMax) {
            int64_t grid = tr;
            const int64_t cap = (int64_t)sm_count() * 16;
            if (grid > cap) grid = cap;
            const uintptr_t o = reinterpret_cast<uintptr_t>(a.out);
            return (o & 3) == 0 ? launch_flat<4>(a, tr, grid, smem, s) : launch_flat<1>(a, tr, grid, smem, s);
        }
        const int64_t gx = ceil_div(ct, kGroup);
        const unsigned gy = (unsigned)(tr < 65535 ? tr : 65535);
        const dim3 grid((unsigned)gx, gy);
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
