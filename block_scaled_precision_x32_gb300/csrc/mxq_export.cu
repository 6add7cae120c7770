// mxq_export.cu -- the copy behind export_components(): compact
// (rows, ceil(K/32)) UE8M0 scales out of a padded or GEMM-swizzled buffer.
//
// TE PR #3790 "MXFP8TensorStorage.export_components()", Description:
// scales are copied only when padded in the last dimension or swizzled for
// GEMM, padding dropped and the swizzle undone.
//
// Swizzled input, nb >= 16, scales and output 16-byte aligned (the usual
// case: every GEMM-swizzled weight with K >= 512): the chunk kernel below,
// which needs no shared memory -- each lane turns 16-byte loads of four rows'
// scales into aligned 16-byte chunks of those rows' compact output -- or,
// for large exports (bulk_wins), the bulk kernel, which stages whole row
// tiles in shared memory by bulk copies so that global memory sees only
// whole-tile reads and contiguous writes.
// Other swizzled input: one CTA per (128-row tile, group of 16 column
// tiles).  The group's bytes are contiguous in the swizzled buffer (16 x 512),
// so they are staged in shared memory with 16-byte loads -- each 512-byte tile
// padded by one word so that lanes reading the same word of consecutive
// tiles hit distinct banks -- and written out row by row, consecutive lanes
// on consecutive output words (4 scales) or bytes.  With nb % 4 != 0 and an
// output that is not 16-byte aligned: one CTA per 128-row tile stages all of
// the tile's column tiles and writes its compact output -- one contiguous
// range -- as aligned words.
// Padded input: one warp per row, lanes on consecutive bytes.
// Grouped export: up to kGroupedMax storages per launch, their descriptors
// passed by value in the kernel parameters; chunk-path storages run the bulk
// or the chunk kernel's code, the others a byte copy; every storage's row
// tiles are walked with a grid stride.
#include <cuda_runtime.h>

#include <algorithm>

#include "mxq_device.cuh"
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

// Swizzled input and compact output both 16-byte aligned, nb >= 16 (any
// nb % 4): no shared memory.  In the swizzled layout the 16 bytes at
// (column tile jt, q) -- offset 512 jt + 16 q of a row tile -- are the
// scales of rows q, q + 32, q + 64, q + 96 at columns 4 jt .. 4 jt + 3, one
// word per row; lane q of a warp owns those four rows, so every 16-byte load
// feeds four rows.  Compact row r starts at byte r nb and the four rows of a
// lane start at the same offset mod 16 (32 nb is a multiple of 16), so with
// b = (-q nb) mod 16 chunk i of each row -- row bytes [b + 16 i, b + 16 i + 16)
// -- is one aligned 16-byte store: the words of column tiles
// 4 i + b / 4 .. 4 i + b / 4 + 4, funnel-shifted by b % 4 bytes.  A row's first
// b bytes close the previous row's last chunk, which takes them from the
// first 16 bytes of its next row (column tiles 0..3 of lane q + 1; a lane
// q = 31 row ends on a 16-byte boundary, as does every row tile).  Since
// nb >= 16 a chunk spans at most two rows.  A warp takes CPW consecutive
// chunks of every row of its lane (chunk group cg); the next chunk's four
// loads are issued before the current chunk is stored.  Only the last row of
// a tensor whose compact end is not 16-byte aligned stores bytes.
__device__ __forceinline__ uint32_t word_of(const uint4& v, int s) {
    return s == 0 ? v.x : s == 1 ? v.y : s == 2 ? v.z : v.w;
}

// Bytes [0, e) of o followed by bytes [0, 16 - e) of h, e in 1..15.
__device__ __forceinline__ void merge_next_row(uint32_t (&o)[4], const uint32_t (&h)[4], int e) {
    const int ea = e >> 2, ec = 8 * (e & 3);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int k = t - ea;  // h word holding byte 4 t - e + 3
        const uint32_t hi = k == 0 ? h[0] : k == 1 ? h[1] : k == 2 ? h[2] : k == 3 ? h[3] : 0u;
        const uint32_t lo = k == 1 ? h[0] : k == 2 ? h[1] : k == 3 ? h[2] : 0u;
        const uint32_t hs = __funnelshift_l(lo, hi, ec);  // bytes 4 t - e .. 4 t - e + 3 of h
        const int keep = min(max(e - 4 * t, 0), 4);       // bytes of this word still from o
        const uint32_t m = keep == 4 ? 0xFFFFFFFFu : (1u << (8 * keep)) - 1u;
        o[t] = (o[t] & m) | (hs & ~m);
    }
}

constexpr int kChunkThreads = 128;

// Chunk group cg (chunks CPW cg .. CPW cg + CPW - 1) of row tile rt, whose
// ct * 512 swizzled bytes start at `tile`.
template <int CPW>
__device__ __forceinline__ void unswizzle_chunks(const ExportArgs& a, int64_t rt, int cg, const uint8_t* tile) {
    const int64_t nb = (a.K + 31) >> 5, ct = (nb + 3) >> 2;
    const int q = threadIdx.x & 31;
    const int n16 = (int)(nb & 15);
    const int b = (16 - ((q * n16) & 15)) & 15;
    const int ab = b >> 2, sh = 8 * (b & 3);
    const int e = 16 - ((16 - (((q + 1) * n16) & 15)) & 15);  // bytes of the last chunk inside the row
    const int64_t ilast = (nb - 1 - b) >> 4;                     // last chunk of each of the lane's rows
    const int64_t i0 = (int64_t)cg * CPW;
    const uint8_t* src = tile + 16 * q;
    const int64_t r0 = rt * 128;
    const int nrows = (int)min((int64_t)128, a.rows - r0);
    auto tile_at = [&](int64_t jt) -> uint4 {
        return jt < ct ? *reinterpret_cast<const uint4*>(src + jt * 512) : make_uint4(0u, 0u, 0u, 0u);
    };
    uint4 w[5];
#pragma unroll
    for (int t = 0; t < 5; ++t) w[t] = tile_at(4 * i0 + ab + t);
#pragma unroll
    for (int c = 0; c < CPW; ++c) {
        const int64_t i = i0 + c;
        if (i > ilast) break;
        uint4 nw[4];
        if (c + 1 < CPW) {
#pragma unroll
            for (int t = 0; t < 4; ++t) nw[t] = tile_at(4 * (i + 1) + ab + 1 + t);
        }
        const bool cross = i == ilast && e < 16;
        uint4 h[4];
        if (cross) {  // the next rows' first 16 bytes: column tiles 0..3 of lane q + 1 (q < 31 here)
#pragma unroll
            for (int t = 0; t < 4; ++t) h[t] = *reinterpret_cast<const uint4*>(src + t * 512 + 16);
        }
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const int rr = q + 32 * s;
            if (rr >= nrows) break;
            uint32_t o[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) o[t] = __funnelshift_r(word_of(w[t], s), word_of(w[t + 1], s), sh);
            uint8_t* dst = a.out + (r0 + rr) * nb + b + 16 * i;
            if (cross) {
                const uint32_t hw[4] = {word_of(h[0], s), word_of(h[1], s), word_of(h[2], s), word_of(h[3], s)};
                merge_next_row(o, hw, e);
                if (rr + 1 >= nrows) {  // the tensor's last row: its chunk stops at the end of the output
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (k < e) dst[k] = (uint8_t)(o[k >> 2] >> (8 * (k & 3)));
                    continue;
                }
            }
            st16(dst, o[0], o[1], o[2], o[3]);
        }
        if (c + 1 < CPW) {
            w[0] = w[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) w[t + 1] = nw[t];
        }
    }
}

template <int CPW>
__global__ void __launch_bounds__(kChunkThreads) unswizzle_chunk_kernel(ExportArgs a, int64_t tiles_r, int ngroups) {
    const int cg = (int)blockIdx.y * (kChunkThreads / 32) + (int)(threadIdx.x >> 5);
    if (cg >= ngroups) return;
    const int64_t ct = (((a.K + 31) >> 5) + 3) >> 2;
    for (int64_t rt = blockIdx.x; rt < tiles_r; rt += gridDim.x)
        unswizzle_chunks<CPW>(a, rt, cg, a.scales + rt * ct * 512);
}

// Swizzled input with many row tiles (nb >= 16, 16-byte aligned scales and
// output): the bulk kernel.  A CTA stages one 128-row tile: one thread copies
// the tile's ct * 512 swizzled bytes -- contiguous -- into shared memory with
// one bulk copy (cp.async.bulk, completed on an mbarrier); the CTA turns them
// into the tile's compact rows with the chunk kernel's arithmetic (16-byte
// shared loads of four rows' words, funnel shifts, 16-byte shared stores) in
// two parts of 64 rows, and one thread writes each part -- 64 nb contiguous
// bytes of the output, 16-byte aligned -- with one bulk store.  Global memory
// sees whole-tile reads and contiguous writes, in place of the chunk
// kernel's 16-byte stores to 32 different rows per warp instruction.
// With kBulkThreads a multiple of 32 a thread always holds the same lane q,
// so everything that depends on q alone is computed once per kernel (3.4 M
// warp instructions on the MoE stack against 4.7 M recomputing it per
// chunk).  Measured on the 32 x 4096 x 7184 MoE stack with inputs larger
// than L2: one CTA of 128 threads per row tile, five resident per SM, 12.8 us
// against 13.4 us for the chunk kernel; the whole tile staged as one part
// (three CTAs per SM) 15.7 us, four 32-row parts (six per SM) 15.1 us, and
// persistent CTAs with two or three tiles' copies in flight 15.5-18.3 us.
// The mbarrier wait is bounded (about a second of SM clocks): a tile whose
// copy has not landed by then is written as 0xFF bytes (the E8M0 NaN code),
// the copy is waited for once more, bounded again, and the CTA stops.
constexpr int kBulkThreads = 128;
static_assert(kBulkThreads % 32 == 0, "a thread keeps one lane q for every tile");

// Shared memory of the bulk kernel: the mbarrier (padded to 128 bytes), the
// swizzled tile -- ROT: and 2 KB past it, so that a row's last chunk reads
// up to four column tiles beyond the tile without a test (those bytes are
// shifted or merged away) -- and one 64-row part of compact output with 16
// spare bytes (the part's last chunk may run up to 15 bytes past it).
// Unrotated, the last chunk tests its column tiles instead: the 2 KB would
// cost the MoE stack's nb = 225 its fifth CTA per SM (13.05 against 12.8 us);
// rotated, lanes reach their last chunk in different steps and the test
// diverges (13.4 against 12.7 us at nb = 256, four CTAs per SM either way).
int64_t bulk_smem_bytes(int64_t nb, bool rot) {
    return 128 + ((nb + 3) >> 2) * 512 + (rot ? 2048 : 0) + ((64 * nb + 15) & ~int64_t(15)) + 16;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Wait for phase `parity` of the mbarrier at `mbar` to complete; false after about 2^31 SM clocks.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t mbar, uint32_t parity) {
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(done)
                     : "r"(mbar), "r"(parity)
                     : "memory");
        if (done) return true;
        if (clock64() - t0 > (1ll << 31)) return false;
    }
}

// What a thread's lane q fixes: row q of each row group s (rows q + 32 s)
// starts its compact output b bytes before a 16-byte boundary's chunk 0,
// ends in chunk ilast with e bytes of it inside the row (e < 16: the chunk
// closes the row with the next row's first 16 - e bytes), and its chunk i
// reads column tiles 4 i + b / 4 .. 4 i + b / 4 + 4 of the tile.
struct BulkLane {
    int q, b, sh, ilast, e, rot;
    int src;  // byte offset in the staged tile of chunk 0's first word: 512 (b / 4) + 16 q
    int dst;  // byte offset in a staged part of row q's chunk 0: q nb + b
};

__device__ __forceinline__ BulkLane bulk_lane(int nb) {
    BulkLane L;
    const int n16 = nb & 15;
    L.q = threadIdx.x & 31;
    L.b = (16 - ((L.q * n16) & 15)) & 15;
    L.sh = 8 * (L.b & 3);
    L.ilast = (nb - 1 - L.b) >> 4;
    L.e = 16 - ((16 - (((L.q + 1) * n16) & 15)) & 15);
    L.rot = (L.q - ((L.q * nb + 15) >> 4)) & 7;
    L.src = 512 * (L.b >> 2) + 16 * L.q;
    L.dst = L.q * nb + L.b;
    return L;
}

// Chunk i of row group S of the staged words w (lane q) -> the part staged at `ob`.
template <int S>
__device__ __forceinline__ void bulk_chunk(const uint4 (&w)[5], const uint4* h, int e, int sh, uint8_t* dst) {
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) o[t] = __funnelshift_r(word_of(w[t], S), word_of(w[t + 1], S), sh);
    if (h != nullptr) {
        const uint32_t hw[4] = {word_of(h[0], S), word_of(h[1], S), word_of(h[2], S), word_of(h[3], S)};
        merge_next_row(o, hw, e);
    }
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
}

// Chunk indices 0..N-1 (ilast <= N - 1).  A 16-byte shared access is served
// eight lanes at a time, conflict-free when the eight hit distinct 16-byte
// units mod 8.  Lane q's loads sit at unit 32 jt + q (distinct for eight
// consecutive q); its row's chunk i at unit ceil((q + 32 s) nb / 16) + i,
// which for one i can collide across q: 2-way at most for most nb (225,
// 240), 8-way for nb = 256.  ROT (chosen by the host where a store would
// collide 4-way or worse): lane q takes chunk (i' + rot_q) mod N in step i',
// rot_q = (q - ceil(q nb / 16)) mod 8, so that its unit is q + i' + 2 s nb
// mod 8 -- distinct again, up to the wrap at N.  Rotated, the chunks that
// close a row with the next row's first bytes would fall in different steps
// for different lanes, and their merge is long, so they take a step of
// their own after the others; unrotated, they are the last step's chunks.
template <bool ROT>
__device__ bool bulk_tile(const ExportArgs& a, int64_t rt, uint8_t* in, uint8_t* ob, uint32_t mb, uint32_t parity,
                          const BulkLane& L, int* ok) {
    const int nb = (int)((a.K + 31) >> 5), ct = (nb + 3) >> 2;
    const int64_t r0 = rt * 128;
    const int nrows = (int)min((int64_t)128, a.rows - r0);
    if (threadIdx.x == 0) {
        const int in_bytes = ct * 512;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(in_bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(smem_addr(in)), "l"(a.scales + rt * in_bytes), "r"(in_bytes), "r"(mb)
                     : "memory");
        *ok = mbar_wait_bounded(mb, parity) ? 1 : 0;
    }
    __syncthreads();
    if (!*ok) {
        for (int64_t k = threadIdx.x; k < (int64_t)nrows * nb; k += kBulkThreads) a.out[r0 * nb + k] = 0xFF;
        if (threadIdx.x == 0) mbar_wait_bounded(mb, parity);  // the copy in flight, if it still lands
        return false;
    }
    // every thread observes the completed phase itself (acquire) before reading the tile
    asm volatile("{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%0], %1; }" ::"r"(mb), "r"(parity)
                 : "memory");
    const int N = ((nb - 1) >> 4) + 1;
    const int steps = N + (ROT && (nb & 15) != 0 ? 1 : 0);
    const bool has_cross = L.e < 16;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        const int pr0 = 64 * part;  // rows q + 32 s, s = 2 part, 2 part + 1
        if (pr0 >= nrows) break;
        if (pr0 + L.q < nrows) {
            const bool second = pr0 + 32 + L.q < nrows;
            for (int ip = threadIdx.x >> 5; ip < steps; ip += kBulkThreads / 32) {
                int i;
                bool cross;
                if constexpr (ROT) {
                    if (ip >= N) {
                        if (!has_cross) continue;
                        i = L.ilast;
                        cross = true;
                    } else {
                        i = ip + L.rot;
                        if (i >= N) i = i - N < N ? i - N : i % N;
                        if (i > L.ilast - (has_cross ? 1 : 0)) continue;
                        cross = false;
                    }
                } else {
                    i = ip;
                    if (i > L.ilast) continue;
                    cross = has_cross && i == L.ilast;
                }
                const uint8_t* src = in + L.src + 2048 * i;
                uint4 w[5];
                if (ROT || i < L.ilast) {  // column tiles 4 i + b / 4 + 4 <= ct - 1, or within the 2 KB past them
#pragma unroll
                    for (int t = 0; t < 5; ++t) w[t] = *reinterpret_cast<const uint4*>(src + 512 * t);
                } else {  // the row's last chunk: column tiles past the tile hold only bytes past the row
                    const int jt0 = 4 * i + (L.b >> 2);
#pragma unroll
                    for (int t = 0; t < 5; ++t)
                        w[t] = jt0 + t < ct ? *reinterpret_cast<const uint4*>(src + 512 * t) : make_uint4(0u, 0u, 0u, 0u);
                }
                uint4 h[4];
                if (cross) {  // the next rows' first 16 bytes: column tiles 0..3 of lane q + 1 (q < 31)
#pragma unroll
                    for (int t = 0; t < 4; ++t) h[t] = *reinterpret_cast<const uint4*>(in + 16 * (L.q + 1) + 512 * t);
                }
                uint8_t* dst = ob + L.dst + 16 * i;
                if (part == 0) {
                    bulk_chunk<0>(w, cross ? h : nullptr, L.e, L.sh, dst);
                    if (second) bulk_chunk<1>(w, cross ? h : nullptr, L.e, L.sh, dst + 32 * nb);
                } else {
                    bulk_chunk<2>(w, cross ? h : nullptr, L.e, L.sh, dst);
                    if (second) bulk_chunk<3>(w, cross ? h : nullptr, L.e, L.sh, dst + 32 * nb);
                }
            }
        }
        // the part's bytes (and, after the last part, the tile's reads) are done: hand them to the copy engine
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        const int tot = (min(nrows, pr0 + 64) - pr0) * nb, main16 = tot & ~15;
        uint8_t* gout = a.out + (r0 + pr0) * nb;
        if (threadIdx.x == 0 && main16 > 0) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gout), "r"(smem_addr(ob)),
                         "r"(main16)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        for (int k = main16 + threadIdx.x; k < tot; k += kBulkThreads) gout[k] = ob[k];  // the tensor's last bytes
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncthreads();  // the output part is rewritten next
    }
    return true;
}

// A CTA's row tiles rt0, rt0 + stride, ... (one, when the grid has a CTA per
// tile), each through the same buffers and alternating mbarrier phases.
template <bool ROT>
__device__ void bulk_walk(const ExportArgs& a, int64_t tiles_r, int64_t rt0, int64_t stride, uint8_t* sm, int* ok) {
    const int nb = (int)((a.K + 31) >> 5);
    uint8_t* in = sm + 128;
    uint8_t* ob = in + ((nb + 3) >> 2) * 512 + (ROT ? 2048 : 0);
    const uint32_t mb = smem_addr(sm);
    const BulkLane L = bulk_lane(nb);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mb) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    uint32_t parity = 0;
    for (int64_t rt = rt0; rt < tiles_r; rt += stride, parity ^= 1u)
        if (!bulk_tile<ROT>(a, rt, in, ob, mb, parity, L, ok)) return;
    if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <bool ROT>
__global__ void __launch_bounds__(kBulkThreads) bulk_export_kernel(ExportArgs a, int64_t tiles_r) {
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ int ok;
    bulk_walk<ROT>(a, tiles_r, blockIdx.x, gridDim.x, sm, &ok);
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

// Many storages in one launch: blockIdx.z picks the storage, blockIdx.x
// walks its 128-row tiles (grid stride, so any number of them), blockIdx.y
// its chunk groups.  The host sets each storage's path: 2 and 3 (bulk,
// unrotated and rotated: the launch's chunk-eligible storages hold many row
// tiles in total) and 1
// (chunk: swizzled, nb >= 16, 16-byte aligned scales and output) run the
// single export's code -- the bulk path in the blockIdx.y == 0 CTAs, with
// the launch's dynamic shared memory; any other swizzled or padded storage
// is copied byte by byte by the blockIdx.y == 0 CTAs.
static_assert(kChunkThreads == kBulkThreads, "the grouped kernel runs both paths with one block size");

template <int CPW>
__global__ void __launch_bounds__(kChunkThreads) grouped_export_kernel(GroupedExport b) {
    extern __shared__ __align__(128) uint8_t sm[];  // bulk path only
    __shared__ int ok;
    const ExportArgs& a = b.item[blockIdx.z];
    const int64_t nb = (a.K + 31) >> 5, Cp = (nb + 3) & ~int64_t(3);
    const int64_t tr = (a.rows + 127) >> 7;
    if (a.path >= 2) {
        if (blockIdx.y != 0) return;
        if (a.path == 3)
            bulk_walk<true>(a, tr, blockIdx.x, gridDim.x, sm, &ok);
        else
            bulk_walk<false>(a, tr, blockIdx.x, gridDim.x, sm, &ok);
        return;
    }
    if (a.path == 1) {
        const int64_t ngroups = ((nb + 15) / 16 + CPW - 1) / CPW;
        const int64_t cg = (int64_t)blockIdx.y * (kChunkThreads / 32) + (threadIdx.x >> 5);
        if (cg >= ngroups) return;
        const int64_t ct = Cp >> 2;
        for (int64_t rt = blockIdx.x; rt < tr; rt += gridDim.x)
            unswizzle_chunks<CPW>(a, rt, (int)cg, a.scales + rt * ct * 512);
        return;
    }
    if (blockIdx.y != 0) return;
    for (int64_t rt = blockIdx.x; rt < tr; rt += gridDim.x) {
        const int64_t r0 = rt * 128, n = min((int64_t)128, a.rows - r0) * nb;
        for (int64_t f = threadIdx.x; f < n; f += kChunkThreads) {
            const int64_t r = r0 + f / nb, j = f % nb;
            const int64_t off = a.lay == 2 ? ((r >> 7) * (Cp >> 2) + (j >> 2)) * 512 + (r & 31) * 16 +
                                                 ((r >> 5) & 3) * 4 + (j & 3)
                                           : r * Cp + j;
            a.out[r * nb + j] = a.scales[off];
        }
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

// The chunk path of a swizzled export: nb >= 16 and 16-byte aligned
// scales and output.  Chunks per warp (CPW), measured on GB300: 2 for small
// exports (up to 8 such warps per SM; 8192 x 8192: 2.3 us against 2.6 us at
// 1), else 1 (the 32 x 4096 x 7184 MoE stack: 13.6 us against 14.4 us at 2
// and 14.2 us at 4 or 8; that stack now takes the bulk kernel).  Also
// measured and dropped: 32-byte chunks (whole sector stores; 150+ registers,
// 20.9 us against 16.9 us for that build's 16-byte chunks), row tiles staged
// through a ring of shared-memory stages by cp.async (barrier-bound, 24 us)
// and persistent warps with the next unit's loads in flight (13.44 us, no
// gain).
struct ChunkPlan {
    bool ok;
    int cpw;
    int64_t nc;  // 16-byte chunks per compact row, at most
};

static ChunkPlan chunk_plan(const ExportArgs& a) {
    ChunkPlan p{false, 1, 0};
    const int64_t nb = ceil_div(a.K, 32);
    if (a.lay != 2 || nb < 16 || (reinterpret_cast<uintptr_t>(a.scales) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(a.out) & 15) != 0)
        return p;
    p.nc = ceil_div(nb, 16);
    if (ceil_div(p.nc, kChunkThreads / 32) > 65535) return p;  // grid y holds the chunk groups
    p.ok = true;
    p.cpw = ceil_div(a.rows, 128) * p.nc <= (int64_t)sm_count() * 8 ? 2 : 1;
    return p;
}

template <int CPW>
static cudaError_t launch_chunks(const ExportArgs& a, int64_t tr, int64_t nc, cudaStream_t s) {
    const int64_t ngroups = ceil_div(nc, CPW);
    const int64_t gy = ceil_div(ngroups, kChunkThreads / 32);
    const int64_t gx = tr < 65535 ? tr : 65535;
    unswizzle_chunk_kernel<CPW><<<dim3((unsigned)gx, (unsigned)gy), kChunkThreads, 0, s>>>(a, tr, (int)ngroups);
    return cudaGetLastError();
}

// The bulk kernel's staging must fit kBulkSmemMax (two CTAs per SM at
// least; K up to 17,000 or so).
constexpr int64_t kBulkSmemMax = 100 * 1024;


// Rotate the bulk kernel's chunks (ROT) when, unrotated, the 16-byte shared
// stores of eight consecutive lanes q would hit one unit 4 or more times:
// unit ceil(q nb / 16) mod 8 (nb = 64, 128, 192, 256, 257, 320, 512, ...).
static bool bulk_rotate(int64_t nb) {
    int worst = 1;
    for (int g = 0; g < 4; ++g) {
        int cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int j = 0; j < 8; ++j) ++cnt[(((8 * g + j) * nb + 15) >> 4) & 7];
        for (int u = 0; u < 8; ++u) worst = std::max(worst, cnt[u]);
    }
    return worst >= 4;
}

static bool bulk_fits(int64_t nb) { return bulk_smem_bytes(nb, bulk_rotate(nb)) <= kBulkSmemMax; }

// Whether the bulk kernel beats the chunk kernel on `tiles` row tiles of nb
// scale columns.  Few row tiles leave most SMs idle in the bulk kernel (one
// CTA per tile).  Measured on GB300 with inputs larger than L2, bulk against
// chunk: nb = 256 (rotated) 6.55 / 6.69 us at 304 tiles, 11.16 / 12.46 us at
// 768, but 5.22 / 3.92 us at 152; nb = 225 and 240 (unrotated) even at 768
// tiles (11.02 / 11.02 and 10.23 / 10.40 us), ahead at 1024 (12.8 / 13.4 us
// for the MoE stack), behind at 512; nb = 100 behind up to 768 tiles.
static bool bulk_wins(int64_t nb, int64_t tiles) {
    if (!bulk_fits(nb)) return false;
    return bulk_rotate(nb) ? tiles >= 304 : nb >= 192 && tiles >= 768;
}

// Dynamic shared memory above the 48 KB default, and the carveout: all of
// it for shared memory when the launch stages tiles (five CTAs of the MoE
// stack's 43.6 KB per SM), the default otherwise (the chunk kernel's loads
// go through L1).  Both are per-kernel settings, so every launch sets them.
template <typename F>
static cudaError_t allow_smem(F* kernel, int64_t smem) {
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                smem > 0 ? (int)cudaSharedmemCarveoutMaxShared : (int)cudaSharedmemCarveoutDefault);
}

template <bool ROT>
static cudaError_t launch_bulk(const ExportArgs& a, int64_t tr, cudaStream_t s) {
    const int64_t smem = bulk_smem_bytes(ceil_div(a.K, 32), ROT);
    const cudaError_t e = allow_smem(bulk_export_kernel<ROT>, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = tr < (int64_t(1) << 24) ? tr : (int64_t(1) << 24);  // one CTA per row tile
    bulk_export_kernel<ROT><<<(unsigned)grid, kBulkThreads, (size_t)smem, s>>>(a, tr);
    return cudaGetLastError();
}

cudaError_t launch_export(const ExportArgs& a, cudaStream_t s) {
    const int64_t nb = ceil_div(a.K, 32);
    if (a.lay == 2) {
        const int64_t ct = ceil_div(nb, 4);
        const int64_t tr = ceil_div(a.rows, 128);
        const bool vin = (reinterpret_cast<uintptr_t>(a.scales) & 15) == 0;
        const ChunkPlan p = chunk_plan(a);
        if (p.ok && bulk_wins(nb, tr))
            return bulk_rotate(nb) ? launch_bulk<true>(a, tr, s) : launch_bulk<false>(a, tr, s);
        if (p.ok) return p.cpw == 1 ? launch_chunks<1>(a, tr, p.nc, s) : launch_chunks<2>(a, tr, p.nc, s);
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

// The grouped kernel runs one CPW for all of its chunk-path storages.
cudaError_t launch_export_grouped(const GroupedExport& b0, cudaStream_t s) {
    if (b0.count <= 0) return cudaSuccess;
    GroupedExport b = b0;
    int64_t gx = 1, gy = 1, warps1 = 0, chunk_tiles = 0, smem = 0;
    for (int i = 0; i < b.count; ++i) {
        ExportArgs& a = b.item[i];
        const ChunkPlan p = chunk_plan(a);
        a.path = p.ok ? 1 : 0;
        gx = std::max(gx, ceil_div(a.rows, 128));
        if (p.ok) chunk_tiles += ceil_div(a.rows, 128);
    }
    // a storage takes the bulk path when the launch's chunk-path storages,
    // one CTA per row tile, fill the GPU as one export of that width would
    for (int i = 0; i < b.count; ++i) {
        ExportArgs& a = b.item[i];
        if (a.path == 1 && bulk_wins(ceil_div(a.K, 32), chunk_tiles)) {
            a.path = bulk_rotate(ceil_div(a.K, 32)) ? 3 : 2;
            smem = std::max(smem, bulk_smem_bytes(ceil_div(a.K, 32), a.path == 3));
        }
        if (a.path == 1) warps1 += ceil_div(a.rows, 128) * chunk_plan(a).nc;
    }
    const int cpw = warps1 <= (int64_t)sm_count() * 8 ? 2 : 1;
    for (int i = 0; i < b.count; ++i) {
        const ExportArgs& a = b.item[i];
        if (a.path == 1) gy = std::max(gy, ceil_div(ceil_div(ceil_div(ceil_div(a.K, 32), 16), cpw), kChunkThreads / 32));
    }
    // every storage's tiles are walked with a grid stride: a cap on gx only
    // bounds the launch, not the sizes it can copy
    const int64_t cap = (int64_t)sm_count() * 64;
    if (gx > cap) gx = cap;
    const dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)b.count);
    cudaError_t e = cpw == 1 ? allow_smem(grouped_export_kernel<1>, smem) : allow_smem(grouped_export_kernel<2>, smem);
    if (e != cudaSuccess) return e;
    if (cpw == 1)
        grouped_export_kernel<1><<<grid, kChunkThreads, (size_t)smem, s>>>(b);
    else
        grouped_export_kernel<2><<<grid, kChunkThreads, (size_t)smem, s>>>(b);
    return cudaGetLastError();
}

}  // namespace mxq
