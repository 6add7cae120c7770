// mxq_block128.cu -- direct MXFP4 -> FP8 128x128 blockwise conversion.
//
// TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling recipes",
// Description, mode 2 (Direct), "blockwise = per-tile exponent folding":
// T = max(max_b e_b - 6, -127) over the 1x32 blocks of a 128x128 tile, each
// payload RTNE_E4M3(p * 2^(e_b - T)) with subnormals, no device-side assert.
//
// One CTA per tile; the tile is read from HBM once.  A tile is 512 blocks of
// 1x32; each lane owns whole blocks (2 per lane for bf16 with 256 threads, 1
// for fp32 with 512), read as 32-byte vectors and kept in registers (32 per
// lane): pass 1 takes the block exponents, the tile maximum is one warp
// redux plus a pass through shared memory, and pass 2 encodes the held
// blocks and writes 32 payload bytes per block.  (Re-reading the tile from
// L1 in pass 2 instead, with no tile data across the barrier, measured
// 33.6 us for bf16 and 81 us for fp32 on 8192 x 8192, against 31.8 and
// 68 us holding.)  fp32 with aligned rows runs block128_pipe_kernel below.
#include <cuda_runtime.h>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kNoBlock = -100000;

template <Elt ELT>
struct T128;
template <>
struct T128<Elt::BF16> {
    static constexpr int NT = 256, BPL = 2, SEGS = 2, SEG_ELEMS = 16, ES = 2, MANT = 7, MINB = 4;
};
template <>
struct T128<Elt::FP32> {
    static constexpr int NT = 512, BPL = 1, SEGS = 4, SEG_ELEMS = 8, ES = 4, MANT = 23, MINB = 2;
};

// One block of the tile as SEGS x 8 words (missing elements read as +0).
template <Elt ELT, bool VEC>
__device__ __forceinline__ void load_blk(uint32_t (&v)[T128<ELT>::SEGS][8], const char* p, int valid) {
    using P = T128<ELT>;
#pragma unroll
    for (int s = 0; s < P::SEGS; ++s) {
        if constexpr (VEC) {
            if (s * P::SEG_ELEMS < valid) {
                ld32(v[s], p + 32 * s);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) v[s][k] = 0u;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint32_t w = 0u;
                if constexpr (ELT == Elt::BF16) {
                    const int e0 = s * 16 + 2 * k;
                    if (e0 < valid) w = reinterpret_cast<const uint16_t*>(p)[e0];
                    if (e0 + 1 < valid) w |= (uint32_t)reinterpret_cast<const uint16_t*>(p)[e0 + 1] << 16;
                } else {
                    const int e0 = s * 8 + k;
                    if (e0 < valid) w = reinterpret_cast<const uint32_t*>(p)[e0];
                }
                v[s][k] = w;
            }
        }
    }
}

// Block exponent of one block (e = clamp(ceil(log2(amax / 6)), -126, 125))
// and whether a NaN / Inf poisons it.
template <Elt ELT>
__device__ __forceinline__ int block_exp(const uint32_t (&v)[T128<ELT>::SEGS][8], bool& pois) {
    using P = T128<ELT>;
    uint32_t m = 0u;
    if constexpr (ELT == Elt::BF16) {
#pragma unroll
        for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
            for (int k = 0; k < 8; ++k) m = bf2_absmax(m, v[s][k]);
        m &= 0x7FFF7FFFu;
        m = max(m & 0xFFFFu, m >> 16);
        pois = m >= 0x7F80u;
    } else {
#pragma unroll
        for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
            for (int k = 0; k < 8; ++k) m = f32_absmax(m, v[s][k]);
        m &= 0x7FFFFFFFu;
        pois = m >= 0x7F800000u;
    }
    return block_exponent<P::MANT>(m);
}

// Encode one block of a tile with tile exponent T and store its 32 payload
// bytes at d (valid of them).
template <Elt ELT, int DST>
__device__ __forceinline__ void encode_block(const uint32_t (&v)[T128<ELT>::SEGS][8], int eb, int T, bool pois,
                                             int valid, uint8_t* d) {
    using P = T128<ELT>;
    // RTNE onto E4M3 of p * 2^(e_b - T): the grid value p is exact in
    // bf16/fp32, the power-of-two fold is exact in fp32 (or far below
    // E4M3's smallest subnormal), and cvt rounds once.
    const uint32_t fold = f32_pow2(max(eb - T, -126));
    const bool top = eb == 125;  // only there can |x| / 2^e round past 6
    uint32_t b[8];
    if constexpr (ELT == Elt::BF16) {
        if (T <= 6 && eb - T >= -4) {
            // Every nonzero payload p * 2^(e_b - T) is >= 2^-5, an E4M3
            // normal, so the encode is exact: round onto the grid in the
            // domain z = x * 2^(-T - 120), where the bf16 exponent field of a
            // value equals its E4M3 one and bits 10..4 are the E4M3 byte.
            Bf16Grid g;
            g.mult = bf16_pow2_pair(-T - 120);
            g.floor = bf16_pow2_pair(eb - T - 120);
#pragma unroll
            for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t w0 = v[s][2 * q], w1 = v[s][2 * q + 1];
                    const uint32_t t0 = bf2_grid(w0, g), t1 = bf2_grid(w1, g);
                    b[4 * s + q] = lop_select(prmt(t0 >> 4, t1 >> 4, 0x6420u), prmt(w0, w1, 0x7531u), 0x7F7F7F7Fu);
                }
        } else {
            const Bf16Grid g = bf16_grid_unit(eb);
#pragma unroll
            for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t h[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t w = v[s][2 * q + u];
                        uint32_t t = bf2_grid(w, g);
                        if (top) t = bf2_sat(t, 0x40C040C0u);
                        const uint32_t sg = t | (w & 0x80008000u);
                        h[u] = e4m3x2_from_f32(f32_mul(sg & 0xFFFF0000u, fold), f32_mul(sg << 16, fold));
                    }
                    b[4 * s + q] = h[0] | (h[1] << 16);
                }
        }
    } else if (eb - T >= -5) {
        // every nonzero payload p * 2^(e_b - T) is an exact E4M3 normal: E2M1
        // codes by the hardware conversion, bytes from a table
        const uint32_t mult = f32_pow2(-eb);
        const E4m3Table tab = e4m3_table(eb - T);
#pragma unroll
        for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
            for (int q = 0; q < 2; ++q)
                b[2 * s + q] = e4m3x4_from_grid(v[s][4 * q], v[s][4 * q + 1], v[s][4 * q + 2], v[s][4 * q + 3], mult, tab);
    } else {
        const uint32_t mult = f32_pow2(-eb);
#pragma unroll
        for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t u4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t w = v[s][4 * q + u];
                    uint32_t tt = f32_grid(w, mult);
                    if (top) tt = f32_sat(tt);
                    u4[u] = f32_mul(tt | (w & 0x80000000u), fold);
                }
                b[2 * s + q] = e4m3x2_from_f32(u4[1], u4[0]) | (e4m3x2_from_f32(u4[3], u4[2]) << 16);
            }
    }
    if (pois)
#pragma unroll
        for (int k = 0; k < 8; ++k) b[k] = 0x7F7F7F7Fu;
    if constexpr (DST == 2) {
        st32(d, b);
    } else if constexpr (DST == 1) {
        st16(d, b[0], b[1], b[2], b[3]);
        if (valid > 16) st16(d + 16, b[4], b[5], b[6], b[7]);
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (k < valid) d[k] = (uint8_t)(b[k >> 2] >> ((k & 3) * 8));
    }
}

template <Elt ELT, bool VEC, int DST>
__global__ void __launch_bounds__(T128<ELT>::NT, T128<ELT>::MINB)
    block128_kernel(Block128Args a, int64_t tiles_r, int64_t tiles_c) {
    using P = T128<ELT>;
    __shared__ int warp_max[P::NT / 32];
    const int t = threadIdx.x;
    const int64_t tj = blockIdx.x;
    if (a.skip != nullptr && *a.skip != 0) return;  // skip-update request: write nothing

    for (int64_t ti = blockIdx.y; ti < tiles_r; ti += gridDim.y) {
        int valid[P::BPL];
        int eb[P::BPL];
        bool pois[P::BPL];
        int local = kNoBlock;
        uint32_t held[P::BPL][P::SEGS][8];  // the lane's blocks, kept for pass 2
        // pass 1: block exponents
#pragma unroll
        for (int i = 0; i < P::BPL; ++i) {
            const int q = i * P::NT + t;  // block of the tile: row q/4, column block q%4
            const int64_t row = ti * 128 + (q >> 2), col0 = tj * 128 + (q & 3) * 32;
            valid[i] = row < a.rows ? (int)max((int64_t)0, min((int64_t)32, a.K - col0)) : 0;
            uint32_t v[P::SEGS][8];
            load_blk<ELT, VEC>(v, static_cast<const char*>(a.x) + (row * a.ldx + col0) * P::ES, valid[i]);
            eb[i] = block_exp<ELT>(v, pois[i]);
            if (!pois[i] && valid[i] > 0) local = max(local, eb[i]);
#pragma unroll
            for (int s2 = 0; s2 < P::SEGS; ++s2)
#pragma unroll
                for (int k = 0; k < 8; ++k) held[i][s2][k] = v[s2][k];
        }
        local = __reduce_max_sync(0xffffffffu, local);
        if ((t & 31) == 0) warp_max[t >> 5] = local;
        __syncthreads();
        int emax = kNoBlock;
#pragma unroll
        for (int w = 0; w < P::NT / 32; ++w) emax = max(emax, warp_max[w]);
        __syncthreads();  // warp_max is rewritten by the next tile of this CTA
        if (emax == kNoBlock) emax = -126;
        const int T = max(emax - 6, -127);
        if (t == 0) reinterpret_cast<uint32_t*>(a.tile_scale_inv)[ti * tiles_c + tj] = f32_pow2(T);

        // pass 2: encode
#pragma unroll
        for (int i = 0; i < P::BPL; ++i) {
            if (valid[i] <= 0) continue;
            uint32_t v[P::SEGS][8];
#pragma unroll
            for (int s2 = 0; s2 < P::SEGS; ++s2)
#pragma unroll
                for (int k = 0; k < 8; ++k) v[s2][k] = held[i][s2][k];
            const int q = i * P::NT + t;
            encode_block<ELT, DST>(v, eb[i], T, pois[i], valid[i],
                                   a.data + (ti * 128 + (q >> 2)) * a.K + tj * 128 + (q & 3) * 32);
        }
    }
}

// fp32 weights with 32-byte aligned rows and K % 32 == 0.  An fp32 tile is
// 64 KB and a lane's block 32 registers, so only two 512-thread CTAs fit per
// SM; a CTA that loads a tile and then converts it leaves the link idle
// while it computes.  Here a persistent CTA stages its next tile in shared
// memory by cp.async while it converts the current one from registers: the
// tile is waited for, each lane copies its block into registers, the buffer
// is refilled with the next tile, and the tile maximum and encode follow.
// Chunk c (0..31, 16 bytes) of tile row r sits at r * 32 + (c ^ ((4 (r & 1)
// + c / 8) & 7)): a block's eight chunks stay in its 128 bytes, and the
// eight lanes of a quarter-warp (two rows, four blocks, one chunk each) hit
// eight different 16-byte bank groups.

// Staged layout of a tile: CPR 16-byte chunks per row (16 bf16 / 32 fp32),
// a block's CPB chunks (4 / 8) contiguous; chunk c of row r sits at
// r * CPR + (c ^ x(r, c)) with x = (2 (r & 1) + c / 8) for bf16 and
// (4 (r & 1) + c / 8) & 7 for fp32: the XOR stays inside the block's
// chunks, and the eight lanes of a quarter-warp (two rows, four blocks, one
// chunk each) hit eight different 16-byte bank groups.
template <Elt ELT>
__device__ __forceinline__ int stage_slot(int r, int c) {
    if constexpr (ELT == Elt::BF16)
        return r * 16 + (c ^ (2 * (r & 1) + (c >> 3)));
    else
        return r * 32 + (c ^ ((4 * (r & 1) + (c >> 3)) & 7));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int bytes) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gmem), "r"(bytes) : "memory");
}

template <Elt ELT>
__global__ void __launch_bounds__(T128<ELT>::NT, ELT == Elt::BF16 ? 4 : 2)
    block128_pipe_kernel(Block128Args a, int64_t tiles_r, int64_t tiles_c) {
    using P = T128<ELT>;
    constexpr int CPR = 128 * P::ES / 16, CPB = CPR / 4;  // chunks per row / per block
    extern __shared__ __align__(16) uint4 stile[];           // 128 rows x CPR chunks
    __shared__ int warp_max[P::NT / 32];
    const int t = threadIdx.x;
    if (a.skip != nullptr && *a.skip != 0) return;  // skip-update request: write nothing
    const int64_t ntiles = tiles_r * tiles_c;
    // The thread's chunks of any tile: row r0 + RPM m, chunk column c (m = 0 ..
    // NCH - 1); RPM is even, so the slot's XOR term is the same for every m and
    // the slot steps by RPM * CPR.  Whole tiles copy without bounds checks.
    constexpr int NCH = 128 * CPR / P::NT, RPM = P::NT / CPR;
    static_assert(RPM % 2 == 0, "the XOR term of stage_slot must not depend on m");
    const int r0 = t / CPR, c = t % CPR;
    const int slot0 = stage_slot<ELT>(r0, c);
    const int64_t rel0 = (int64_t)r0 * a.ldx + c * (16 / P::ES), relm = (int64_t)RPM * a.ldx;  // elements
    auto stage = [&](int64_t lin) {
        const int64_t ti = lin / tiles_c, tj = lin - ti * tiles_c;
        const char* base = static_cast<const char*>(a.x) + (ti * 128 * a.ldx + tj * 128) * P::ES;
        if (ti * 128 + 128 <= a.rows && tj * 128 + 128 <= a.K) {
#pragma unroll
            for (int m = 0; m < NCH; ++m)
                cp_async16(&stile[slot0 + m * RPM * CPR], base + (rel0 + m * relm) * P::ES, 16);
        } else {
#pragma unroll
            for (int m = 0; m < NCH; ++m) {
                const int64_t row = ti * 128 + r0 + RPM * m, col = tj * 128 + c * (16 / P::ES);
                const bool in = row < a.rows && col < a.K;
                cp_async16(&stile[slot0 + m * RPM * CPR], in ? base + (rel0 + m * relm) * P::ES : base, in ? 16 : 0);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    int64_t lin = blockIdx.x;
    if (lin < ntiles) stage(lin);
    for (; lin < ntiles; lin += gridDim.x) {
        const int64_t ti = lin / tiles_c, tj = lin - ti * tiles_c;
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        uint32_t v[P::BPL][P::SEGS][8];
#pragma unroll
        for (int i = 0; i < P::BPL; ++i) {
            const int q = i * P::NT + t, r = q >> 2, j = q & 3;  // block q: tile row r, column block j
#pragma unroll
            for (int k = 0; k < CPB; ++k) {
                const uint4 c = stile[stage_slot<ELT>(r, CPB * j + k)];
                uint32_t* d = &v[i][k >> 1][(k & 1) * 4];
                d[0] = c.x;
                d[1] = c.y;
                d[2] = c.z;
                d[3] = c.w;
            }
        }
        __syncthreads();  // every lane has its blocks: the buffer takes the next tile
        if (lin + gridDim.x < ntiles) stage(lin + gridDim.x);
        int eb[P::BPL], valid[P::BPL];
        bool pois[P::BPL];
        int local = kNoBlock;
#pragma unroll
        for (int i = 0; i < P::BPL; ++i) {
            const int q = i * P::NT + t;
            const int64_t row = ti * 128 + (q >> 2), col0 = tj * 128 + (q & 3) * 32;
            valid[i] = row < a.rows && col0 < a.K ? 32 : 0;  // K % 32 == 0: whole blocks
            eb[i] = block_exp<ELT>(v[i], pois[i]);
            if (!pois[i] && valid[i] > 0) local = max(local, eb[i]);
        }
        local = __reduce_max_sync(0xffffffffu, local);
        if ((t & 31) == 0) warp_max[t >> 5] = local;
        __syncthreads();
        int emax = kNoBlock;
#pragma unroll
        for (int w = 0; w < P::NT / 32; ++w) emax = max(emax, warp_max[w]);
        if (emax == kNoBlock) emax = -126;
        const int T = max(emax - 6, -127);
        if (t == 0) reinterpret_cast<uint32_t*>(a.tile_scale_inv)[ti * tiles_c + tj] = f32_pow2(T);
#pragma unroll
        for (int i = 0; i < P::BPL; ++i) {
            const int q = i * P::NT + t;
            if (valid[i] > 0)
                encode_block<ELT, 2>(v[i], eb[i], T, pois[i], valid[i],
                                     a.data + (ti * 128 + (q >> 2)) * a.K + tj * 128 + (q & 3) * 32);
        }
    }
}

template <Elt ELT, bool VEC, int DST>
cudaError_t launch_one(const Block128Args& a, cudaStream_t s) {
    const int64_t tr = ceil_div(a.rows, 128), tc = ceil_div(a.K, 128);
    if (tc > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const unsigned gy = (unsigned)(tr < 65535 ? tr : 65535);
    block128_kernel<ELT, VEC, DST><<<dim3((unsigned)tc, gy), T128<ELT>::NT, 0, s>>>(a, tr, tc);
    return cudaGetLastError();
}

bool aligned(const void* p, int64_t n) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)n) == 0; }

template <Elt ELT>
cudaError_t dispatch(const Block128Args& a, cudaStream_t s) {
    using P = T128<ELT>;
    const bool vec = aligned(a.x, 32) && (a.ldx * P::ES) % 32 == 0 && (a.K * P::ES) % 32 == 0;
    const int dst = (aligned(a.data, 32) && a.K % 32 == 0) ? 2 : (aligned(a.data, 16) && a.K % 16 == 0) ? 1 : 0;
    if (!vec) return launch_one<ELT, false, 0>(a, s);
    // fp32: the pipelined kernel (57 us on 8192 x 8192 against 58 us without the
    // staging); bf16 keeps its blocks in registers across the tile-max barrier
    // in block128_kernel (31.6 us against 34.8 us pipelined)
    if (ELT == Elt::FP32 && dst == 2) {
        const int64_t tr = ceil_div(a.rows, 128), tc = ceil_div(a.K, 128);
        const int bytes = 128 * 128 * P::ES;
        // per call: the attribute belongs to the current device
        const cudaError_t e =
            cudaFuncSetAttribute(block128_pipe_kernel<ELT>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        int64_t grid = tr * tc;
        const int64_t cap = (int64_t)sm_count() * (ELT == Elt::BF16 ? 4 : 2);  // CTAs resident per SM
        if (grid > cap) grid = cap;
        block128_pipe_kernel<ELT><<<(unsigned)grid, P::NT, bytes, s>>>(a, tr, tc);
        return cudaGetLastError();
    }
    if (dst == 2) return launch_one<ELT, true, 2>(a, s);
    if (dst == 1) return launch_one<ELT, true, 1>(a, s);
    return launch_one<ELT, true, 0>(a, s);
}

}  // namespace

cudaError_t launch_block128(Elt elt, const Block128Args& a, cudaStream_t s) {
    return elt == Elt::BF16 ? dispatch<Elt::BF16>(a, s) : dispatch<Elt::FP32>(a, s);
}

}  // namespace mxq
