// mxq_block128.cu -- direct MXFP4 -> FP8 128x128 blockwise conversion.
//
// TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling recipes",
// Description, mode 2 (Direct), "blockwise = per-tile exponent folding":
// T = max(max_b e_b - 6, -127) over the 1x32 blocks of a 128x128 tile, each
// payload RTNE_E4M3(p * 2^(e_b - T)) with subnormals, no device-side assert.
//
// One CTA per tile, the whole tile held in registers: 256 threads x 8
// chunks of 16 bytes (bf16) or 512 x 8 (fp32), a tile row being 16 (bf16)
// or 32 (fp32) consecutive lanes.  Block exponents come from 4- or 8-lane
// shuffles, the tile maximum from one redux per warp plus shared memory;
// the tile is read from HBM exactly once.
#include <cuda_runtime.h>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kChunks = 8;  // chunks per thread
constexpr int kNoBlock = -100000;

template <Elt ELT>
struct T128;
template <>
struct T128<Elt::BF16> {
    static constexpr int NT = 256, CPR = 16, CH = 8, ES = 2, MANT = 7, MINB = 3;
};
template <>
struct T128<Elt::FP32> {
    static constexpr int NT = 512, CPR = 32, CH = 4, ES = 4, MANT = 23, MINB = 1;
};

template <Elt ELT, bool VEC>
__global__ void __launch_bounds__(T128<ELT>::NT, T128<ELT>::MINB) block128_kernel(Block128Args a, int64_t tiles_r, int64_t tiles_c) {
    using P = T128<ELT>;
    __shared__ int warp_max[P::NT / 32];
    const int t = threadIdx.x;
    const int cc = t % P::CPR;  // chunk within the tile row
    const int64_t tj = blockIdx.x;

    for (int64_t ti = blockIdx.y; ti < tiles_r; ti += gridDim.y) {
        const int64_t col0 = tj * 128 + (int64_t)cc * P::CH;
        const int64_t row0 = ti * 128 + t / P::CPR;  // this thread's rows: row0 + 16 i
        const int64_t nvalid = col0 < a.K ? a.rows - row0 : 0;  // valid iff 16 i < nvalid
        const char* xp = static_cast<const char*>(a.x) + (row0 * a.ldx + col0) * P::ES;
        const int64_t xstep = 16 * a.ldx * P::ES;
        uint4 v[kChunks];
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            v[i] = make_uint4(0u, 0u, 0u, 0u);
            if (16 * i < nvalid) {
                const char* p = xp + i * xstep;
                if constexpr (VEC) {
                    v[i] = __ldcs(reinterpret_cast<const uint4*>(p));
                } else {
                    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int k = 0; k < P::CH; ++k) {
                        if (col0 + k < a.K) {
                            if constexpr (ELT == Elt::BF16)
                                w[k >> 1] |= (uint32_t)reinterpret_cast<const uint16_t*>(p)[k] << ((k & 1) * 16);
                            else
                                w[k] = reinterpret_cast<const uint32_t*>(p)[k];
                        }
                    }
                    v[i] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }

        // block exponents (one byte each, 0xFF = poisoned) and the tile
        // maximum over finite blocks
        uint32_t ebp[2] = {0u, 0u};
        int local = kNoBlock;
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            uint32_t m;
            if constexpr (ELT == Elt::BF16) {
                const uint32_t M = 0x7FFF7FFFu;
                m = u16x2_max(u16x2_max(v[i].x & M, v[i].y & M), u16x2_max(v[i].z & M, v[i].w & M));
                m = u16x2_max(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = u16x2_max(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = max(m & 0xFFFFu, m >> 16);
                if (m >= 0x7F80u) m = 0xFFFFFFFFu;
            } else {
                const uint32_t M = 0x7FFFFFFFu;
                m = max(max(v[i].x & M, v[i].y & M), max(v[i].z & M, v[i].w & M));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
                if (m >= 0x7F800000u) m = 0xFFFFFFFFu;
            }
            const int e = block_exponent<P::MANT>(m);
            const uint32_t byte = m == 0xFFFFFFFFu ? 0xFFu : (uint32_t)(e + 126);  // 0..251
            ebp[i >> 2] |= byte << ((i & 3) * 8);
            if (m != 0xFFFFFFFFu) local = max(local, e);
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

        uint8_t* dp = a.data + row0 * a.K + col0;
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            const uint32_t byte = (ebp[i >> 2] >> ((i & 3) * 8)) & 0xFFu;
            const bool poisoned = byte == 0xFFu;
            const int eb = (int)byte - 126;
            const uint32_t fold = f32_pow2(max(eb - T, -126));
            uint32_t lo, hi;
            if constexpr (ELT == Elt::BF16) {
                const Bf16Grid g = bf16_grid_unit(eb);
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t b[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t s = bf2_grid(w[k] & 0x7FFF7FFFu, g) | (w[k] & 0x80008000u);
                    b[k] = e4m3x2_from_f32(f32_mul(s & 0xFFFF0000u, fold), f32_mul(s << 16, fold));
                }
                lo = b[0] | (b[1] << 16);
                hi = b[2] | (b[3] << 16);
            } else {
                const uint32_t mult = f32_pow2(-eb);
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t u[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    u[k] = f32_mul(f32_grid(w[k] & 0x7FFFFFFFu, mult) | (w[k] & 0x80000000u), fold);
                lo = e4m3x2_from_f32(u[1], u[0]) | (e4m3x2_from_f32(u[3], u[2]) << 16);
                hi = 0u;
            }
            if (poisoned) lo = hi = 0x7F7F7F7Fu;
            if (16 * i >= nvalid) continue;
            uint8_t* d = dp + (int64_t)i * 16 * a.K;
            if constexpr (VEC) {
                if constexpr (ELT == Elt::BF16)
                    __stcs(reinterpret_cast<uint2*>(d), make_uint2(lo, hi));
                else
                    __stcs(reinterpret_cast<unsigned int*>(d), lo);
            } else {
#pragma unroll
                for (int k = 0; k < P::CH; ++k)
                    if (col0 + k < a.K) d[k] = (uint8_t)((k < 4 ? lo : hi) >> ((k & 3) * 8));
            }
        }
    }
}

template <Elt ELT, bool VEC>
cudaError_t launch_one(const Block128Args& a, cudaStream_t s) {
    const int64_t tr = ceil_div(a.rows, 128), tc = ceil_div(a.K, 128);
    if (tc > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const unsigned gy = (unsigned)(tr < 65535 ? tr : 65535);
    block128_kernel<ELT, VEC><<<dim3((unsigned)tc, gy), T128<ELT>::NT, 0, s>>>(a, tr, tc);
    return cudaGetLastError();
}

bool aligned(const void* p, int64_t n) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)n) == 0; }

template <Elt ELT>
cudaError_t dispatch(const Block128Args& a, cudaStream_t s) {
    using P = T128<ELT>;
    const bool vec =
        aligned(a.x, 16) && (a.ldx * P::ES) % 16 == 0 && a.K % P::CH == 0 && aligned(a.data, P::CH);
    return vec ? launch_one<ELT, true>(a, s) : launch_one<ELT, false>(a, s);
}

}  // namespace

cudaError_t launch_block128(Elt elt, const Block128Args& a, cudaStream_t s) {
    return elt == Elt::BF16 ? dispatch<Elt::BF16>(a, s) : dispatch<Elt::FP32>(a, s);
}

}  // namespace mxq
