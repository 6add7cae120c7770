// mxq_dequant.cu -- MXFP8 rowwise and FP8 128x128 blockwise -> bf16 / fp32.
//
// TE PR #3790 "MXFP8TensorStorage.export_components()", Description and
// tests (the export decodes to dequantize() exactly); TE PR #3264 "MXFP4
// weight QAT on MXFP8 and FP8 block-scaling recipes", Description (UE8M0
// code 0 decodes to 2^-127, code 255 to NaN).
//
// Each thread takes 16 payload bytes (one half of a 1x32 block, inside one
// 128x128 tile), decodes them by placing the fp8 fields in an fp32 pattern
// and multiplying by 2^120 (E4M3) or 2^112 (E5M2) -- exact, subnormals
// included -- then multiplies by the scale with IEEE fp32 rounding.
#include <cuda_runtime.h>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 2;

__device__ __forceinline__ int64_t scale_offset(int64_t r, int64_t j, int64_t nb, int64_t Cp, int lay) {
    if (lay == 0) return r * nb + j;
    if (lay == 1) return r * Cp + j;
    return ((r >> 7) * (Cp >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

// fp8 byte -> exact fp32 pattern times `scale`, NaN made canonical.
template <bool E5M2>
__device__ __forceinline__ uint32_t decode_scaled(uint32_t b, uint32_t scale) {
    const uint32_t mag = b & 0x7Fu;
    uint32_t f;
    bool nan;
    if (E5M2) {
        f = f32_mul((mag << 21) | ((b & 0x80u) << 24), 0x77800000u);  // * 2^112
        nan = mag > 0x7Cu;
        if (mag == 0x7Cu) f = 0x7F800000u | ((b & 0x80u) << 24);
    } else {
        f = f32_mul((mag << 20) | ((b & 0x80u) << 24), 0x7B800000u);  // * 2^120
        nan = mag == 0x7Fu;
    }
    const uint32_t r = f32_mul(f, scale);
    return (nan || (r & 0x7FFFFFFFu) > 0x7F800000u) ? 0x7FC00000u : r;
}

// fp32 pattern -> bf16 pattern, round to nearest even (canonical NaN stays
// canonical, overflow goes to Inf).
__device__ __forceinline__ uint32_t bf16_rne(uint32_t u) { return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16; }

template <bool E5M2, bool BF16OUT, bool VEC>
__global__ void __launch_bounds__(kThreads) dequant_kernel(DequantArgs a, int64_t cpr, int64_t step_r,
                                                           int64_t step_c) {
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t total = a.rows * cpr;
    const int64_t nb = (a.K + 31) >> 5;
    const int64_t Cp = (nb + 3) & ~int64_t(3);
    const int64_t tc = (a.K + 127) >> 7;

    int64_t r[kItems], cc[kItems];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
        const int64_t w = tid + u * S;
        r[u] = w / cpr;
        cc[u] = w - r[u] * cpr;
    }
    for (int64_t wb = tid; wb < total; wb += kItems * S) {
        uint4 v[kItems];
        uint32_t scale[kItems];
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
            const int64_t col0 = cc[u] * 16;
            const bool ok = r[u] < a.rows;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            scale[u] = 0u;
            if (!ok) continue;
            const uint8_t* drow = a.data + r[u] * a.K;
            if (VEC) {
                v[u] = __ldcs(reinterpret_cast<const uint4*>(drow + col0));
            } else {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (col0 + k < a.K) w[k >> 2] |= (uint32_t)drow[col0 + k] << ((k & 3) * 8);
                v[u] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (a.kind == 0) {
                const uint32_t c = a.scales[scale_offset(r[u], col0 >> 5, nb, Cp, a.lay)];
                scale[u] = c == 255u ? 0x7FC00000u : f32_pow2((int)c - 127);
            } else {
                scale[u] = reinterpret_cast<const uint32_t*>(a.tile_scale_inv)[(r[u] >> 7) * tc + (col0 >> 7)];
            }
        }
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
            if (r[u] >= a.rows) continue;
            const int64_t col0 = cc[u] * 16;
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            uint32_t o[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) o[k] = decode_scaled<E5M2>((w[k >> 2] >> ((k & 3) * 8)) & 0xFFu, scale[u]);
            if (BF16OUT) {
                uint32_t h[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) h[k] = bf16_rne(o[2 * k]) | (bf16_rne(o[2 * k + 1]) << 16);
                uint16_t* orow = static_cast<uint16_t*>(a.out) + r[u] * a.K;
                if (VEC) {
                    __stcs(reinterpret_cast<uint4*>(orow + col0), make_uint4(h[0], h[1], h[2], h[3]));
                    __stcs(reinterpret_cast<uint4*>(orow + col0 + 8), make_uint4(h[4], h[5], h[6], h[7]));
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (col0 + k < a.K) orow[col0 + k] = (uint16_t)(h[k >> 1] >> ((k & 1) * 16));
                }
            } else {
                uint32_t* orow = static_cast<uint32_t*>(a.out) + r[u] * a.K;
                if (VEC) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        __stcs(reinterpret_cast<uint4*>(orow + col0 + 4 * q),
                               make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]));
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (col0 + k < a.K) orow[col0 + k] = o[k];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
            cc[u] += step_c;
            r[u] += step_r;
            if (cc[u] >= cpr) {
                cc[u] -= cpr;
                r[u] += 1;
            }
        }
    }
}

template <bool E5M2, bool BF16OUT, bool VEC>
cudaError_t launch_one(const DequantArgs& a, cudaStream_t s) {
    const int64_t cpr = ceil_div(a.K, 16);
    const int64_t total = a.rows * cpr;
    static int occ = 0;
    if (occ == 0) {
        cudaError_t err =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dequant_kernel<E5M2, BF16OUT, VEC>, kThreads, 0);
        if (err != cudaSuccess) return err;
        if (occ < 1) occ = 1;
    }
    int64_t grid = ceil_div(total, (int64_t)kThreads * kItems);
    const int64_t resident = (int64_t)sm_count() * occ;
    if (grid > resident) grid = resident;
    if (grid < 1) grid = 1;
    const int64_t stride = grid * kThreads * kItems;
    dequant_kernel<E5M2, BF16OUT, VEC><<<(unsigned)grid, kThreads, 0, s>>>(a, cpr, stride / cpr, stride % cpr);
    return cudaGetLastError();
}

bool aligned(const void* p, int64_t n) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)n) == 0; }

template <bool E5M2, bool BF16OUT>
cudaError_t pick_vec(const DequantArgs& a, cudaStream_t s) {
    const bool vec = aligned(a.data, 16) && aligned(a.out, 16) && a.K % 16 == 0;
    return vec ? launch_one<E5M2, BF16OUT, true>(a, s) : launch_one<E5M2, BF16OUT, false>(a, s);
}

}  // namespace

cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t s) {
    const bool e5 = a.fp8 == 1;
    if (e5) return a.out_bf16 ? pick_vec<true, true>(a, s) : pick_vec<true, false>(a, s);
    return a.out_bf16 ? pick_vec<false, true>(a, s) : pick_vec<false, false>(a, s);
}

}  // namespace mxq
