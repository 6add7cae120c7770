// mxq_rowwise.cu -- the two 1x32-block kernels: MXFP4 projection and the
// direct MXFP4 -> MXFP8 rowwise conversion.
//
// TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling recipes",
// Description, mode 1 (projection) and mode 2 (direct, MXFP8 rowwise).
//
// Work split.  A "chunk" is 16 bytes of one row (8 bf16 or 4 fp32); a 1x32
// block is L = 4 (bf16) or 8 (fp32) consecutive lanes, so the block amax is
// two or three xor-shuffles.  Rows are cut into nb*L chunks (chunks past K
// in a short last block load zeros and store nothing).  Threads walk the
// flattened (row, chunk) space with a grid stride, kItems chunks in flight
// per thread, the row/column cursor advanced incrementally.  The grid is a
// resident multiple of the SM count.
#include <cuda_runtime.h>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 4;

__device__ __forceinline__ int64_t scale_offset(int64_t r, int64_t j, int64_t nb, int64_t Cp, int lay) {
    if (lay == 0) return r * nb + j;
    if (lay == 1) return r * Cp + j;
    return ((r >> 7) * (Cp >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

template <Elt ELT>
struct Traits;
template <>
struct Traits<Elt::BF16> {
    static constexpr int ES = 2, CH = 8, L = 4, MANT = 7;
};
template <>
struct Traits<Elt::FP32> {
    static constexpr int ES = 4, CH = 4, L = 8, MANT = 23;
};

template <Elt ELT, bool VEC>
__device__ __forceinline__ uint4 load_chunk(const char* row, int64_t col0, int64_t K, bool ok) {
    using T = Traits<ELT>;
    if (!ok) return make_uint4(0u, 0u, 0u, 0u);
    if constexpr (VEC) {
        return __ldcs(reinterpret_cast<const uint4*>(row + col0 * T::ES));
    } else {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < T::CH; ++i) {
            const int64_t c = col0 + i;
            if (c < K) {
                if constexpr (ELT == Elt::BF16)
                    w[i >> 1] |= (uint32_t)reinterpret_cast<const uint16_t*>(row)[c] << ((i & 1) * 16);
                else
                    w[i] = reinterpret_cast<const uint32_t*>(row)[c];
            }
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <Elt ELT, bool VEC>
__device__ __forceinline__ void store_chunk(char* row, int64_t col0, int64_t K, uint4 v) {
    using T = Traits<ELT>;
    if constexpr (VEC) {
        __stcs(reinterpret_cast<uint4*>(row + col0 * T::ES), v);
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < T::CH; ++i) {
            const int64_t c = col0 + i;
            if (c < K) {
                if constexpr (ELT == Elt::BF16)
                    reinterpret_cast<uint16_t*>(row)[c] = (uint16_t)(w[i >> 1] >> ((i & 1) * 16));
                else
                    reinterpret_cast<uint32_t*>(row)[c] = w[i];
            }
        }
    }
}

// Largest magnitude pattern of the chunk, reduced over the block's lanes.
template <Elt ELT>
__device__ __forceinline__ uint32_t block_amax(uint4 v) {
    if constexpr (ELT == Elt::BF16) {
        const uint32_t M = 0x7FFF7FFFu;
        uint32_t m = u16x2_max(u16x2_max(v.x & M, v.y & M), u16x2_max(v.z & M, v.w & M));
        m = u16x2_max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = u16x2_max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        return max(m & 0xFFFFu, m >> 16);
    } else {
        const uint32_t M = 0x7FFFFFFFu;
        uint32_t m = max(max(v.x & M, v.y & M), max(v.z & M, v.w & M));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
        return m;
    }
}

// Projection of one chunk: sign(x) * p * 2^e.
template <Elt ELT>
__device__ __forceinline__ uint4 project_chunk(uint4 v, int e, bool poisoned) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (ELT == Elt::BF16) {
        const Bf16Grid g = bf16_grid_unit(e);
        const uint32_t scl = bf16_pow2_pair(e);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t t = bf2_grid(w[i] & 0x7FFF7FFFu, g);
            w[i] = poisoned ? 0x7FC07FC0u : (bf2_mul(t, scl) | (w[i] & 0x80008000u));
        }
    } else {
        const uint32_t mult = f32_pow2(-e), scl = f32_pow2(e);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t t = f32_grid(w[i] & 0x7FFFFFFFu, mult);
            w[i] = poisoned ? 0x7FC00000u : (f32_mul(t, scl) | (w[i] & 0x80000000u));
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Fixed-shift-6 lift of one chunk into E4M3 payload bytes (8 for bf16 in a
// uint2, 4 for fp32 in .x).  code = max(e + 121, 0) is the UE8M0 scale; the
// payload is p * 2^(e + 127 - code).
template <Elt ELT>
__device__ __forceinline__ uint2 mxfp8_chunk(uint4 v, int e, int code, bool poisoned) {
    const int shift = e + 127 - code;  // 6, or 1..5 when the scale code is clamped at 0
    if constexpr (ELT == Elt::BF16) {
        // Round in a domain where the payload P appears as P * 2^(-120 + 16k):
        // there the bf16 exponent field is the E4M3 one plus 16k, so bits
        // 10..4 of each bf16 pattern are the E4M3 exponent and mantissa.  k
        // keeps the multiplier 2^(7 - code + 16k) a normal bf16.
        const int k = code > 133 ? (code - 133 + 15) >> 4 : 0;
        Bf16Grid g;
        g.mult = bf16_pow2_pair(7 - code + 16 * k);
        g.floor = bf16_pow2_pair(shift - 120 + 16 * k);
        g.sat = g.floor + 0x01400140u;  // 6 * floor
        const uint32_t t0 = bf2_grid(v.x & 0x7FFF7FFFu, g);
        const uint32_t t1 = bf2_grid(v.y & 0x7FFF7FFFu, g);
        const uint32_t t2 = bf2_grid(v.z & 0x7FFF7FFFu, g);
        const uint32_t t3 = bf2_grid(v.w & 0x7FFF7FFFu, g);
        uint32_t lo = lop_select(prmt(t0 >> 4, t1 >> 4, 0x6420u), prmt(v.x, v.y, 0x7531u), 0x7F7F7F7Fu);
        uint32_t hi = lop_select(prmt(t2 >> 4, t3 >> 4, 0x6420u), prmt(v.z, v.w, 0x7531u), 0x7F7F7F7Fu);
        if (poisoned) lo = hi = 0x7F7F7F7Fu;
        return make_uint2(lo, hi);
    } else {
        const uint32_t mult = f32_pow2(-e), up = f32_pow2(shift);
        uint32_t p[4];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            p[i] = f32_mul(f32_grid(w[i] & 0x7FFFFFFFu, mult), up) | (w[i] & 0x80000000u);
        uint32_t out = e4m3x2_from_f32(p[1], p[0]) | (e4m3x2_from_f32(p[3], p[2]) << 16);
        if (poisoned) out = 0x7F7F7F7Fu;
        return make_uint2(out, 0u);
    }
}

template <Elt ELT, bool VEC>
__device__ __forceinline__ void store_payload(uint8_t* drow, int64_t col0, int64_t K, uint2 b) {
    using T = Traits<ELT>;
    if constexpr (VEC) {
        if constexpr (ELT == Elt::BF16)
            __stcs(reinterpret_cast<uint2*>(drow + col0), b);
        else
            __stcs(reinterpret_cast<unsigned int*>(drow + col0), b.x);
    } else {
#pragma unroll
        for (int i = 0; i < T::CH; ++i) {
            const int64_t c = col0 + i;
            if (c < K) drow[c] = (uint8_t)((i < 4 ? b.x : b.y) >> ((i & 3) * 8));
        }
    }
}

template <RowMode MODE, Elt ELT, bool VEC>
__global__ void __launch_bounds__(kThreads) rowwise_kernel(RowwiseArgs a, int64_t cpr, int64_t step_r,
                                                           int64_t step_c) {
    using T = Traits<ELT>;
    const int lane = threadIdx.x & 31;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t total = a.rows * cpr;
    const int64_t nb = (a.K + 31) >> 5;
    const int64_t Cp = (nb + 3) & ~int64_t(3);

    int64_t r[kItems], cc[kItems];
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
        const int64_t w = tid + u * S;
        r[u] = w / cpr;
        cc[u] = w - r[u] * cpr;
    }

    for (int64_t wbase = tid - lane; wbase < total; wbase += kItems * S) {
        uint4 v[kItems];
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
            const bool ok = r[u] < a.rows && cc[u] * T::CH < a.K;
            const char* xrow = static_cast<const char*>(a.x) + (ok ? r[u] * a.ldx * T::ES : 0);
            v[u] = load_chunk<ELT, VEC>(xrow, cc[u] * T::CH, a.K, ok);
        }
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
            const uint32_t amax = block_amax<ELT>(v[u]);
            const bool poisoned = amax >= (ELT == Elt::BF16 ? 0x7F80u : 0x7F800000u);
            const int e = block_exponent<T::MANT>(amax);
            const bool ok = r[u] < a.rows && cc[u] * T::CH < a.K;
            const int64_t col0 = cc[u] * T::CH;
            if constexpr (MODE == RowMode::PROJECT) {
                const uint4 y = project_chunk<ELT>(v[u], e, poisoned);
                if (ok) store_chunk<ELT, VEC>(static_cast<char*>(a.y) + r[u] * a.ldy * T::ES, col0, a.K, y);
            } else {
                const int code = poisoned ? 255 : max(e + 121, 0);
                const uint2 b = mxfp8_chunk<ELT>(v[u], poisoned ? 0 : e, poisoned ? 0 : code, poisoned);
                if (ok) {
                    store_payload<ELT, VEC>(a.data + r[u] * a.K, col0, a.K, b);
                    if ((lane & (T::L - 1)) == 0)
                        a.scales[scale_offset(r[u], cc[u] / T::L, nb, Cp, a.lay)] = (uint8_t)code;
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

    if (MODE == RowMode::MXFP8 && a.lay != 0) {
        // zero the padding of the padded / swizzled scale buffer
        const int64_t Rp = (a.rows + 127) & ~int64_t(127);
        const int64_t extra = Cp - nb;
        const int64_t padA = a.rows * extra, padB = (Rp - a.rows) * Cp;
        for (int64_t p = tid; p < padA + padB; p += S) {
            int64_t rr, jj;
            if (p < padA) {
                rr = p / extra;
                jj = nb + (p - rr * extra);
            } else {
                const int64_t q = p - padA;
                rr = a.rows + q / Cp;
                jj = q - (rr - a.rows) * Cp;
            }
            a.scales[scale_offset(rr, jj, nb, Cp, a.lay)] = 0;
        }
    }
}

template <RowMode MODE, Elt ELT, bool VEC>
cudaError_t launch_one(const RowwiseArgs& a, cudaStream_t s) {
    using T = Traits<ELT>;
    const int64_t nb = (a.K + 31) / 32;
    const int64_t cpr = nb * T::L;
    const int64_t total = a.rows * cpr;
    static int occ = 0;
    if (occ == 0) {
        cudaError_t err =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rowwise_kernel<MODE, ELT, VEC>, kThreads, 0);
        if (err != cudaSuccess) return err;
        if (occ < 1) occ = 1;
    }
    int64_t grid = ceil_div(total, (int64_t)kThreads * kItems);
    const int64_t resident = (int64_t)sm_count() * occ;
    if (grid > resident) grid = resident;
    if (grid < 1) grid = 1;
    const int64_t stride = grid * kThreads * kItems;
    rowwise_kernel<MODE, ELT, VEC><<<(unsigned)grid, kThreads, 0, s>>>(a, cpr, stride / cpr, stride % cpr);
    return cudaGetLastError();
}

bool aligned(const void* p, int64_t n) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)n) == 0; }

template <RowMode MODE, Elt ELT>
cudaError_t dispatch(const RowwiseArgs& a, cudaStream_t s) {
    using T = Traits<ELT>;
    bool vec = aligned(a.x, 16) && (a.ldx * T::ES) % 16 == 0 && a.K % T::CH == 0;
    if (MODE == RowMode::PROJECT) vec = vec && aligned(a.y, 16) && (a.ldy * T::ES) % 16 == 0;
    if (MODE == RowMode::MXFP8) vec = vec && aligned(a.data, T::CH);
    return vec ? launch_one<MODE, ELT, true>(a, s) : launch_one<MODE, ELT, false>(a, s);
}

}  // namespace

cudaError_t launch_rowwise(RowMode mode, Elt elt, const RowwiseArgs& a, cudaStream_t s) {
    if (mode == RowMode::PROJECT)
        return elt == Elt::BF16 ? dispatch<RowMode::PROJECT, Elt::BF16>(a, s)
                                : dispatch<RowMode::PROJECT, Elt::FP32>(a, s);
    return elt == Elt::BF16 ? dispatch<RowMode::MXFP8, Elt::BF16>(a, s) : dispatch<RowMode::MXFP8, Elt::FP32>(a, s);
}

}  // namespace mxq
