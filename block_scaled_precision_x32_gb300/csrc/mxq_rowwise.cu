// mxq_rowwise.cu -- the 1x32-block kernels: MXFP4 projection, the direct
// MXFP4 -> MXFP8 rowwise conversion and the packed MXFP4 deployment form.
//
// TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling recipes",
// Description, mode 1 (projection) and mode 2 (direct, MXFP8 rowwise);
// "Known limitations" (packed deployment's scale 2^126 past the cap).
//
// Work split.  Each lane owns whole 1x32 blocks: it reads a block as two
// (bf16) or four (fp32) 32-byte vectors -- one full sector each, so a warp's
// request is sector-exact -- finds the amax, the scale exponent and the
// block constants once, converts the 32 elements and writes them back with
// 32-byte stores.  No shuffles, no shared memory.  Lanes walk the flattened
// (row, block) space with a grid stride over a resident grid (a multiple of
// the SM count); the row/block cursor advances by one add per step.
// Misaligned or ragged views use the same code with element-wise loads.
#include <cuda_runtime.h>

#include <algorithm>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int64_t scale_offset(int64_t r, int64_t j, int64_t nb, int64_t Cp, int lay) {
    if (lay == 0) return r * nb + j;
    if (lay == 1) return r * Cp + j;
    return ((r >> 7) * (Cp >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

template <Elt ELT>
struct Traits;
template <>
struct Traits<Elt::BF16> {
    static constexpr int ES = 2, SEGS = 2, SEG_ELEMS = 16, MANT = 7;
};
template <>
struct Traits<Elt::FP32> {
    static constexpr int ES = 4, SEGS = 4, SEG_ELEMS = 8, MANT = 23;
};

// Load one block (valid = elements present, 1..32) as SEGS x 8 words;
// missing elements read as +0.
template <Elt ELT, bool VEC>
__device__ __forceinline__ void load_block(uint32_t (&v)[Traits<ELT>::SEGS][8], const char* p, int valid) {
    using T = Traits<ELT>;
#pragma unroll
    for (int s = 0; s < T::SEGS; ++s) {
        if constexpr (VEC) {
            if (s * T::SEG_ELEMS < valid) {
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
                    const int i0 = s * 16 + 2 * k;
                    if (i0 < valid) w = reinterpret_cast<const uint16_t*>(p)[i0];
                    if (i0 + 1 < valid) w |= (uint32_t)reinterpret_cast<const uint16_t*>(p)[i0 + 1] << 16;
                } else {
                    const int i0 = s * 8 + k;
                    if (i0 < valid) w = reinterpret_cast<const uint32_t*>(p)[i0];
                }
                v[s][k] = w;
            }
        }
    }
}

template <Elt ELT, bool VEC>
__device__ __forceinline__ void store_block(char* p, const uint32_t (&y)[Traits<ELT>::SEGS][8], int valid) {
    using T = Traits<ELT>;
#pragma unroll
    for (int s = 0; s < T::SEGS; ++s) {
        if constexpr (VEC) {
            if (s * T::SEG_ELEMS < valid) st32(p + 32 * s, y[s]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if constexpr (ELT == Elt::BF16) {
                    const int i0 = s * 16 + 2 * k;
                    if (i0 < valid) reinterpret_cast<uint16_t*>(p)[i0] = (uint16_t)y[s][k];
                    if (i0 + 1 < valid) reinterpret_cast<uint16_t*>(p)[i0 + 1] = (uint16_t)(y[s][k] >> 16);
                } else {
                    const int i0 = s * 8 + k;
                    if (i0 < valid) reinterpret_cast<uint32_t*>(p)[i0] = y[s][k];
                }
            }
        }
    }
}

// 32 payload bytes of one block; DST 2: one 32-byte store, 1: two 16-byte
// stores, 0: bytes.
template <int DST>
__device__ __forceinline__ void store_payload(uint8_t* p, const uint32_t (&b)[8], int valid) {
    if constexpr (DST == 2) {
        st32(p, b);
    } else if constexpr (DST == 1) {
        st16(p, b[0], b[1], b[2], b[3]);
        if (valid > 16) st16(p + 16, b[4], b[5], b[6], b[7]);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < valid) p[i] = (uint8_t)(b[i >> 2] >> ((i & 3) * 8));
    }
}

// Largest magnitude pattern of the block; any NaN gives a NaN pattern
// (above every finite and infinite magnitude).
// 16 bytes of nibbles (32 elements; valid of them present).  DST 2: one
// 16-byte store, 1: 8-byte stores, 0: bytes.
template <int DST>
__device__ __forceinline__ void store_nibbles(uint8_t* p, const uint32_t (&n)[4], int valid) {
    const int nbytes = (valid + 1) >> 1;
    if constexpr (DST == 2) {
        st16(p, n[0], n[1], n[2], n[3]);
    } else if constexpr (DST == 1) {
        *reinterpret_cast<uint2*>(p) = make_uint2(n[0], n[1]);
        if (nbytes > 8) *reinterpret_cast<uint2*>(p + 8) = make_uint2(n[2], n[3]);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < nbytes) p[i] = (uint8_t)(n[i >> 2] >> ((i & 3) * 8));
    }
}

template <Elt ELT>
__device__ __forceinline__ uint32_t block_amax(const uint32_t (&v)[Traits<ELT>::SEGS][8]) {
    using T = Traits<ELT>;
    uint32_t m = 0u;
    if constexpr (ELT == Elt::BF16) {
#pragma unroll
        for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
            for (int k = 0; k < 8; ++k) m = bf2_absmax(m, v[s][k]);
        m &= 0x7FFF7FFFu;
        return max(m & 0xFFFFu, m >> 16);
    } else {
#pragma unroll
        for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
            for (int k = 0; k < 8; ++k) m = f32_absmax(m, v[s][k]);
        return m & 0x7FFFFFFFu;
    }
}

template <RowMode MODE, Elt ELT, bool VEC, int DST>
__global__ void __launch_bounds__(kThreads) rowwise_kernel(RowwiseArgs a, int64_t nb, int64_t step_r,
                                                           int64_t step_c) {
    using T = Traits<ELT>;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    const int64_t total = a.rows * nb;
    const int64_t Cp = (nb + 3) & ~int64_t(3);
    if (a.skip != nullptr && *a.skip != 0) return;  // skip-update request: write nothing
    int64_t r, j;
    split_index(tid, nb, r, j);

    for (int64_t w = tid; w < total; w += S) {
        const int64_t col0 = j * 32;
        const int valid = (int)min((int64_t)32, a.K - col0);
        const char* xp = static_cast<const char*>(a.x) + (r * a.ldx + col0) * T::ES;
        uint32_t v[T::SEGS][8];
        load_block<ELT, VEC>(v, xp, valid);

        const uint32_t amax = block_amax<ELT>(v);
        const bool poisoned = amax >= (ELT == Elt::BF16 ? 0x7F80u : 0x7F800000u);
        const int e = block_exponent<T::MANT, MODE == RowMode::MXFP4 ? 126 : 125>(amax);

        if constexpr (MODE == RowMode::PROJECT) {
            uint32_t y[T::SEGS][8];
            const bool top = e == 125;  // only there can |x| / 2^e round past 6
            if constexpr (ELT == Elt::BF16) {
                const Bf16Grid g = bf16_grid_unit(e);
                const uint32_t scl = bf16_pow2_pair(e);
#pragma unroll
                for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
                    for (int k = 0; k < 8; ++k) y[s][k] = bf2_grid(v[s][k], g);
                if (top)
#pragma unroll
                    for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
                        for (int k = 0; k < 8; ++k) y[s][k] = bf2_sat(y[s][k], 0x40C040C0u);
#pragma unroll
                for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        y[s][k] = poisoned ? 0x7FC07FC0u : (bf2_mul(y[s][k], scl) | (v[s][k] & 0x80008000u));
            } else {
                const uint32_t mult = f32_pow2(-e), scl = f32_pow2(e);
#pragma unroll
                for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
                    for (int k = 0; k < 8; ++k) y[s][k] = f32_grid(v[s][k], mult);
                if (top)
#pragma unroll
                    for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
                        for (int k = 0; k < 8; ++k) y[s][k] = f32_sat(y[s][k]);
#pragma unroll
                for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        y[s][k] = poisoned ? 0x7FC00000u : (f32_mul(y[s][k], scl) | (v[s][k] & 0x80000000u));
            }
            store_block<ELT, VEC>(static_cast<char*>(a.y) + (r * a.ldy + col0) * T::ES, y, valid);
        } else if constexpr (MODE == RowMode::MXFP4) {
            // E2M1 codes of x / 2^e by the hardware conversion (round to nearest
            // even; |x| / 2^e <= 6 by the choice of e, so nothing saturates).
            const uint32_t mult = f32_pow2(-e);
            uint32_t n[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if constexpr (ELT == Elt::BF16) {
                        const uint32_t w = v[s][k];
                        const int i = s * 8 + k;  // byte i holds elements 2i, 2i+1
                        n[i >> 2] |= e2m1x2_from_f32(f32_mul(w & 0xFFFF0000u, mult), f32_mul(w << 16, mult))
                                     << ((i & 3) * 8);
                    } else if ((k & 1) == 0) {
                        const int i = (s * 8 + k) >> 1;
                        n[i >> 2] |= e2m1x2_from_f32(f32_mul(v[s][k + 1], mult), f32_mul(v[s][k], mult))
                                     << ((i & 3) * 8);
                    }
                }
            if (poisoned) n[0] = n[1] = n[2] = n[3] = 0u;
            store_nibbles<DST>(a.data + r * ((a.K + 1) >> 1) + j * 16, n, valid);
            a.scales[scale_offset(r, j, nb, Cp, a.lay)] = (uint8_t)(poisoned ? 255 : e + 127);
        } else {
            // Fixed-shift-6 lift: UE8M0 code max(e + 121, 0); payload p * 2^(e + 127 - code).
            const int code = poisoned ? 255 : max(e + 121, 0);
            const int shift = e + 127 - code;  // 6, or 1..5 when the code is clamped at 0
            uint32_t b[8];
            if constexpr (ELT == Elt::BF16) {
                // Round where the payload P reads as P * 2^(-120 + 16k): there the
                // bf16 exponent field is the E4M3 one plus 16k, so bits 10..4 of each
                // pattern are the E4M3 exponent and mantissa.  k keeps the
                // multiplier 2^(7 - code + 16k) a normal bf16.
                const int k16 = code > 133 ? ((code - 133 + 15) >> 4) << 4 : 0;
                Bf16Grid g;
                g.mult = bf16_pow2_pair(7 - code + k16);
                g.floor = bf16_pow2_pair(shift - 120 + k16);
                const uint32_t sat6 = g.floor + 0x01400140u;  // 6 * floor
                const bool top = e == 125;
#pragma unroll
                for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t w0 = v[s][2 * q], w1 = v[s][2 * q + 1];
                        uint32_t t0 = bf2_grid(w0, g), t1 = bf2_grid(w1, g);
                        if (top) {
                            t0 = bf2_sat(t0, sat6);
                            t1 = bf2_sat(t1, sat6);
                        }
                        // magnitude bytes from the rounded values, sign bits from the inputs
                        b[4 * s + q] = lop_select(prmt(t0 >> 4, t1 >> 4, 0x6420u), prmt(w0, w1, 0x7531u), 0x7F7F7F7Fu);
                    }
            } else {
                // payload p * 2^shift, shift in 1..6: an exact E4M3 normal; E2M1
                // codes by the hardware conversion, bytes from a table
                const uint32_t mult = f32_pow2(-e);
                const E4m3Table tab = e4m3_table(shift);
#pragma unroll
                for (int s = 0; s < T::SEGS; ++s)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        b[2 * s + q] =
                            e4m3x4_from_grid(v[s][4 * q], v[s][4 * q + 1], v[s][4 * q + 2], v[s][4 * q + 3], mult, tab);
            }
            if (poisoned)
#pragma unroll
                for (int i = 0; i < 8; ++i) b[i] = 0x7F7F7F7Fu;
            store_payload<DST>(a.data + r * a.K + col0, b, valid);
            a.scales[scale_offset(r, j, nb, Cp, a.lay)] = (uint8_t)code;
        }

        j += step_c;
        r += step_r;
        if (j >= nb) {
            j -= nb;
            r += 1;
        }
    }

    if (MODE != RowMode::PROJECT && a.lay != 0) {
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

// The projection of fp32 input, K % 32 == 0, 32-byte aligned input and
// output rows: four lanes share a 1x32 block, each with 8 elements -- one
// 32-byte load, one 32-byte store -- so a warp's load and store each cover
// 1 KB of contiguous memory (8 blocks).  With a lane per block the 128 bytes
// a lane reads and writes made every load and store instruction touch 32
// separate lines: 86.4 against 77.7 us on 8192 x 8192 fp32.  The block's
// amax joins over its four lanes by two shuffles (the lane units are a
// multiple of 4, and so is the grid stride, so a block's four lanes are
// always active together); each lane then projects its 8 elements with
// rowwise_kernel's arithmetic.  The read-heavy fp32 forms (MXFP8, packed
// MXFP4) keep a lane per block: four lanes repeat the block's exponent,
// table and scale work, and with 1-8 units a thread in flight they ran at
// 59.9 / 55.8 us or more against 53.4 / 48.8 us.
__global__ void __launch_bounds__(kThreads) project_f32_quad_kernel(RowwiseArgs a, int64_t nb, int64_t step_r,
                                                                    int64_t step_c) {
    const int64_t nq = a.rows * nb * 4;  // lanes: 4 per block
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t S = (int64_t)gridDim.x * kThreads;  // step_r rows + step_c blocks
    if (a.skip != nullptr && *a.skip != 0) return;  // skip-update request: write nothing
    const unsigned gmask = 0xFu << (threadIdx.x & 28);  // the block's four lanes
    const int p = (int)(tid & 3);                       // elements 8 p .. 8 p + 7 of each block
    int64_t r, j;
    split_index(tid >> 2, nb, r, j);
    for (int64_t tq = tid; tq < nq; tq += S) {
        uint32_t v[8];
        ld32(v, static_cast<const char*>(a.x) + (r * a.ldx + j * 32 + 8 * p) * 4);
        uint32_t m = 0u;
#pragma unroll
        for (int k = 0; k < 8; ++k) m = f32_absmax(m, v[k]);
        m &= 0x7FFFFFFFu;  // magnitude patterns: NaN > Inf > finite
        m = max(m, __shfl_xor_sync(gmask, m, 1));
        m = max(m, __shfl_xor_sync(gmask, m, 2));
        const bool poisoned = m >= 0x7F800000u;
        const int e = block_exponent<23>(m);
        const uint32_t mult = f32_pow2(-e), scl = f32_pow2(e);
        const bool top = e == 125;  // only there can |x| / 2^e round past 6
        uint32_t y[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            uint32_t t = f32_grid(v[k], mult);
            if (top) t = f32_sat(t);
            y[k] = poisoned ? 0x7FC00000u : (f32_mul(t, scl) | (v[k] & 0x80000000u));
        }
        st32(static_cast<char*>(a.y) + (r * a.ldy + j * 32 + 8 * p) * 4, y);
        j += step_c;
        r += step_r;
        if (j >= nb) {
            j -= nb;
            r += 1;
        }
    }
}

// MXFP8 rowwise and packed MXFP4 of fp32 input, K % 32 == 0, 32-byte
// aligned input rows, 16-byte aligned output: LANES = 2 lanes share a 1x32
// block, each with 16 elements (two 32-byte loads, half a line), joining the
// block's amax by one shuffle; each lane encodes its 16 elements as
// rowwise_kernel does, and lane 0 writes the scale byte.  8192 x 8192:
// MXFP8 54.1 -> 52.1 us, MXFP4 49.2 -> 47.8 us against a lane per block
// (128 bytes a lane; every warp load touched 32 lines); four lanes per
// block, which repeat the block's exponent, table and scale work four times,
// took 71.0 / 67.9 us.
template <RowMode MODE, int LANES>
__global__ void __launch_bounds__(kThreads) rowwise_f32_lanes_kernel(RowwiseArgs a, int64_t nb, int64_t step_r,
                                                                     int64_t step_c) {
    constexpr int EPL = 32 / LANES, SEG = EPL / 8;
    const int64_t nq = a.rows * nb * LANES;
    const int64_t Cp = (nb + 3) & ~int64_t(3);
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t S = (int64_t)gridDim.x * kThreads;
    if (a.skip != nullptr && *a.skip != 0) return;  // skip-update request: write nothing
    const unsigned gmask = ((1u << LANES) - 1u) << (threadIdx.x & (32 - LANES));  // the block's lanes
    const int p = (int)(tid % LANES);
    int64_t r, j;
    split_index(tid / LANES, nb, r, j);
    for (int64_t tq = tid; tq < nq; tq += S) {
        uint32_t v[SEG][8];
#pragma unroll
        for (int sg = 0; sg < SEG; ++sg) ld32(v[sg], static_cast<const char*>(a.x) + (r * a.ldx + j * 32 + EPL * p + 8 * sg) * 4);
        uint32_t m = 0u;
#pragma unroll
        for (int sg = 0; sg < SEG; ++sg)
#pragma unroll
            for (int k = 0; k < 8; ++k) m = f32_absmax(m, v[sg][k]);
        m &= 0x7FFFFFFFu;
#pragma unroll
        for (int o = 1; o < LANES; o <<= 1) m = max(m, __shfl_xor_sync(gmask, m, o));
        const bool poisoned = m >= 0x7F800000u;
        const int e = block_exponent<23, MODE == RowMode::MXFP4 ? 126 : 125>(m);
        const uint32_t mult = f32_pow2(-e);
        if constexpr (MODE == RowMode::MXFP8) {
            const int code = poisoned ? 255 : max(e + 121, 0);
            const E4m3Table tab = e4m3_table(e + 127 - code);
            uint32_t b[EPL / 4];
#pragma unroll
            for (int q = 0; q < EPL / 4; ++q)
                b[q] = poisoned ? 0x7F7F7F7Fu
                                : e4m3x4_from_grid(v[q >> 1][4 * (q & 1)], v[q >> 1][4 * (q & 1) + 1], v[q >> 1][4 * (q & 1) + 2],
                                                   v[q >> 1][4 * (q & 1) + 3], mult, tab);
            uint8_t* d = a.data + r * a.K + j * 32 + EPL * p;
            if constexpr (EPL == 16) st16(d, b[0], b[1], b[2], b[3]);
            else *reinterpret_cast<uint2*>(d) = make_uint2(b[0], b[1]);
            if (p == 0) a.scales[scale_offset(r, j, nb, Cp, a.lay)] = (uint8_t)code;
        } else {
            uint32_t n[EPL / 8];
#pragma unroll
            for (int q = 0; q < EPL / 8; ++q) {
                n[q] = 0u;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    n[q] |= e2m1x2_from_f32(f32_mul(v[q][2 * i + 1], mult), f32_mul(v[q][2 * i], mult)) << (8 * i);
                if (poisoned) n[q] = 0u;
            }
            uint8_t* d = a.data + r * (a.K >> 1) + j * 16 + (EPL / 2) * p;
            if constexpr (EPL == 16) *reinterpret_cast<uint2*>(d) = make_uint2(n[0], n[1]);
            else *reinterpret_cast<uint32_t*>(d) = n[0];
            if (p == 0) a.scales[scale_offset(r, j, nb, Cp, a.lay)] = (uint8_t)(poisoned ? 255 : e + 127);
        }
        j += step_c;
        r += step_r;
        if (j >= nb) {
            j -= nb;
            r += 1;
        }
    }
    if (a.lay != 0) {
        // zero the padding of the padded / swizzled scale buffer
        const int64_t Rp = (a.rows + 127) & ~int64_t(127);
        const int64_t extra = Cp - nb;
        const int64_t padA = a.rows * extra, padB = (Rp - a.rows) * Cp;
        for (int64_t q = tid; q < padA + padB; q += S) {
            int64_t rr, jj;
            if (q < padA) {
                rr = q / extra;
                jj = nb + (q - rr * extra);
            } else {
                const int64_t w = q - padA;
                rr = a.rows + w / Cp;
                jj = w - (rr - a.rows) * Cp;
            }
            a.scales[scale_offset(rr, jj, nb, Cp, a.lay)] = 0;
        }
    }
}

template <RowMode MODE>
cudaError_t launch_f32_lanes(const RowwiseArgs& a, cudaStream_t s) {
    constexpr int L = 2;
    const int64_t nb = a.K / 32;
    int64_t grid = ceil_div(a.rows * nb * L, (int64_t)kThreads);
    const int64_t cap = (int64_t)1 << 30;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    const int64_t sb = grid * kThreads / L;
    rowwise_f32_lanes_kernel<MODE, L><<<(unsigned)grid, kThreads, 0, s>>>(a, nb, sb / nb, sb % nb);
    return cudaGetLastError();
}

cudaError_t launch_project_f32_quad(const RowwiseArgs& a, cudaStream_t s) {
    const int64_t nb = a.K / 32;
    int64_t grid = ceil_div(a.rows * nb * 4, (int64_t)kThreads);
    const int64_t cap = (int64_t)1 << 30;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    const int64_t sb = grid * kThreads / 4;  // blocks per grid stride
    project_f32_quad_kernel<<<(unsigned)grid, kThreads, 0, s>>>(a, nb, sb / nb, sb % nb);
    return cudaGetLastError();
}

template <RowMode MODE, Elt ELT, bool VEC, int DST>
cudaError_t launch_one(const RowwiseArgs& a, cudaStream_t s) {
    const int64_t nb = (a.K + 31) / 32;
    const int64_t total = a.rows * nb;
    // resident CTAs per SM, asked once (thread-safe static initialisation)
    static const int occ = [] {
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, rowwise_kernel<MODE, ELT, VEC, DST>, kThreads, 0) !=
                cudaSuccess ||
            o < 1)
            o = 1;
        return o;
    }();
    // Grid size, measured on 8192 x 8192 (a sweep of 1..12 x the resident grid
    // and one thread per block): the projection, whose traffic is half writes,
    // and every fp32 form (128 bytes per thread) are fastest with a thread per
    // block (bf16 projection 41 us against 46 us for a resident grid; fp32
    // MXFP8 / MXFP4 54.0 / 49.2 us against 57.3 / 52.0 us at 4 x resident);
    // the read-heavy bf16 MXFP8 and MXFP4 forms with 4 x the resident grid,
    // about two blocks per thread (32.3 / 27.1 us against 34.5 / 29.6 us
    // resident, 34.9 / 27.7 us one per thread).  Larger tensors want the grid
    // to grow with them: about 3 (MXFP8) or 2 (MXFP4) blocks per thread, never
    // fewer CTAs than 4 x resident (MoE stack 32 x 4096 x 7184: MXFP8 449.5 ->
    // 406.8 us, MXFP4 362.2 -> 330.7 us; 32768 x 16384: 248.3 -> 228.8 us and
    // 203.5 -> 189.7 us; 8192 x 8192 keeps 4 x resident).  (Aligned fp32 views
    // with K % 32 == 0 take the four- and two-lane kernels above instead.)
    int64_t grid = ceil_div(total, (int64_t)kThreads);
    const bool one_per_thread = MODE == RowMode::PROJECT || ELT == Elt::FP32;
    int64_t cap = (int64_t)1 << 30;
    if (!one_per_thread) {
        const int64_t bpt = MODE == RowMode::MXFP4 ? 2 : 3;  // blocks per thread
        cap = std::min(std::max((int64_t)sm_count() * occ * 4, ceil_div(total, (int64_t)kThreads * bpt)), cap);
    }
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    const int64_t stride = grid * kThreads;
    rowwise_kernel<MODE, ELT, VEC, DST><<<(unsigned)grid, kThreads, 0, s>>>(a, nb, stride / nb, stride % nb);
    return cudaGetLastError();
}

bool aligned(const void* p, int64_t n) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)n) == 0; }

template <RowMode MODE, Elt ELT>
cudaError_t dispatch(const RowwiseArgs& a, cudaStream_t s) {
    using T = Traits<ELT>;
    // vector path: every 32-byte segment of the input (and projection output) is aligned
    bool vec = aligned(a.x, 32) && (a.ldx * T::ES) % 32 == 0 && (a.K * T::ES) % 32 == 0;
    if constexpr (ELT == Elt::FP32 && MODE == RowMode::PROJECT) {
        // whole blocks, aligned input and output rows: four lanes per block
        if (vec && a.K % 32 == 0 && aligned(a.y, 32) && (a.ldy * 4) % 32 == 0) return launch_project_f32_quad(a, s);
    }
    if constexpr (ELT == Elt::FP32 && MODE != RowMode::PROJECT) {
        // whole blocks, aligned input rows and 16-byte aligned output: two lanes per block
        if (vec && a.K % 32 == 0 && aligned(a.data, 16)) return launch_f32_lanes<MODE>(a, s);
    }
    if constexpr (MODE == RowMode::PROJECT) {
        vec = vec && aligned(a.y, 32) && (a.ldy * T::ES) % 32 == 0;
        return vec ? launch_one<MODE, ELT, true, 0>(a, s) : launch_one<MODE, ELT, false, 0>(a, s);
    }
    if constexpr (MODE == RowMode::MXFP4) {
        // nibble rows are ceil(K/2) bytes: 16-byte stores need K % 32 == 0, 8-byte ones K % 16 == 0
        const int dst = (aligned(a.data, 16) && a.K % 32 == 0) ? 2 : (aligned(a.data, 8) && a.K % 16 == 0) ? 1 : 0;
        if (vec) {
            if (dst == 2) return launch_one<MODE, ELT, true, 2>(a, s);
            if (dst == 1) return launch_one<MODE, ELT, true, 1>(a, s);
            return launch_one<MODE, ELT, true, 0>(a, s);
        }
        return launch_one<MODE, ELT, false, 0>(a, s);
    }
    const int dst = (aligned(a.data, 32) && a.K % 32 == 0) ? 2 : (aligned(a.data, 16) && a.K % 16 == 0) ? 1 : 0;
    if (vec) {
        if (dst == 2) return launch_one<MODE, ELT, true, 2>(a, s);
        if (dst == 1) return launch_one<MODE, ELT, true, 1>(a, s);
        return launch_one<MODE, ELT, true, 0>(a, s);
    }
    return launch_one<MODE, ELT, false, 0>(a, s);
}

}  // namespace

cudaError_t launch_rowwise(RowMode mode, Elt elt, const RowwiseArgs& a, cudaStream_t s) {
    if (mode == RowMode::PROJECT)
        return elt == Elt::BF16 ? dispatch<RowMode::PROJECT, Elt::BF16>(a, s)
                                : dispatch<RowMode::PROJECT, Elt::FP32>(a, s);
    if (mode == RowMode::MXFP4)
        return elt == Elt::BF16 ? dispatch<RowMode::MXFP4, Elt::BF16>(a, s) : dispatch<RowMode::MXFP4, Elt::FP32>(a, s);
    return elt == Elt::BF16 ? dispatch<RowMode::MXFP8, Elt::BF16>(a, s) : dispatch<RowMode::MXFP8, Elt::FP32>(a, s);
}

}  // namespace mxq
