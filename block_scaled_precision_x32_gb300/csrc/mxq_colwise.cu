// mxq_colwise.cu -- direct MXFP4 -> MXFP8 columnwise (32x1 blocks) and its
// dequantize.
//
// TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling recipes",
// Description, mode 2: "MXFP8 columnwise = fresh 32x1 quantization with the
// host amax rule" of the projected weight.  The host rule is read as the
// round-up power of two: s = ceil(log2(amax / 448)) clamped to [-127, 127]
// (zero amax: -127), payloads RTNE_E4M3(y / 2^s).
//
// 32-byte aligned rows and K % 32 == 0 (tile64_kernel, bf16 or fp32): a warp owns
// a 32-row band x 64 columns.  Four lanes share a row, each with a 16-column
// chunk, so one 32-byte load per lane covers eight whole 128-byte lines and
// each row's two 1x32 blocks are read with full lines (a lane-per-row layout
// touches 32 half lines per load, which the L1 pays for).  A block's two
// lanes join their amax with one shuffle; each lane projects its chunks in
// registers (the projection never goes back to HBM).  bf16 input: the lane
// keeps its four projected chunks in registers and stages only their
// column maxima over its four rows (packed NaN-propagating abs-max), so lane
// t finds the 32x1 maxima of the column pair (2t, 2t+1) from 8 staged rows
// (72 registers, at least 12 CTAs of 2 warps per SM; 32.8 against 34.3 us on
// 8192 x 8192 with the whole projected tile staged, scanned over 32 rows
// and read back).  fp32 input is loaded one row chunk at a time, projected
// through the E2M1 conversion into the same bf16 values (f32_chunk_project)
// and staged whole in a padded shared tile, which lane t scans over the 32
// rows and the encode reads back (64 registers, held by its loads in
// flight; staging four-row maxima besides the tile took 65.7 against
// 51.9 us on 8192 x 8192).  The lanes
// encode their chunks with the bf16 multipliers 2^-s of the columns -- an
// exact product, as the projected value has two significant bits -- and
// the E4M3 conversion.  Other
// views (unaligned, or K % 32 != 0) use colwise_kernel: a warp per 32-row
// band x 32 columns, a lane per row, the same steps.
#include <cuda_runtime.h>

#include "mxq_device.cuh"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

__device__ __forceinline__ int64_t scale_offset(int64_t r, int64_t j, int64_t nb, int64_t Cp, int lay) {
    if (lay == 0) return r * nb + j;
    if (lay == 1) return r * Cp + j;
    return ((r >> 7) * (Cp >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

template <Elt ELT>
struct CW;
template <>
struct CW<Elt::BF16> {
    static constexpr int ES = 2, SEGS = 2, SEG_ELEMS = 16, MANT = 7, ROW_WORDS = 16 + 4;  // 64 B + 16 B pad
};
template <>
struct CW<Elt::FP32> {
    static constexpr int ES = 4, SEGS = 4, SEG_ELEMS = 8, MANT = 23, ROW_WORDS = 32 + 4;  // 128 B + 16 B pad
};

// Host MXFP8 exponent from the magnitude pattern of a finite amax:
// amax = (1 + f) * 2^E, amax / 448 = ((1 + f) / 1.75) * 2^(E - 8), so
// ceil(log2(amax / 448)) = E - 8 + [1 + f > 1.75].  Zero and subnormal
// amax fall below 448 * 2^-127 and clamp to -127.
template <int MANT>
__device__ __forceinline__ int host_exponent(uint32_t amax_mag) {
    const int E = (int)(amax_mag >> MANT);
    const uint32_t frac = amax_mag & ((1u << MANT) - 1u);
    int s = E - 135 + (frac > (3u << (MANT - 2)) ? 1 : 0);
    s = E == 0 ? -127 : s;
    return min(max(s, -127), 127);
}

// Zero the padding of a padded / swizzled (transposed, K x ceil(rows/32))
// scale buffer: thread p of `stride` threads takes entries p, p + stride, ...
__device__ __forceinline__ void zero_scale_padding(const ColwiseArgs& a, int64_t p0, int64_t stride) {
    const int64_t nbr = (a.rows + 31) >> 5, Cpt = (nbr + 3) & ~int64_t(3);
    const int64_t Rp = (a.K + 127) & ~int64_t(127);
    const int64_t extra = Cpt - nbr;
    const int64_t padA = a.K * extra, padB = (Rp - a.K) * Cpt;
    for (int64_t p = p0; p < padA + padB; p += stride) {
        int64_t rr, jj;
        if (p < padA) {
            rr = p / extra;
            jj = nbr + (p - rr * extra);
        } else {
            const int64_t q = p - padA;
            rr = a.K + q / Cpt;
            jj = q - (rr - a.K) * Cpt;
        }
        a.scales[scale_offset(rr, jj, nbr, Cpt, a.lay)] = 0;
    }
}

template <Elt ELT, bool VEC, int DST>
__global__ void __launch_bounds__(kThreads) colwise_kernel(ColwiseArgs a, int64_t bands) {
    using P = CW<ELT>;
    __shared__ __align__(16) uint32_t tile[kWarps][32 * P::ROW_WORDS];
    __shared__ __align__(16) uint32_t colmul[kWarps][32];
    const int w = threadIdx.x >> 5, t = threadIdx.x & 31;
    const int64_t nb = (a.K + 31) >> 5;                  // 1x32 blocks per row
    const int64_t nbr = (a.rows + 31) >> 5;              // 32x1 blocks per column
    const int64_t Cpt = (nbr + 3) & ~int64_t(3);         // padded columns of the transposed scale matrix
    const int64_t jb = (int64_t)blockIdx.x * kWarps + w;  // 1x32 block column of this warp
    const int64_t col0 = jb * 32;
    uint32_t* my = tile[w] + t * P::ROW_WORDS;
    if (a.skip != nullptr && *a.skip != 0) return;  // skip-update request: write nothing

    for (int64_t band = blockIdx.y; band < bands; band += gridDim.y) {
        const int64_t r = band * 32 + t;
        const int valid = (r < a.rows && jb < nb) ? (int)min((int64_t)32, a.K - col0) : 0;
        uint32_t v[P::SEGS][8];
        const char* xp = static_cast<const char*>(a.x) + (r * a.ldx + col0) * P::ES;
#pragma unroll
        for (int s = 0; s < P::SEGS; ++s) {
            if constexpr (VEC) {
                if (s * P::SEG_ELEMS < valid) {
                    ld32(v[s], xp + 32 * s);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) v[s][k] = 0u;
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint32_t word = 0u;
                    if constexpr (ELT == Elt::BF16) {
                        const int i0 = s * 16 + 2 * k;
                        if (i0 < valid) word = reinterpret_cast<const uint16_t*>(xp)[i0];
                        if (i0 + 1 < valid) word |= (uint32_t)reinterpret_cast<const uint16_t*>(xp)[i0 + 1] << 16;
                    } else {
                        const int i0 = s * 8 + k;
                        if (i0 < valid) word = reinterpret_cast<const uint32_t*>(xp)[i0];
                    }
                    v[s][k] = word;
                }
            }
        }

        // projection of the lane's 1x32 row block (same rule and arithmetic as mxq_fake_quant_mxfp4)
        uint32_t m = 0u;
        if constexpr (ELT == Elt::BF16) {
#pragma unroll
            for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
                for (int k = 0; k < 8; ++k) m = bf2_absmax(m, v[s][k]);
            m &= 0x7FFF7FFFu;
            m = max(m & 0xFFFFu, m >> 16);
        } else {
#pragma unroll
            for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
                for (int k = 0; k < 8; ++k) m = f32_absmax(m, v[s][k]);
            m &= 0x7FFFFFFFu;
        }
        const bool poisoned = m >= (ELT == Elt::BF16 ? 0x7F80u : 0x7F800000u);
        const int e = block_exponent<P::MANT>(m);
        if constexpr (ELT == Elt::BF16) {
            const Bf16Grid g = bf16_grid_unit(e);
            const uint32_t scl = bf16_pow2_pair(e);
#pragma unroll
            for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint32_t y = bf2_grid(v[s][k], g);
                    if (e == 125) y = bf2_sat(y, 0x40C040C0u);
                    v[s][k] = poisoned ? 0x7FC07FC0u : (bf2_mul(y, scl) | (v[s][k] & 0x80008000u));
                }
        } else {
            const uint32_t mult = f32_pow2(-e), scl = f32_pow2(e);
#pragma unroll
            for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint32_t y = f32_grid(v[s][k], mult);
                    if (e == 125) y = f32_sat(y);
                    v[s][k] = poisoned ? 0x7FC00000u : (f32_mul(y, scl) | (v[s][k] & 0x80000000u));
                }
        }
        // rows and columns outside the tensor hold +0: they add nothing to a column amax
        if (valid < 32) {
#pragma unroll
            for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int i0 = ELT == Elt::BF16 ? s * 16 + 2 * k : s * 8 + k;
                    if (ELT == Elt::BF16) {
                        if (i0 >= valid) v[s][k] &= 0xFFFF0000u;
                        if (i0 + 1 >= valid) v[s][k] &= 0x0000FFFFu;
                    } else if (i0 >= valid) {
                        v[s][k] = 0u;
                    }
                }
        }
#pragma unroll
        for (int s = 0; s < P::SEGS; ++s)
#pragma unroll
            for (int q = 0; q < 2; ++q)
                *reinterpret_cast<uint4*>(my + 8 * s + 4 * q) =
                    make_uint4(v[s][4 * q], v[s][4 * q + 1], v[s][4 * q + 2], v[s][4 * q + 3]);
        __syncwarp();

        // 32x1 column maxima.  bf16: lane t scans the column pair (2p, 2p+1),
        // p = t % 16, over rows 16h..16h+15, h = t / 16, with the packed
        // NaN-propagating abs-max, joins the other half by one shuffle, and
        // takes column 2p + h.  fp32: lane t scans column t.
        uint32_t cm;
        int cl;  // column of the tile this lane finishes
        if constexpr (ELT == Elt::BF16) {
            const int pr = t & 15, h = t >> 4;
            uint32_t m2 = 0u;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) m2 = bf2_absmax(m2, tile[w][(16 * h + rr) * P::ROW_WORDS + pr]);
            m2 = bf2_absmax(m2, __shfl_xor_sync(0xffffffffu, m2, 16));
            cm = (h ? (m2 >> 16) : m2) & 0x7FFFu;
            cl = 2 * pr + h;
        } else {
            uint32_t m1 = 0u;
#pragma unroll 8
            for (int rr = 0; rr < 32; ++rr) m1 = f32_absmax(m1, tile[w][rr * P::ROW_WORDS + t]);
            cm = m1 & 0x7FFFFFFFu;
            cl = t;
        }
        const bool cpois = cm >= (ELT == Elt::BF16 ? 0x7F80u : 0x7F800000u);
        const int sx = host_exponent<P::MANT>(cm);
        // a poisoned column block multiplies by NaN, which the E4M3 conversion turns into 0x7F
        colmul[w][cl] = cpois ? 0x7FC00000u : f32_pow2(-sx);
        const int64_t c = col0 + cl;
        if (c < a.K && band < nbr) a.scales[scale_offset(c, band, nbr, Cpt, a.lay)] = (uint8_t)(cpois ? 255 : sx + 127);
        __syncwarp();

        // encode the lane's row with the column scales
        uint32_t mul[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint4 mq = *reinterpret_cast<const uint4*>(&colmul[w][4 * q]);
            mul[4 * q] = mq.x;
            mul[4 * q + 1] = mq.y;
            mul[4 * q + 2] = mq.z;
            mul[4 * q + 3] = mq.w;
        }
        uint32_t b[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t f[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = 4 * q + u;
                uint32_t yv;
                if constexpr (ELT == Elt::BF16) {
                    const uint32_t word = v[i >> 4][(i & 15) >> 1];
                    yv = (i & 1) ? (word & 0xFFFF0000u) : (word << 16);
                } else {
                    yv = v[i >> 3][i & 7];
                }
                f[u] = f32_mul(yv, mul[i]);
            }
            b[q] = e4m3x2_from_f32(f[1], f[0]) | (e4m3x2_from_f32(f[3], f[2]) << 16);
        }
        if (valid > 0) {
            uint8_t* d = a.data + r * a.K + col0;
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
        __syncwarp();  // the tile is rewritten by the next band
    }

    if (a.lay != 0 && blockIdx.y == 0) zero_scale_padding(a, (int64_t)blockIdx.x * kThreads + threadIdx.x,
                                                          (int64_t)gridDim.x * kThreads);
}

// E4M3 conversion of two fp32 values into one 16-bit half, and two halves
// into a word.
__device__ __forceinline__ uint16_t e4m3x2_h(uint32_t hi, uint32_t lo) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "r"(hi), "r"(lo));
    return d;
}
__device__ __forceinline__ uint32_t pack_halves(uint16_t lo, uint16_t hi) {
    uint32_t d;
    asm("mov.b32 %0, {%1, %2};" : "=r"(d) : "h"(lo), "h"(hi));
    return d;
}

// 8-byte global load that skips L1 allocation.
__device__ __forceinline__ void ld8(uint32_t& lo, uint32_t& hi, const void* p) {
    asm volatile("ld.global.L1::no_allocate.v2.b32 {%0,%1}, [%2];" : "=r"(lo), "=r"(hi) : "l"(p));
}

// bf16 2^-s (s in [-127, 127]: a normal, or the subnormal 2^-127); NaN for
// a poisoned column block, so that its payloads convert to 0x7F.
__device__ __forceinline__ uint32_t bf16_col_multiplier(uint32_t cm, int sx) {
    if (cm >= 0x7F80u) return 0x7FC0u;
    return sx <= 126 ? (uint32_t)(127 - sx) << 7 : 0x0040u;
}

// fp32 input: 16 elements of one 1x32 block (exponent e) -> the projected
// values as 8 bf16x2 words.  E2M1 codes by the hardware conversion of
// x * 2^-e (round to nearest even, ties to the even code, saturating at
// +-6, sign kept); each code's grid value p as a bf16 pattern from byte
// tables indexed by PRMT (high bytes 00 3F 3F 3F 40 40 40 40, low bytes
// 00 00 80 C0 00 40 80 C0 for codes 0..7), the sign spread by one
// multiply, then p * 2^e by one exact bf16 multiply: the same value as the
// projection of the bf16 path.
__device__ __forceinline__ void f32_chunk_project(const uint32_t (&x)[16], int e, bool pois, uint32_t (&y)[8]) {
    const uint32_t mult = f32_pow2(-e), scl = bf16_pow2_pair(e);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint32_t n = e2m1x2_from_f32(f32_mul(x[4 * u + 1], mult), f32_mul(x[4 * u], mult)) |
                           (e2m1x2_from_f32(f32_mul(x[4 * u + 3], mult), f32_mul(x[4 * u + 2], mult)) << 8);
        const uint32_t sel = n & 0x7777u, sg = n & 0x8888u;
        const uint32_t hi4 = prmt(0x3F3F3F00u, 0x40404040u, sel);
        const uint32_t lo4 = prmt(0xC0800000u, 0xC0804000u, sel);
        const uint32_t p0 = prmt(lo4, hi4, 0x5140u) | ((sg * 0x01001000u) & 0x80008000u);
        const uint32_t p1 = prmt(lo4, hi4, 0x7362u) | ((sg * 0x00010010u) & 0x80008000u);
        y[2 * u] = pois ? 0x7FC07FC0u : bf2_mul(p0, scl);
        y[2 * u + 1] = pois ? 0x7FC07FC0u : bf2_mul(p1, scl);
    }
}

constexpr int kTileWarps = 2;

template <Elt ELT>
__global__ void __launch_bounds__(32 * kTileWarps, ELT == Elt::BF16 ? 12 : 16) tile64_kernel(ColwiseArgs a, int64_t bands) {
    constexpr int ES = ELT == Elt::BF16 ? 2 : 4;
    constexpr int RW = 32 + 4;  // words per staged row: 64 bf16 + 16 B pad (conflict-free 16-byte stores)
    constexpr bool F32 = ELT == Elt::FP32;
    // fp32: the projected tile, scanned for the column maxima and read back by the
    // encode; bf16 keeps its chunks in registers and stages only their column
    // maxima over each lane's four rows
    __shared__ __align__(16) uint32_t tile[kTileWarps][F32 ? 32 * RW : 8 * RW];
    __shared__ __align__(16) uint32_t colmul[kTileWarps][32];
    const int w = threadIdx.x >> 5, t = threadIdx.x & 31, q = t & 3, g = t >> 2;
    const int64_t nbr = (a.rows + 31) >> 5, Cpt = (nbr + 3) & ~int64_t(3);
    const int64_t col0 = ((int64_t)blockIdx.x * kTileWarps + w) * 64;  // first column of the warp tile
    const bool cvalid = col0 + 16 * q < a.K;                             // this lane's chunk is in the tensor
    const int64_t c0 = col0 + 2 * t;                                     // the column pair this lane scans
    // scale offsets of columns c0 and c0 + 1 without their band term (c0 is even, so
    // in the swizzled layout c0 + 1 sits 16 bytes further)
    int64_t coff, cstep;
    if (a.lay == 0) {
        coff = c0 * nbr;
        cstep = nbr;
    } else if (a.lay == 1) {
        coff = c0 * Cpt;
        cstep = Cpt;
    } else {
        coff = (c0 >> 7) * (Cpt >> 2) * 512 + (c0 & 31) * 16 + ((c0 >> 5) & 3) * 4;
        cstep = 16;
    }
    uint32_t* trow = tile[w] + g * RW + 8 * q;
    if (a.skip != nullptr && *a.skip != 0) return;  // skip-update request: write nothing

    for (int64_t band = blockIdx.y; band < bands; band += gridDim.y) {
        const int64_t rbase = band * 32 + g;  // rows rbase + 8i, i = 0..3
        const char* xp = static_cast<const char*>(a.x) + (rbase * a.ldx + col0 + 16 * q) * ES;
        const int64_t xstep = 8 * ES * a.ldx;  // 8 rows, in bytes
        uint32_t y[4][8];  // bf16: the projected chunks, held until the encode
        if constexpr (ELT == Elt::FP32) {
            // one row chunk (16 fp32, two 32-byte loads) at a time, the next one in flight
            uint32_t x[16], nx[16];
            const bool v0 = cvalid && rbase < a.rows;
            if (v0) {
                ld32(*reinterpret_cast<uint32_t(*)[8]>(&nx[0]), xp);
                ld32(*reinterpret_cast<uint32_t(*)[8]>(&nx[8]), xp + 32);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool vi = cvalid && rbase + 8 * i < a.rows;
#pragma unroll
                for (int k = 0; k < 16; ++k) x[k] = vi ? nx[k] : 0u;  // +0 adds nothing to an amax
                if (i < 3 && cvalid && rbase + 8 * (i + 1) < a.rows) {
                    ld32(*reinterpret_cast<uint32_t(*)[8]>(&nx[0]), xp + (i + 1) * xstep);
                    ld32(*reinterpret_cast<uint32_t(*)[8]>(&nx[8]), xp + (i + 1) * xstep + 32);
                }
                uint32_t m = 0u;
#pragma unroll
                for (int k = 0; k < 16; ++k) m = f32_absmax(m, x[k]);
                m &= 0x7FFFFFFFu;
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));  // the block's other half
                uint32_t yc[8];
                f32_chunk_project(x, block_exponent<23>(m), m >= 0x7F800000u, yc);
                uint32_t* d = trow + 8 * i * RW;
                *reinterpret_cast<uint4*>(d) = make_uint4(yc[0], yc[1], yc[2], yc[3]);
                *reinterpret_cast<uint4*>(d + 4) = make_uint4(yc[4], yc[5], yc[6], yc[7]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (cvalid && rbase + 8 * i < a.rows) {
                    ld32(y[i], xp + i * xstep);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) y[i][k] = 0u;  // +0 adds nothing to an amax
                }
            }
            // projection, one chunk at a time (same rule and arithmetic as mxq_fake_quant_mxfp4)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t m = 0u;
#pragma unroll
                for (int k = 0; k < 8; ++k) m = bf2_absmax(m, y[i][k]);
                m &= 0x7FFF7FFFu;
                m = max(m & 0xFFFFu, m >> 16);
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));  // the block's other half
                const int e = block_exponent<7>(m);
                const Bf16Grid gr = bf16_grid_unit(e);
                const uint32_t scl = bf16_pow2_pair(e);
                if (e != 125) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) y[i][k] = bf2_mul(bf2_grid(y[i][k], gr) | (y[i][k] & 0x80008000u), scl);
                } else {  // the upper clamp: saturate at +-6; a NaN or Inf block poisons its outputs
                    const bool pois = m >= 0x7F80u;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t u = bf2_sat(bf2_grid(y[i][k], gr) | (y[i][k] & 0x80008000u), 0x40C040C0u);
                        y[i][k] = pois ? 0x7FC07FC0u : bf2_mul(u, scl);
                    }
                }
            }
            // the lane's 16 columns, maximum over its four rows (sign bits arbitrary)
            uint32_t pm[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) pm[k] = bf2_absmax(bf2_absmax(y[0][k], y[1][k]), bf2_absmax(y[2][k], y[3][k]));
            *reinterpret_cast<uint4*>(trow) = make_uint4(pm[0], pm[1], pm[2], pm[3]);
            *reinterpret_cast<uint4*>(trow + 4) = make_uint4(pm[4], pm[5], pm[6], pm[7]);
        }
        __syncwarp();

        // 32x1 maxima of the column pair (2t, 2t+1) -- over the 32 staged rows (fp32) or
        // the eight staged four-row maxima (bf16) -- and their scales
        uint32_t m2 = 0u;
#pragma unroll
        for (int rr = 0; rr < (F32 ? 32 : 8); ++rr) m2 = bf2_absmax(m2, tile[w][rr * RW + t]);
        m2 &= 0x7FFF7FFFu;
        const uint32_t cm0 = m2 & 0xFFFFu, cm1 = m2 >> 16;
        const int sx0 = host_exponent<7>(cm0), sx1 = host_exponent<7>(cm1);
        colmul[w][t] = bf16_col_multiplier(cm0, sx0) | (bf16_col_multiplier(cm1, sx1) << 16);
        if (band < nbr && c0 < a.K) {  // K is even: c0 + 1 is in the tensor too
            uint8_t* sp = a.scales + coff + (a.lay == 2 ? ((band >> 2) << 9) + (band & 3) : band);
            sp[0] = (uint8_t)(cm0 >= 0x7F80u ? 255 : sx0 + 127);
            sp[cstep] = (uint8_t)(cm1 >= 0x7F80u ? 255 : sx1 + 127);
        }
        __syncwarp();

        // encode: the lane's chunk columns 16q.. have the multiplier words 8q..8q+7
        const uint4 ma = *reinterpret_cast<const uint4*>(&colmul[w][8 * q]);
        const uint4 mb = *reinterpret_cast<const uint4*>(&colmul[w][8 * q + 4]);
        const uint32_t mul[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        uint8_t* dp = a.data + rbase * a.K + col0 + 16 * q;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t yy[8];
            if constexpr (F32) {
                const uint32_t* d = trow + 8 * i * RW;
                const uint4 ya = *reinterpret_cast<const uint4*>(d), yb = *reinterpret_cast<const uint4*>(d + 4);
                yy[0] = ya.x, yy[1] = ya.y, yy[2] = ya.z, yy[3] = ya.w;
                yy[4] = yb.x, yy[5] = yb.y, yy[6] = yb.z, yy[7] = yb.w;
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) yy[k] = y[i][k];
            }
            uint32_t b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t z0 = bf2_mul(yy[2 * u], mul[2 * u]);
                const uint32_t z1 = bf2_mul(yy[2 * u + 1], mul[2 * u + 1]);
                b[u] = pack_halves(e4m3x2_h(z0 & 0xFFFF0000u, z0 << 16), e4m3x2_h(z1 & 0xFFFF0000u, z1 << 16));
            }
            if (cvalid && rbase + 8 * i < a.rows) st16(dp + 8 * i * a.K, b[0], b[1], b[2], b[3]);
        }
        __syncwarp();  // the tile is rewritten by the next band
    }

    if (a.lay != 0 && blockIdx.y == 0) zero_scale_padding(a, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                                                          (int64_t)gridDim.x * blockDim.x);
}

// Dequantize of the columnwise form: out[r, c] = payload * 2^(code(c, r/32) - 127).
// One thread per (32-row band, column), consecutive threads on consecutive
// columns, so every row access of a warp is contiguous.
template <bool E5M2, bool BF16OUT>
__global__ void __launch_bounds__(kThreads) colwise_dequant_kernel(DequantArgs a) {
    const int64_t nbr = (a.rows + 31) >> 5;
    const int64_t Cpt = (nbr + 3) & ~int64_t(3);
    const int64_t total = nbr * a.K;
    for (int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * kThreads) {
        const int64_t band = idx / a.K, c = idx - band * a.K;
        const uint32_t code = a.scales[scale_offset(c, band, nbr, Cpt, a.lay)];
        const uint32_t scale = code == 255u ? 0x7FC00000u : f32_pow2((int)code - 127);
        const int64_t r1 = min(a.rows, band * 32 + 32);
        for (int64_t r = band * 32; r < r1; ++r) {
            const uint32_t b = a.data[r * a.K + c];
            const uint32_t mag = b & 0x7Fu;
            uint32_t f;
            bool nan;
            if constexpr (E5M2) {
                f = f32_mul((mag << 21) | ((b & 0x80u) << 24), 0x77800000u);
                nan = mag > 0x7Cu;
                if (mag == 0x7Cu) f = 0x7F800000u | ((b & 0x80u) << 24);
            } else {
                f = f32_mul((mag << 20) | ((b & 0x80u) << 24), 0x7B800000u);
                nan = mag == 0x7Fu;
            }
            uint32_t o = f32_mul(f, scale);
            if (nan || (o & 0x7FFFFFFFu) > 0x7F800000u) o = 0x7FC00000u;
            if constexpr (BF16OUT)
                static_cast<uint16_t*>(a.out)[r * a.K + c] = (uint16_t)((o + 0x7FFFu + ((o >> 16) & 1u)) >> 16);
            else
                static_cast<uint32_t*>(a.out)[r * a.K + c] = o;
        }
    }
}

// Dequantize of the columnwise form, K % 32 == 0 and 32-byte aligned rows:
// a CTA of 128 threads owns a 32-row band x 128 columns, four threads to a
// row.  The band's 128 column codes become bf16 multipliers 2^(code-127) in
// shared memory, built by every warp for itself when the scales are
// swizzled (the 128 codes share four lines, so the extra loads hit L1 and no
// CTA barrier is needed) and by warp 0 for the CTA otherwise (compact and
// padded codes lie in 128 lines).  Each element is placed into a bf16
// pattern as payload * 2^-120 (2^-112), multiplied exactly by 2^120 (2^112)
// and once by its column's multiplier -- one rounding of the exact product,
// as for the rowwise form.  Whether a column code is 255 (or, for fp32
// output, below the code under which products leave bf16's normal range) is
// one warp vote over the lanes that loaded the codes.  Such a chunk, or one
// with a NaN / Inf payload, takes the element-wise fp32 path.
// bf16 output: a thread takes one row's 32 columns of chunk q (one 32-byte
// payload load; four threads cover a row's 128 bytes, so a warp load reads
// whole lines).  fp32 output: thread q of a row takes columns 8q..8q+7 of
// each 32-column group, so that the four threads of a row store 128
// contiguous bytes per instruction (128 bytes per thread stored as four
// 32-byte pieces of one chunk touched 32 lines per warp store: 66.7 against
// 51.1 us on 8192 x 8192).  One band per CTA; 12 (bf16) / 10 (fp32) CTAs
// per SM.  8192 x 8192 to bf16: 31.0 us, against 33.9 us with the codes
// loaded once per CTA behind a barrier and tested code by code per thread.
constexpr int kDqThreads = 128;

template <bool E5M2, bool BF16OUT, bool PERWARP>
__global__ void __launch_bounds__(kDqThreads, BF16OUT ? 12 : 10) colwise_dequant_tile_kernel(DequantArgs a, int64_t bands) {
    // the multiplier words of chunk q at 16 q + 4 (q / 2) -- the four chunks'
    // words read by one warp instruction fall in different banks -- and the
    // codes, four columns per word: one copy per warp (PERWARP) or per CTA
    constexpr int kW = PERWARP ? kDqThreads / 32 : 1;
    __shared__ __align__(16) uint32_t colmul[kW][64 + 8];
    __shared__ __align__(16) uint32_t colcode[kW][32];
    __shared__ uint32_t slow_sh;
    const int t = threadIdx.x & 31, w = threadIdx.x >> 5, q = t & 3, rr = threadIdx.x >> 2;
    const int ww = PERWARP ? w : 0;
    const int64_t nbr = (a.rows + 31) >> 5, Cpt = (nbr + 3) & ~int64_t(3);
    const int64_t col0 = (int64_t)blockIdx.x * 128;
    const bool cvalid = col0 + 32 * q < a.K;
    constexpr uint32_t kMinCode = E5M2 ? 17u : 10u;  // fp32 output: smallest code kept on the bf16 path
    constexpr uint32_t fix = E5M2 ? 0x77807780u : 0x7B807B80u;  // 2^112 / 2^120, both halves
    // lane t loads the codes of columns cA .. cA + 3; their scale offsets without the band
    // term are coff + u * cstep (cA is a multiple of 4: in the swizzled layout the four
    // sit 16 bytes apart)
    const int64_t cA = col0 + 4 * t;
    int64_t coff, cstep;
    if (a.lay == 0) {
        coff = cA * nbr;
        cstep = nbr;
    } else if (a.lay == 1) {
        coff = cA * Cpt;
        cstep = Cpt;
    } else {
        coff = (cA >> 7) * (Cpt >> 2) * 512 + (cA & 31) * 16 + ((cA >> 5) & 3) * 4;
        cstep = 16;
    }
    const int mbase = 16 * (t >> 3) + 4 * (t >> 4) + 2 * (t & 7);  // multiplier words of columns cA..cA+3
    for (int64_t band = blockIdx.y; band < bands; band += gridDim.y) {
        const int64_t r = band * 32 + rr;
        const bool rvalid = cvalid && r < a.rows;
        // bf16 output: the row's 32 payload bytes of chunk q; fp32 output: bytes 8q..8q+7 of
        // each 32-column group gg in words 2gg, 2gg+1 (the four lanes of a row then store
        // 128 contiguous bytes per instruction).  In flight while the scales are prepared.
        uint32_t pw[8];
        if constexpr (BF16OUT) {
            if (rvalid) ld32(pw, a.data + r * a.K + col0 + 32 * q);
        } else {
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) {
                pw[2 * gg] = pw[2 * gg + 1] = 0u;
                if (r < a.rows && col0 + 32 * gg < a.K) ld8(pw[2 * gg], pw[2 * gg + 1], a.data + r * a.K + col0 + 32 * gg + 8 * q);
            }
        }
        uint32_t slowmask = 0u;  // bit 8q + j: lane 8q + j, which holds codes of chunk q, found a slow code
        if (PERWARP || w == 0) {
            uint32_t codes = 0u;
            if (cA < a.K) {  // K % 32 == 0: all four columns are in the tensor
                const uint8_t* sp = a.scales + coff + (a.lay == 2 ? ((band >> 2) << 9) + (band & 3) : band);
                codes = (uint32_t)sp[0] | ((uint32_t)sp[cstep] << 8) | ((uint32_t)sp[2 * cstep] << 16) |
                        ((uint32_t)sp[3 * cstep] << 24);
            }
            // a code 255 (a zero byte of ~codes) or, for fp32 output, a code below kMinCode:
            // the byte tests are exact for "some byte", which is all that is asked
            uint32_t bad = (~codes - 0x01010101u) & codes & 0x80808080u;
            if constexpr (!BF16OUT) bad |= (codes - 0x01010101u * kMinCode) & ~codes & 0x80808080u;
            slowmask = __ballot_sync(0xffffffffu, bad != 0u);
            colcode[ww][t] = codes;
            colmul[ww][mbase] = (bf16_scale_pair(codes & 0xFFu) & 0xFFFFu) | (bf16_scale_pair((codes >> 8) & 0xFFu) << 16);
            colmul[ww][mbase + 1] =
                (bf16_scale_pair((codes >> 16) & 0xFFu) & 0xFFFFu) | (bf16_scale_pair(codes >> 24) << 16);
            if (!PERWARP && t == 0) slow_sh = slowmask;
        }
        if constexpr (PERWARP) {
            __syncwarp();
        } else {
            __syncthreads();
            slowmask = slow_sh;
        }
        if constexpr (BF16OUT) {
            if (rvalid) {
                const bool slow = ((slowmask >> (8 * q)) & 0xFFu) != 0u;
                uint32_t sp = 0u;
#pragma unroll
                for (int k = 0; k < 8; ++k) sp |= special_bytes<E5M2>(pw[k]);
                char* op = static_cast<char*>(a.out) + (r * a.K + col0 + 32 * q) * 2;
                if (sp == 0u && !slow) {
                    const uint32_t* mw = colmul[ww] + 16 * q + 4 * (q >> 1);
                    uint32_t mreg[16];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint4 mm = *reinterpret_cast<const uint4*>(mw + 4 * m);
                        mreg[4 * m] = mm.x;
                        mreg[4 * m + 1] = mm.y;
                        mreg[4 * m + 2] = mm.z;
                        mreg[4 * m + 3] = mm.w;
                    }
#pragma unroll
                    for (int s8 = 0; s8 < 2; ++s8) {
                        uint32_t seg[8];
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            const int pidx = 8 * s8 + v;  // column pair within the chunk
                            const uint32_t pr = place_pair<E5M2>(pw[pidx >> 1], (pidx & 1) ? 0x4342u : 0x4140u);
                            seg[v] = bf2_mul(bf2_mul(pr, fix), mreg[pidx]);
                        }
                        st32(op + 32 * s8, seg);
                    }
                } else {
#pragma unroll 1
                    for (int s8 = 0; s8 < 2; ++s8) {
                        uint32_t seg[8];
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            uint32_t o = 0u;
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                const int e = 16 * s8 + 2 * v + hh;  // element of the chunk
                                const uint32_t code = (colcode[ww][8 * q + (e >> 2)] >> (8 * (e & 3))) & 0xFFu;
                                const uint32_t scale = code == 255u ? 0x7FC00000u : f32_pow2((int)code - 127);
                                const uint32_t f = decode_scaled<E5M2>((pw[e >> 2] >> (8 * (e & 3))) & 0xFFu, scale);
                                o |= bf16_rne(f) << (16 * hh);
                            }
                            seg[v] = o;
                        }
                        st32(op + 32 * s8, seg);
                    }
                }
            }
        } else if (r < a.rows) {
            // any slow code among the band's columns, or a NaN / Inf payload: element-wise
            uint32_t sp = 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) sp |= special_bytes<E5M2>(pw[k]);
            const bool slow = slowmask != 0u || sp != 0u;
            char* op = static_cast<char*>(a.out) + (r * a.K + col0 + 8 * q) * 4;
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) {
                if (col0 + 32 * gg >= a.K) break;
                uint32_t seg[8];
                if (!slow) {
                    // columns 32gg + 8q .. + 7: multiplier words 4q .. 4q + 3 of chunk gg
                    const uint4 mm = *reinterpret_cast<const uint4*>(colmul[ww] + 16 * gg + 4 * (gg >> 1) + 4 * q);
                    const uint32_t mreg[4] = {mm.x, mm.y, mm.z, mm.w};
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint32_t pr = place_pair<E5M2>(pw[2 * gg + (v >> 1)], (v & 1) ? 0x4342u : 0x4140u);
                        const uint32_t y = bf2_mul(bf2_mul(pr, fix), mreg[v]);
                        seg[2 * v] = y << 16;
                        seg[2 * v + 1] = y & 0xFFFF0000u;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t code = (colcode[ww][8 * gg + 2 * q + (j >> 2)] >> (8 * (j & 3))) & 0xFFu;
                        const uint32_t scale = code == 255u ? 0x7FC00000u : f32_pow2((int)code - 127);
                        seg[j] = decode_scaled<E5M2>((pw[2 * gg + (j >> 2)] >> (8 * (j & 3))) & 0xFFu, scale);
                    }
                }
                st32(op + 128 * gg, seg);
            }
        }
        // colmul / colcode / slow_sh are rewritten by the next band
        if constexpr (PERWARP)
            __syncwarp();
        else
            __syncthreads();
    }
}

bool aligned(const void* p, int64_t n) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)n) == 0; }

template <bool PERWARP>
cudaError_t launch_dequant_tile(const DequantArgs& a, bool e5, dim3 grid, int64_t bands, cudaStream_t s) {
    if (e5)
        a.out_bf16 ? colwise_dequant_tile_kernel<true, true, PERWARP><<<grid, kDqThreads, 0, s>>>(a, bands)
                   : colwise_dequant_tile_kernel<true, false, PERWARP><<<grid, kDqThreads, 0, s>>>(a, bands);
    else
        a.out_bf16 ? colwise_dequant_tile_kernel<false, true, PERWARP><<<grid, kDqThreads, 0, s>>>(a, bands)
                   : colwise_dequant_tile_kernel<false, false, PERWARP><<<grid, kDqThreads, 0, s>>>(a, bands);
    return cudaGetLastError();
}

template <Elt ELT, bool VEC, int DST>
cudaError_t launch_one(const ColwiseArgs& a, cudaStream_t s) {
    const int64_t nb = ceil_div(a.K, 32), bands = ceil_div(a.rows, 32);
    const int64_t gx = ceil_div(nb, kWarps);
    const unsigned gy = (unsigned)(bands < 65535 ? bands : 65535);
    colwise_kernel<ELT, VEC, DST><<<dim3((unsigned)gx, gy), kThreads, 0, s>>>(a, bands);
    return cudaGetLastError();
}

template <Elt ELT>
cudaError_t dispatch(const ColwiseArgs& a, cudaStream_t s) {
    const int es = ELT == Elt::BF16 ? 2 : 4;
    const bool vec = aligned(a.x, 32) && (a.ldx * es) % 32 == 0 && (a.K * es) % 32 == 0;
    const int dst = (aligned(a.data, 32) && a.K % 32 == 0) ? 2 : (aligned(a.data, 16) && a.K % 16 == 0) ? 1 : 0;
    if (!vec) return launch_one<ELT, false, 0>(a, s);
    if (a.K % 32 == 0 && aligned(a.data, 16)) {
        const int64_t bands = ceil_div(a.rows, 32), gx = ceil_div(ceil_div(a.K, 64), kTileWarps);
        const unsigned gy = (unsigned)(bands < 65535 ? bands : 65535);
        tile64_kernel<ELT><<<dim3((unsigned)gx, gy), 32 * kTileWarps, 0, s>>>(a, bands);
        return cudaGetLastError();
    }
    if (dst == 2) return launch_one<ELT, true, 2>(a, s);
    if (dst == 1) return launch_one<ELT, true, 1>(a, s);
    return launch_one<ELT, true, 0>(a, s);
}

}  // namespace

cudaError_t launch_colwise(Elt elt, const ColwiseArgs& a, cudaStream_t s) {
    return elt == Elt::BF16 ? dispatch<Elt::BF16>(a, s) : dispatch<Elt::FP32>(a, s);
}

cudaError_t launch_colwise_dequant(const DequantArgs& a, cudaStream_t s) {
    const bool e5 = a.fp8 == 1;
    const int oes = a.out_bf16 ? 2 : 4;
    if (a.K % 32 == 0 && aligned(a.data, 32) && aligned(a.out, 32) && (a.K * oes) % 32 == 0) {
        // swizzled scales: every warp loads the band's codes itself (they share 4 lines);
        // compact / padded ones lie in 128 different lines, loaded once per CTA
        const int64_t bands = ceil_div(a.rows, 32), gx = ceil_div(a.K, 128);
        const dim3 grid((unsigned)gx, (unsigned)(bands < 65535 ? bands : 65535));
        if (a.lay == 2)
            return launch_dequant_tile<true>(a, e5, grid, bands, s);
        return launch_dequant_tile<false>(a, e5, grid, bands, s);
    }
    const int64_t total = ceil_div(a.rows, 32) * a.K;
    int64_t grid = ceil_div(total, (int64_t)kThreads);
    const int64_t cap = (int64_t)sm_count() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    if (e5)
        a.out_bf16 ? colwise_dequant_kernel<true, true><<<(unsigned)grid, kThreads, 0, s>>>(a)
                   : colwise_dequant_kernel<true, false><<<(unsigned)grid, kThreads, 0, s>>>(a);
    else
        a.out_bf16 ? colwise_dequant_kernel<false, true><<<(unsigned)grid, kThreads, 0, s>>>(a)
                   : colwise_dequant_kernel<false, false><<<(unsigned)grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace mxq
