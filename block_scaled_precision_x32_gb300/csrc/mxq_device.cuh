// mxq_device.cuh -- device-side arithmetic shared by the libmxq kernels.
//
// Every rounding here is IEEE round-to-nearest-even on operands for which
// the rounded result is the exact answer of the method, so the kernels need
// no special-case integer code.  All floating-point instructions are inline
// PTX with an explicit .rn and no .ftz: nvcc never contracts or flushes
// them, so a --use_fast_math build gives the same bytes.
#pragma once

#include <cstdint>

namespace mxq {

// ------------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf2_min(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// max(|a|, |b|) per half, NaN if either is NaN (the sign bit of the result
// is the xor of the signs and is ignored by the callers).
__device__ __forceinline__ uint32_t bf2_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t f32_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t u16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t f32_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t f32_add(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t f32_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t f32_min(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.f32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// Two fp32 values -> two E4M3 bytes, round to nearest even, subnormals
// included; `hi` goes to bits 15..8, `lo` to bits 7..0.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(uint32_t hi, uint32_t lo) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "r"(hi), "r"(lo));
    return d;
}
// Two fp32 values -> two E2M1 codes (round to nearest even, saturating at
// +-6, sign in bit 3); `hi` goes to bits 7..4, `lo` to bits 3..0.
__device__ __forceinline__ uint32_t e2m1x2_from_f32(uint32_t hi, uint32_t lo) {
    uint32_t d;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(d) : "r"(hi), "r"(lo));
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// 32-byte global loads and stores (one full sector per lane).  The load
// skips L1 allocation; it is coherent, so in-place projection is safe.
__device__ __forceinline__ void ld32(uint32_t (&w)[8], const void* p) {
    asm volatile("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
__device__ __forceinline__ void st32(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void st16(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint32_t lop_select(uint32_t a, uint32_t b, uint32_t mask) {
    // (a & mask) | (b & ~mask), one LOP3
    return (a & mask) | (b & ~mask);
}

// Row and block of a flattened (row, block) index: q = i / n, i - q n, by one
// 32-bit division when both fit in 32 bits (the usual case; a 64-bit division
// is several times longer), else by a 64-bit one.
__device__ __forceinline__ void split_index(int64_t i, int64_t n, int64_t& q, int64_t& rem) {
    if ((((uint64_t)i | (uint64_t)n) >> 32) == 0) {
        const uint32_t q32 = (uint32_t)i / (uint32_t)n;
        q = q32;
        rem = (int64_t)((uint32_t)i - q32 * (uint32_t)n);
    } else {
        q = i / n;
        rem = i - q * n;
    }
}

// ------------------------------------------------------ block scale rule

// e = clamp(ceil(log2(amax/6)), -126, 125) from the magnitude pattern of a
// finite amax (TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling
// recipes", Description, mode 1).  amax = (1 + f) * 2^E gives E - 2 when
// f <= 1/2, else E - 1; zero and subnormal amax clamp to -126.
// The packed MXFP4 form keeps the rule but clamps above at 126 (TOP).
template <int MANT, int TOP = 125>
__device__ __forceinline__ int block_exponent(uint32_t amax_mag) {
    const int E = (int)(amax_mag >> MANT);
    const uint32_t frac = amax_mag & ((1u << MANT) - 1u);
    int e = E - 129 + (frac > (1u << (MANT - 1)) ? 1 : 0);
    e = E == 0 ? -126 : e;
    return min(max(e, -126), TOP);
}

// ------------------------------------------------ E2M1 grid rounding, bf16

// Elements x (two bf16 patterns, signed) of a block with exponent e are
// scaled into v = x * 2^-e (exact whenever |v| can round to a nonzero grid
// point: then |v| >= 2^-2 is a normal bf16) and rounded to the signed E2M1
// grid {0, .5, 1, 1.5, 2, 3, 4, 6} by adding and subtracting
// c = 1.5 * 2^(6 + max(exp|v|, 0)).  For |v| < 2, in [2, 4) and in [4, 8)
// the sum v + c stays inside one binade of c whose unit in the last place
// is 0.5, 1 and 2 -- the grid spacing there -- and c / ulp = 192 is even, so
// round-to-nearest-even of the sum ties to the even grid multiple, which is
// the even E2M1 code.  A result of +-8 (|v| >= 7) occurs only at the upper
// clamp e = 125 and is saturated by the caller.  A zero result may carry the
// wrong sign; callers OR the input's sign back in.
struct Bf16Grid {
    uint32_t mult;  // v = x * mult: 2^-e, or 2^-e * 2^s for a shifted domain
    uint32_t floor; // 1.0 in v units (both halves)
};

__device__ __forceinline__ uint32_t bf2_grid(uint32_t x, const Bf16Grid& g) {
    const uint32_t v = bf2_mul(x, g.mult);
    const uint32_t c = bf2_max(v & 0x7F807F80u, g.floor) + 0x03400340u;  // * 96
    return bf2_sub(bf2_add(v, c), c);
}

// Clamp a signed grid value (in units of `one`) to [-6, 6]: sat6 = 6 * one.
__device__ __forceinline__ uint32_t bf2_sat(uint32_t t, uint32_t sat6) {
    return bf2_max(bf2_min(t, sat6), sat6 | 0x80008000u);
}

__device__ __forceinline__ uint32_t bf16_pow2_pair(int k) {  // 2^k, k in [-126, 127]
    const uint32_t p = (uint32_t)(k + 127) << 7;
    return p | (p << 16);
}

// Grid in the v = x / 2^e domain.
__device__ __forceinline__ Bf16Grid bf16_grid_unit(int e) {
    Bf16Grid g;
    g.mult = bf16_pow2_pair(-e);
    g.floor = 0x3F803F80u;  // 1.0
    return g;
}

// ------------------------------------------------ E2M1 grid rounding, fp32

// Same construction with fp32: c = 1.5 * 2^(22 + max(exp|v|, 0)).
__device__ __forceinline__ uint32_t f32_grid(uint32_t x, uint32_t mult) {
    const uint32_t v = f32_mul(x, mult);
    const uint32_t c = max(v & 0x7F800000u, 0x3F800000u) + (22u << 23) + 0x00400000u;
    return f32_sub(f32_add(v, c), c);
}

__device__ __forceinline__ uint32_t f32_sat(uint32_t t) {  // clamp to [-6, 6]
    uint32_t d;
    asm("{ .reg .f32 a; min.f32 a, %1, 0f40C00000; max.f32 %0, a, 0fC0C00000; }" : "=r"(d) : "r"(t));
    return d;
}

__device__ __forceinline__ uint32_t f32_pow2(int k) {  // 2^k, k in [-127, 127]
    return k >= -126 ? (uint32_t)(k + 127) << 23 : 0x00400000u;
}

// ------------------------------------------- E2M1 grid -> E4M3 bytes (fp32)

// Four fp32 elements x of a block with exponent e, and a payload shift d
// in [-5, 6]: v = x * 2^-e is rounded onto the signed E2M1 grid by the
// hardware conversion (round to nearest even -- ties to the even code --
// saturating at +-6, the sign kept, -0 included), and each code c becomes
// the E4M3 byte of p(c) * 2^d, every nonzero one an exact E4M3 normal.
// The bytes come from an 8-entry table indexed by PRMT on the code's
// magnitude: entry c is the byte of p(c) (0.5 -> 0x30 ... 6 -> 0x4C) plus
// 8d in the exponent field; the sign goes to bit 7 through a second PRMT
// that replicates it.
struct E4m3Table {
    uint32_t lo, hi;
};

__device__ __forceinline__ E4m3Table e4m3_table(int d) {
    const uint32_t d8 = (uint32_t)(8 * d);
    E4m3Table t;
    t.lo = 0x3C383000u + d8 * 0x01010100u;  // codes 0..3: 0, 0.5, 1, 1.5 (code 0 stays 0)
    t.hi = 0x4C484440u + d8 * 0x01010101u;  // codes 4..7: 2, 3, 4, 6
    return t;
}

__device__ __forceinline__ uint32_t e4m3x4_from_grid(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, uint32_t mult,
                                                     const E4m3Table& t) {
    const uint32_t n = e2m1x2_from_f32(f32_mul(x1, mult), f32_mul(x0, mult)) |
                       (e2m1x2_from_f32(f32_mul(x3, mult), f32_mul(x2, mult)) << 8);  // codes of x0..x3 in nibbles 0..3
    const uint32_t mag = prmt(t.lo, t.hi, n & 0x7777u);
    const uint32_t sg = ((prmt(0x80808080u, 0x80808080u, n) & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) & 0x80808080u;
    return mag | sg;
}

// ------------------------------------------------------ fp8 payload decode

// fp8 byte -> exact fp32 pattern times `scale` (IEEE fp32 product), NaN made canonical.
template <bool E5M2>
__device__ __forceinline__ uint32_t decode_scaled(uint32_t b, uint32_t scale) {
    const uint32_t mag = b & 0x7Fu;
    uint32_t f;
    bool nan;
    if constexpr (E5M2) {
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

// Any byte of w a NaN/Inf payload?  (E4M3: low 7 bits all ones; E5M2:
// exponent all ones.)
template <bool E5M2>
__device__ __forceinline__ uint32_t special_bytes(uint32_t w) {
    if constexpr (E5M2)
        return ((w & 0x7C7C7C7Cu) + 0x04040404u) & 0x80808080u;
    else
        return ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
}

// Payload bytes (lo, hi) of one word's pair -> bf16x2 of payload * 2^-120 / 2^-112.
template <bool E5M2>
__device__ __forceinline__ uint32_t place_pair(uint32_t w, uint32_t sel) {
    const uint32_t t = prmt(w, 0u, sel);  // byte k of the pair at bits 16k..16k+7
    constexpr int SH = E5M2 ? 5 : 4;
    return ((t & 0x007F007Fu) << SH) | ((t & 0x00800080u) << 8);
}

// bf16x2 2^(code - 127) for a UE8M0 code in 0..254 (code 0: the bf16 subnormal 2^-127).
__device__ __forceinline__ uint32_t bf16_scale_pair(uint32_t code) {
    return code == 0u ? 0x00400040u : ((code << 7) | (code << 23));
}

}  // namespace mxq
