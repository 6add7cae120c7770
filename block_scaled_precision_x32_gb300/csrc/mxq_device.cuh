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
// 32-byte loads with an L1 eviction hint: "keep" for a first read whose
// lines are read again soon, "drop" for that second, last read.
__device__ __forceinline__ void ld32_keep(uint32_t (&w)[8], const void* p) {
    asm volatile("ld.global.L1::evict_last.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
__device__ __forceinline__ void ld32_drop(uint32_t (&w)[8], const void* p) {
    asm volatile("ld.global.L1::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
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

// ------------------------------------------------------ block scale rule

// e = clamp(ceil(log2(amax/6)), -126, 125) from the magnitude pattern of a
// finite amax (TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling
// recipes", Description, mode 1).  amax = (1 + f) * 2^E gives E - 2 when
// f <= 1/2, else E - 1; zero and subnormal amax clamp to -126.
template <int MANT>
__device__ __forceinline__ int block_exponent(uint32_t amax_mag) {
    const int E = (int)(amax_mag >> MANT);
    const uint32_t frac = amax_mag & ((1u << MANT) - 1u);
    int e = E - 129 + (frac > (1u << (MANT - 1)) ? 1 : 0);
    e = E == 0 ? -126 : e;
    return min(max(e, -126), 125);
}

// ------------------------------------------------ E2M1 grid rounding, bf16

// Magnitudes a (two bf16 patterns, sign cleared) of a block with exponent e
// are scaled into v = a * 2^-e (exact: v >= 2^-126 whenever it can round to
// a nonzero grid point) and rounded to the E2M1 grid {0, .5, 1, 1.5, 2, 3,
// 4, 6} by one add and one subtract of c = 2^(6 + max(exp(v), 0)): the sum
// v + c has unit in the last place 0.5 for v < 2, 1 for v in [2, 4) and 2
// for v in [4, 8) -- the grid spacing -- and its ties go to an even
// significand, which is the even E2M1 code.  A result of 8 (v >= 7, only
// possible at the upper clamp e = 125) saturates to 6.
struct Bf16Grid {
    uint32_t mult;  // v = a * mult: 2^-e, or 2^-e * 2^s for a shifted domain
    uint32_t floor; // smallest power of two allowed for c / 64: 2^0 in v units
    uint32_t sat;   // 6 in v units
};

__device__ __forceinline__ uint32_t bf2_grid(uint32_t a, const Bf16Grid& g) {
    const uint32_t v = bf2_mul(a, g.mult);
    const uint32_t c = bf2_max(v & 0x7F807F80u, g.floor) + 0x03000300u;  // * 64
    return bf2_min(bf2_sub(bf2_add(v, c), c), g.sat);
}

__device__ __forceinline__ uint32_t bf16_pow2_pair(int k) {  // 2^k, k in [-126, 127]
    const uint32_t p = (uint32_t)(k + 127) << 7;
    return p | (p << 16);
}

// Grid in the v = |x| / 2^e domain.
__device__ __forceinline__ Bf16Grid bf16_grid_unit(int e) {
    Bf16Grid g;
    g.mult = bf16_pow2_pair(-e);
    g.floor = 0x3F803F80u;  // 1.0
    g.sat = 0x40C040C0u;    // 6.0
    return g;
}

// ------------------------------------------------ E2M1 grid rounding, fp32

// Same construction with fp32 (c = 2^(22 + max(exp(v), 0))).
__device__ __forceinline__ uint32_t f32_grid(uint32_t a, uint32_t mult) {
    const uint32_t v = f32_mul(a, mult);
    const uint32_t c = max(v & 0x7F800000u, 0x3F800000u) + (22u << 23);
    return f32_min(f32_sub(f32_add(v, c), c), 0x40C00000u);
}

__device__ __forceinline__ uint32_t f32_pow2(int k) {  // 2^k, k in [-127, 127]
    return k >= -126 ? (uint32_t)(k + 127) << 23 : 0x00400000u;
}

}  // namespace mxq
