/*
 * mxq_oracle.c -- plain, slow CPU oracle for block-scaled weight conversion.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the package smoke check and the
 * CPU-baseline leg of the benchmark use it.  It shares no code, header,
 * table or constant with the CUDA library; the two meet only on the bytes
 * of seeded inputs and outputs.
 *
 * What it computes, and where each rule comes from:
 *
 *  - "TE PR #3264: MXFP4 weight QAT on MXFP8 and FP8 block-scaling recipes",
 *    Description, mode 1 (Projection): every 1x32 block along the last
 *    dimension gets the scale 2^clamp(ceil(log2(amax/6)), -126, 125), taken
 *    from the bit pattern of amax, and each element is rounded to nearest
 *    (ties to even) onto the E2M1 grid {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *  - Same page, Description, mode 2 (Direct): MXFP8 rowwise is the fixed
 *    shift-6 lift (E4M3 payload p*2^6, UE8M0 scale 2^(e-6), the scale
 *    clamping at code 0 = 2^-127 while the payload absorbs the rest); the
 *    128x128 blockwise form uses the tile scale 2^(max_b e_b - 6) clamped at
 *    2^-127 and rounds each p*2^(e_b - T) to nearest-even E4M3, subnormals
 *    included.
 *  - Same page, Description (API paragraph): UE8M0 code 0 decodes to 2^-127
 *    and code 255 to NaN.
 *  - Same page, "Test results (B200)": non-finite values poison their block;
 *    "Known limitations": the projection saturates at 6*2^125.
 *  - "TE PR #3790: MXFP8TensorStorage.export_components()", Description:
 *    compact uint8 scales of shape (rows, ceil(K/32)), a short last block
 *    keeping its own scale, padding and the GEMM swizzle removed.
 *
 * Method.  Every bf16/fp32/fp8 value is decoded from its IEEE bit fields
 * into an exact double (all of them fit).  The scale exponent is read off
 * the amax bit pattern, as the pages say.  Rounding steps are the
 * definitions written out: the nearest point of a finite grid, found by
 * comparing distances, ties going to the even code.  Those distances are
 * exact in double: a value v of at most 24 significant bits that is >= 2^-3
 * differs from a multiple of 2^-9 by a multiple of 2^-26 below 2^9, which
 * needs < 35 bits; below 2^-3 the grid point 0 is strictly nearest on the
 * E2M1 grid.  For the E4M3 grid the same holds with the subnormal step 2^-9.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - a poisoned block projects to the canonical quiet NaN (bf16 0x7FC0,
 *    fp32 0x7FC00000); its MXFP8 scale code is 0xFF and its payloads 0x7F;
 *    in the blockwise form its payloads are 0x7F and it is left out of the
 *    tile maximum (a tile with no finite block takes T = -127);
 *  - the sign of zero is kept (a negative input that rounds to 0 gives -0);
 *  - a zero or subnormal amax gives e = -126 (the lower clamp);
 *  - the blockwise tile scale is stored as the fp32 scale_inv = 2^T;
 *  - padded scale buffers have ceil(rows/128)*128 rows and ceil(nb/4)*4
 *    columns; padding bytes are written as 0;
 *  - the GEMM-swizzled layout is the public cuBLAS 128x4 block-scaling
 *    layout: byte (r, j) sits at ((r/128)*(Cp/4) + j/4)*512
 *    + (r%32)*16 + ((r%128)/32)*4 + j%4, with Cp the padded column count;
 *  - dequantize returns fp32 = round-to-nearest(payload * scale), and bf16
 *    as one more round-to-nearest-even of that fp32; every NaN result is
 *    the canonical quiet NaN above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_BF16 0
#define OR_FP32 1

#define OR_E4M3 0
#define OR_E5M2 1

#define OR_COMPACT 0
#define OR_PADDED 1
#define OR_SWIZZLED 2

#define OR_OK 0
#define OR_BAD 1

/* ---------------------------------------------------------------- fields */

typedef struct {
    int mant_bits; /* stored mantissa bits */
    int exp_bits;
    int bias;
} ieee_fmt;

static ieee_fmt fmt_of(int dt) {
    ieee_fmt f;
    if (dt == OR_BF16) {
        f.mant_bits = 7;
        f.exp_bits = 8;
        f.bias = 127;
    } else {
        f.mant_bits = 23;
        f.exp_bits = 8;
        f.bias = 127;
    }
    return f;
}

static uint32_t load_bits(const void* base, int dt, int64_t idx) {
    if (dt == OR_BF16) return ((const uint16_t*)base)[idx];
    return ((const uint32_t*)base)[idx];
}

static void store_bits(void* base, int dt, int64_t idx, uint32_t bits) {
    if (dt == OR_BF16)
        ((uint16_t*)base)[idx] = (uint16_t)bits;
    else
        ((uint32_t*)base)[idx] = bits;
}

static int is_nonfinite(uint32_t bits, int dt) {
    ieee_fmt f = fmt_of(dt);
    uint32_t e = (bits >> f.mant_bits) & ((1u << f.exp_bits) - 1u);
    return e == (1u << f.exp_bits) - 1u;
}

static int sign_of(uint32_t bits, int dt) {
    ieee_fmt f = fmt_of(dt);
    return (int)((bits >> (f.mant_bits + f.exp_bits)) & 1u);
}

static uint32_t magnitude_bits(uint32_t bits, int dt) {
    ieee_fmt f = fmt_of(dt);
    return bits & ((1u << (f.mant_bits + f.exp_bits)) - 1u);
}

/* |value| of a finite pattern, from its fields, as an exact double. */
static double abs_value(uint32_t bits, int dt) {
    ieee_fmt f = fmt_of(dt);
    uint32_t m = bits & ((1u << f.mant_bits) - 1u);
    int e = (int)((bits >> f.mant_bits) & ((1u << f.exp_bits) - 1u));
    if (e == 0) return ldexp((double)m, 1 - f.bias - f.mant_bits);
    return ldexp((double)((1u << f.mant_bits) + m), e - f.bias - f.mant_bits);
}

/* The pattern of a double that the caller knows to be exactly
 * representable in dt; aborts if it is not (a self-check of the oracle). */
static uint32_t encode_exact(double v, int dt) {
    float fv = (float)v;
    if ((double)fv != v) abort();
    uint32_t u;
    memcpy(&u, &fv, 4);
    if (dt == OR_FP32) return u;
    if (u & 0xFFFFu) abort();
    return u >> 16;
}

static uint32_t canonical_nan(int dt) { return dt == OR_BF16 ? 0x7FC0u : 0x7FC00000u; }

/* ------------------------------------------------------ MXFP4 decomposition */

/* ceil(log2(amax/6)) from the amax bit pattern (TE PR #3264, Description,
 * mode 1: the scale is "derived from the amax bit pattern").
 *
 * With amax = (1 + m/2^M) * 2^E normal, amax/6 lies in
 * [2^(E-2)/1.5, 2^(E-1)/1.5), so ceil(log2(amax/6)) = E - 2 when
 * 1 + m/2^M <= 1.5 and E - 1 otherwise.  A zero or subnormal amax sits below
 * 6*2^-129; it is returned as -1000, below every clamp. */
static int ceil_log2_amax_over_6(uint32_t amax_mag_bits, int dt) {
    ieee_fmt f = fmt_of(dt);
    uint32_t m = amax_mag_bits & ((1u << f.mant_bits) - 1u);
    int E = (int)(amax_mag_bits >> f.mant_bits);
    if (E == 0) return -1000;
    uint32_t half = 1u << (f.mant_bits - 1);
    return (E - f.bias) - 2 + (m > half ? 1 : 0);
}

/* Block scale exponent of the projection: clamp(ceil(log2(amax/6)), -126, 125). */
static int block_exponent(uint32_t amax_mag_bits, int dt) {
    int e = ceil_log2_amax_over_6(amax_mag_bits, dt);
    if (e < -126) e = -126;
    if (e > 125) e = 125;
    return e;
}

static const double E2M1_GRID[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Round v >= 0 to the nearest E2M1 grid point, ties to the even code
 * (TE PR #3264, Description, mode 1: "RTNE onto E2M1").  Values above 6 go
 * to 6, which is the nearest grid point ("Known limitations": saturation at
 * 6*2^125).  Returns the code 0..7. */
static int e2m1_rtne_code(double v) {
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        double dc = fabs(v - E2M1_GRID[c]);
        double db = fabs(v - E2M1_GRID[best]);
        if (dc < db || (dc == db && (c % 2) == 0)) best = c;
    }
    return best;
}

typedef struct {
    int poisoned;
    int e; /* block scale exponent */
} block_info;

/* Scan one 1x32 block (the last may be shorter, TE PR #3790 Description). */
static block_info scan_block(const void* row, int dt, int64_t j0, int64_t j1) {
    block_info b;
    uint32_t amax = 0;
    b.poisoned = 0;
    for (int64_t i = j0; i < j1; ++i) {
        uint32_t bits = load_bits(row, dt, i);
        if (is_nonfinite(bits, dt)) b.poisoned = 1;
        uint32_t mag = magnitude_bits(bits, dt);
        /* for finite patterns the magnitude order is the integer order */
        if (mag > amax) amax = mag;
    }
    b.e = b.poisoned ? 0 : block_exponent(amax, dt);
    return b;
}

/* E2M1 code and sign of one finite element of a block with exponent e. */
static int element_code(uint32_t bits, int dt, int e) {
    double v = ldexp(abs_value(bits, dt), -e); /* exact: a power-of-two scaling */
    return e2m1_rtne_code(v);
}

int oracle_block_exponent(uint32_t amax_mag_bits, int dt) { return block_exponent(amax_mag_bits, dt); }

int oracle_e2m1_rtne_code(double v) { return e2m1_rtne_code(v); }

/* ------------------------------------------------------------ projection */

/* y = sign(x) * p * 2^e per element, p the E2M1 grid value (TE PR #3264,
 * Description, mode 1).  ldx/ldy are row strides in elements. */
int oracle_fake_quant_mxfp4(const void* x, void* y, int dt, int64_t rows, int64_t K, int64_t ldx,
                            int64_t ldy) {
    if (dt != OR_BF16 && dt != OR_FP32) return OR_BAD;
    size_t es = dt == OR_BF16 ? 2 : 4;
    for (int64_t r = 0; r < rows; ++r) {
        const char* xr = (const char*)x + (size_t)(r * ldx) * es;
        char* yr = (char*)y + (size_t)(r * ldy) * es;
        for (int64_t j0 = 0; j0 < K; j0 += 32) {
            int64_t j1 = j0 + 32 < K ? j0 + 32 : K;
            block_info b = scan_block(xr, dt, j0, j1);
            for (int64_t i = j0; i < j1; ++i) {
                uint32_t bits = load_bits(xr, dt, i);
                if (b.poisoned) {
                    store_bits(yr, dt, i, canonical_nan(dt));
                    continue;
                }
                int c = element_code(bits, dt, b.e);
                double mag = ldexp(E2M1_GRID[c], b.e);
                double val = sign_of(bits, dt) ? -mag : mag;
                if (c == 0) val = sign_of(bits, dt) ? -0.0 : 0.0;
                store_bits(yr, dt, i, encode_exact(val, dt));
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------- fp8 codes */

/* Value of an fp8 byte from its fields (E4M3: bias 7, no Inf, S.1111.111 is
 * NaN; E5M2: bias 15, exponent 31 is Inf (m = 0) or NaN). */
double oracle_fp8_value(uint8_t b, int kind) {
    int s = b >> 7;
    double v;
    if (kind == OR_E4M3) {
        int E = (b >> 3) & 15, m = b & 7;
        if (E == 15 && m == 7) return NAN;
        v = E == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), E - 10);
    } else {
        int E = (b >> 2) & 31, m = b & 3;
        if (E == 31) {
            if (m) return NAN;
            v = INFINITY;
        } else {
            v = E == 0 ? ldexp((double)m, -16) : ldexp((double)(4 + m), E - 17);
        }
    }
    return s ? -v : v;
}

/* Round a finite double to the nearest E4M3 value, ties to the even code
 * (even mantissa), subnormals included (TE PR #3264, Description, mode 2:
 * "RTNE onto E4M3 incl. subnormals").  The sign is kept for zero.  The
 * blockwise lift never exceeds 384; larger inputs are not used. */
uint8_t oracle_e4m3_rtne(double u) {
    int neg = signbit(u) ? 1 : 0;
    double a = fabs(u);
    int best = 0;
    for (int c = 1; c < 127; ++c) {
        double dc = fabs(a - oracle_fp8_value((uint8_t)c, OR_E4M3));
        double db = fabs(a - oracle_fp8_value((uint8_t)best, OR_E4M3));
        if (dc < db || (dc == db && (c % 2) == 0)) best = c;
    }
    return (uint8_t)(best | (neg << 7));
}

/* E4M3 byte whose value is exactly u (the caller knows one exists). */
static uint8_t e4m3_exact(double u) {
    uint8_t b = oracle_e4m3_rtne(u);
    if (oracle_fp8_value(b, OR_E4M3) != u) abort();
    return b;
}

/* UE8M0 scale byte: code c < 255 is 2^(c-127), code 0 being 2^-127, and 255
 * is NaN (TE PR #3264, Description: the exp2f(e8m0) fix). */
double oracle_e8m0_value(uint8_t c) {
    if (c == 255) return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* --------------------------------------------------------- scale layouts */

int64_t oracle_scale_cols(int64_t K) { return (K + 31) / 32; }

/* Byte offset of scale (r, j) in a layout whose padded column count is Cp.
 * Swizzled: the cuBLAS block-scaling-factor layout of 128x4 tiles of 512
 * bytes, tiles in row-major order. */
int64_t oracle_scale_offset(int64_t r, int64_t j, int64_t nb, int lay) {
    int64_t Cp = (nb + 3) / 4 * 4;
    if (lay == OR_COMPACT) return r * nb + j;
    if (lay == OR_PADDED) return r * Cp + j;
    return ((r / 128) * (Cp / 4) + j / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4);
}

int64_t oracle_scale_bytes(int64_t rows, int64_t K, int lay) {
    int64_t nb = oracle_scale_cols(K);
    if (lay == OR_COMPACT) return rows * nb;
    return (rows + 127) / 128 * 128 * ((nb + 3) / 4 * 4);
}

/* Place compact scales into a layout; padding bytes are 0. */
int oracle_scales_to_layout(const uint8_t* compact, int64_t rows, int64_t K, int lay, uint8_t* out) {
    int64_t nb = oracle_scale_cols(K);
    memset(out, 0, (size_t)oracle_scale_bytes(rows, K, lay));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < nb; ++j) out[oracle_scale_offset(r, j, nb, lay)] = compact[r * nb + j];
    return OR_OK;
}

/* ------------------------------------------------------ direct MXFP8 row */

/* Fixed-shift-6 lift (TE PR #3264, Description, mode 2): the UE8M0 code of
 * 2^(e-6) is e+121; below 0 it clamps to 0 (2^-127) and the payload
 * p*2^e / 2^(code-127) absorbs the rest exactly.  data is [rows, K]
 * contiguous; scales is compact [rows, ceil(K/32)]. */
int oracle_mxfp8_row_direct(const void* x, int dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* data,
                            uint8_t* scales) {
    if (dt != OR_BF16 && dt != OR_FP32) return OR_BAD;
    size_t es = dt == OR_BF16 ? 2 : 4;
    int64_t nb = oracle_scale_cols(K);
    for (int64_t r = 0; r < rows; ++r) {
        const char* xr = (const char*)x + (size_t)(r * ldx) * es;
        for (int64_t j0 = 0; j0 < K; j0 += 32) {
            int64_t j1 = j0 + 32 < K ? j0 + 32 : K;
            block_info b = scan_block(xr, dt, j0, j1);
            if (b.poisoned) {
                scales[r * nb + j0 / 32] = 0xFF;
                for (int64_t i = j0; i < j1; ++i) data[r * K + i] = 0x7F;
                continue;
            }
            int code = b.e + 121;
            if (code < 0) code = 0;
            scales[r * nb + j0 / 32] = (uint8_t)code;
            for (int64_t i = j0; i < j1; ++i) {
                uint32_t bits = load_bits(xr, dt, i);
                int c = element_code(bits, dt, b.e);
                double q = ldexp(E2M1_GRID[c], b.e - (code - 127));
                if (sign_of(bits, dt)) q = -q;
                if (c == 0) q = sign_of(bits, dt) ? -0.0 : 0.0;
                data[r * K + i] = e4m3_exact(q);
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------ direct FP8 128x128 tiles */

/* Per-tile exponent folding (TE PR #3264, Description, mode 2): with e_b the
 * exponent of each 1x32 block of the tile, T = max(max_b e_b - 6, -127) and
 * each payload is RTNE_E4M3(p * 2^(e_b - T)).  data is [rows, K]
 * contiguous; tile_scale_inv is [ceil(rows/128), ceil(K/128)] of 2^T. */
int oracle_fp8_block128_direct(const void* x, int dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* data,
                               float* tile_scale_inv) {
    if (dt != OR_BF16 && dt != OR_FP32) return OR_BAD;
    size_t es = dt == OR_BF16 ? 2 : 4;
    int64_t tr = (rows + 127) / 128, tc = (K + 127) / 128;
    for (int64_t ti = 0; ti < tr; ++ti) {
        for (int64_t tj = 0; tj < tc; ++tj) {
            int64_t r0 = ti * 128, r1 = r0 + 128 < rows ? r0 + 128 : rows;
            int64_t c0 = tj * 128, c1 = c0 + 128 < K ? c0 + 128 : K;
            int emax = -126, any = 0;
            for (int64_t r = r0; r < r1; ++r) {
                const char* xr = (const char*)x + (size_t)(r * ldx) * es;
                for (int64_t j0 = c0; j0 < c1; j0 += 32) {
                    int64_t j1 = j0 + 32 < c1 ? j0 + 32 : c1;
                    block_info b = scan_block(xr, dt, j0, j1);
                    if (b.poisoned) continue;
                    if (!any || b.e > emax) emax = b.e;
                    any = 1;
                }
            }
            int T = emax - 6;
            if (T < -127) T = -127;
            tile_scale_inv[ti * tc + tj] = (float)ldexp(1.0, T);
            for (int64_t r = r0; r < r1; ++r) {
                const char* xr = (const char*)x + (size_t)(r * ldx) * es;
                for (int64_t j0 = c0; j0 < c1; j0 += 32) {
                    int64_t j1 = j0 + 32 < c1 ? j0 + 32 : c1;
                    block_info b = scan_block(xr, dt, j0, j1);
                    for (int64_t i = j0; i < j1; ++i) {
                        if (b.poisoned) {
                            data[r * K + i] = 0x7F;
                            continue;
                        }
                        uint32_t bits = load_bits(xr, dt, i);
                        int c = element_code(bits, dt, b.e);
                        double u = ldexp(E2M1_GRID[c], b.e - T);
                        if (sign_of(bits, dt)) u = -u;
                        if (c == 0) u = sign_of(bits, dt) ? -0.0 : 0.0;
                        data[r * K + i] = oracle_e4m3_rtne(u);
                    }
                }
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------- dequantize */

/* Nearest bf16 of an fp32 pattern, ties to even; the bf16 pattern 0x7F80
 * counts as 2^128 so that overflow goes to Inf as IEEE rounding does. */
static double bf16_value_for_rounding(uint32_t b16) {
    uint32_t mag = b16 & 0x7FFFu;
    double v = mag == 0x7F80u ? ldexp(1.0, 128) : abs_value(mag, OR_BF16);
    return v;
}

uint16_t oracle_f32_to_bf16(uint32_t f32_bits) {
    if (is_nonfinite(f32_bits, OR_FP32)) {
        if (f32_bits & 0x7FFFFFu) return 0x7FC0u;
        return (uint16_t)(f32_bits >> 16);
    }
    uint32_t s = f32_bits & 0x80000000u;
    double a = abs_value(f32_bits & 0x7FFFFFFFu, OR_FP32);
    uint32_t lo = (f32_bits & 0x7FFFFFFFu) >> 16; /* truncation: below or equal */
    uint32_t hi = lo + 1;
    double dlo = a - bf16_value_for_rounding(lo);
    double dhi = bf16_value_for_rounding(hi) - a;
    uint32_t pick = (dlo < dhi || (dlo == dhi && (lo % 2) == 0)) ? lo : hi;
    return (uint16_t)((s >> 16) | pick);
}

static void store_result(void* out, int out_dt, int64_t idx, double prod) {
    float f;
    uint32_t u;
    if (isnan(prod)) {
        u = 0x7FC00000u;
    } else {
        f = (float)prod; /* IEEE round to nearest even, subnormals and overflow included */
        memcpy(&u, &f, 4);
    }
    if (out_dt == OR_FP32)
        ((uint32_t*)out)[idx] = u;
    else
        ((uint16_t*)out)[idx] = oracle_f32_to_bf16(u);
}

/* MXFP8 rowwise: out = payload * 2^(code-127) (TE PR #3790, Description:
 * export decodes to dequantize(); TE PR #3264, Description: UE8M0 decode).
 * scales are in layout lay. */
int oracle_dequant_mxfp8(const uint8_t* data, const uint8_t* scales, int lay, int kind, int64_t rows, int64_t K,
                         void* out, int out_dt) {
    int64_t nb = oracle_scale_cols(K);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < K; ++i) {
            uint8_t c = scales[oracle_scale_offset(r, i / 32, nb, lay)];
            double prod = oracle_fp8_value(data[r * K + i], kind) * oracle_e8m0_value(c);
            store_result(out, out_dt, r * K + i, prod);
        }
    return OR_OK;
}

/* 128x128 blockwise: out = payload * tile_scale_inv[r/128, i/128]. */
int oracle_dequant_block128(const uint8_t* data, const float* tile_scale_inv, int64_t rows, int64_t K, void* out,
                            int out_dt) {
    int64_t tc = (K + 127) / 128;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < K; ++i) {
            double prod = oracle_fp8_value(data[r * K + i], OR_E4M3) * (double)tile_scale_inv[(r / 128) * tc + i / 128];
            store_result(out, out_dt, r * K + i, prod);
        }
    return OR_OK;
}

/* -------------------------------------------------- MXFP8 columnwise */

/* Scale exponent of the host MXFP8 quantizer for a 32x1 block: the smallest
 * s with amax <= 448 * 2^s (448 = E4M3's largest finite), i.e.
 * ceil(log2(amax / 448)), clamped to [-127, 127]; a zero amax gives -127.
 * Reading: the pages name "the host amax rule" without stating it; this is
 * the round-up power-of-two rule of MXFP8 quantizers, under which
 * amax / 2^s never exceeds 448. */
int oracle_mxfp8_host_exponent(double amax) {
    if (amax == 0.0) return -127;
    int s = ilogb(amax) - 12;
    while (ldexp(448.0, s) < amax) ++s;
    while (ldexp(448.0, s - 1) >= amax) --s;
    if (s < -127) s = -127;
    if (s > 127) s = 127;
    return s;
}

/* Direct MXFP8 columnwise (TE PR #3264, Description, mode 2: "MXFP8
 * columnwise = fresh 32x1 quantization with the host amax rule"; its bytes
 * match quantizing the projected weight): y = projection of x, then for
 * each 32x1 block (rows 32i..32i+31 of column c; the last may be shorter)
 * the host exponent s of max|y|, UE8M0 code s + 127 and payloads
 * RTNE_E4M3(y / 2^s).  A block holding a NaN (from a poisoned 1x32 block)
 * gets code 0xFF and payloads 0x7F.  data is [rows, K]; scales are compact
 * and transposed: scale (c, i) at c * ceil(rows/32) + i. */
int oracle_mxfp8_col_direct(const void* x, int dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* data,
                            uint8_t* scales) {
    if (dt != OR_BF16 && dt != OR_FP32) return OR_BAD;
    size_t es = dt == OR_BF16 ? 2 : 4;
    int64_t nbr = (rows + 31) / 32;
    void* y = malloc((size_t)(rows * K) * es + 1);
    if (!y) abort();
    oracle_fake_quant_mxfp4(x, y, dt, rows, K, ldx, K);
    for (int64_t c = 0; c < K; ++c) {
        for (int64_t i = 0; i < nbr; ++i) {
            int64_t r0 = 32 * i, r1 = r0 + 32 < rows ? r0 + 32 : rows;
            int poisoned = 0;
            double amax = 0.0;
            for (int64_t r = r0; r < r1; ++r) {
                uint32_t bits = load_bits(y, dt, r * K + c);
                if (is_nonfinite(bits, dt)) poisoned = 1;
                else if (abs_value(bits, dt) > amax) amax = abs_value(bits, dt);
            }
            if (poisoned) {
                scales[c * nbr + i] = 0xFF;
                for (int64_t r = r0; r < r1; ++r) data[r * K + c] = 0x7F;
                continue;
            }
            int sx = oracle_mxfp8_host_exponent(amax);
            scales[c * nbr + i] = (uint8_t)(sx + 127);
            for (int64_t r = r0; r < r1; ++r) {
                uint32_t bits = load_bits(y, dt, r * K + c);
                double v = ldexp(abs_value(bits, dt), -sx);
                data[r * K + c] = oracle_e4m3_rtne(sign_of(bits, dt) ? -v : v);
            }
        }
    }
    free(y);
    return OR_OK;
}

/* ------------------------------------------------------ packed MXFP4 */

/* Packed MXFP4 deployment form (TE PR #3264, Description: training sees
 * exactly the deployment weight, E2M1 payloads with 1x32 power-of-two
 * UE8M0 scales; "Known limitations": above amax = 6*2^125 packed deployment
 * moves to the scale 2^126, which bf16/fp32 cannot materialise).  Reading:
 * the block exponent is clamp(ceil(log2(amax/6)), -126, 126) -- the
 * projection's rule with the upper clamp at 126 -- its UE8M0 code is
 * e + 127, and each element is the E2M1 code nearest |x|/2^e (ties to the
 * even code) with the sign in bit 3.  Element 2i sits in the low nibble of
 * byte i of the row, element 2i+1 in the high nibble; a missing last
 * element leaves a zero nibble.  A poisoned block has scale code 0xFF and
 * zero nibbles.  packed is [rows, ceil(K/2)], scales compact [rows, nb]. */
int oracle_mxfp4_pack(const void* x, int dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* packed,
                      uint8_t* scales) {
    if (dt != OR_BF16 && dt != OR_FP32) return OR_BAD;
    size_t es = dt == OR_BF16 ? 2 : 4;
    int64_t nb = oracle_scale_cols(K), pb = (K + 1) / 2;
    for (int64_t r = 0; r < rows; ++r) {
        const char* xr = (const char*)x + (size_t)(r * ldx) * es;
        memset(packed + r * pb, 0, (size_t)pb);
        for (int64_t j0 = 0; j0 < K; j0 += 32) {
            int64_t j1 = j0 + 32 < K ? j0 + 32 : K;
            block_info b = scan_block(xr, dt, j0, j1);
            if (b.poisoned) {
                scales[r * nb + j0 / 32] = 0xFF;
                continue;
            }
            uint32_t amax = 0;
            for (int64_t i = j0; i < j1; ++i) {
                uint32_t mag = magnitude_bits(load_bits(xr, dt, i), dt);
                if (mag > amax) amax = mag;
            }
            /* the projection's rule with the upper clamp moved to 126 */
            int e = ceil_log2_amax_over_6(amax, dt);
            if (e < -126) e = -126;
            if (e > 126) e = 126;
            scales[r * nb + j0 / 32] = (uint8_t)(e + 127);
            for (int64_t i = j0; i < j1; ++i) {
                uint32_t bits = load_bits(xr, dt, i);
                int c = element_code(bits, dt, e) | (sign_of(bits, dt) << 3);
                packed[r * pb + i / 2] |= (uint8_t)(c << ((i % 2) * 4));
            }
        }
    }
    return OR_OK;
}

/* Value of a signed E2M1 nibble. */
double oracle_e2m1_value(uint8_t nibble) {
    double v = E2M1_GRID[nibble & 7];
    return (nibble & 8) ? -v : v;
}

/* Packed MXFP4 -> fp32 / bf16: out = value(nibble) * 2^(code-127), rounded
 * to nearest in fp32 (exact, or Inf where 2^126 * 4 or more overflows),
 * then to bf16.  scales are in layout lay. */
int oracle_dequant_mxfp4(const uint8_t* packed, const uint8_t* scales, int lay, int64_t rows, int64_t K, void* out,
                         int out_dt) {
    int64_t nb = oracle_scale_cols(K), pb = (K + 1) / 2;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < K; ++i) {
            uint8_t c = scales[oracle_scale_offset(r, i / 32, nb, lay)];
            uint8_t nib = (uint8_t)((packed[r * pb + i / 2] >> ((i % 2) * 4)) & 15);
            store_result(out, out_dt, r * K + i, oracle_e2m1_value(nib) * oracle_e8m0_value(c));
        }
    return OR_OK;
}

/* ----------------------------------------------------------------- export */

/* Compact (rows, ceil(K/32)) scales from a layout (TE PR #3790, Description:
 * unpadded, unswizzled; a short last block keeps its own column). */
int oracle_export_scales(const uint8_t* scales, int lay, int64_t rows, int64_t K, uint8_t* compact) {
    int64_t nb = oracle_scale_cols(K);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < nb; ++j) compact[r * nb + j] = scales[oracle_scale_offset(r, j, nb, lay)];
    return OR_OK;
}
