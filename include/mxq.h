/*
 * mxq.h -- C ABI of libmxq: block-scaled weight conversion on NVIDIA GB300
 * (sm_103a).  MXFP4 projection for quantization-aware training, direct
 * MXFP4 -> MXFP8 rowwise and MXFP4 -> FP8 128x128 blockwise conversion,
 * dequantize, and export of MXFP8 values with compact E8M0 scales.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All buffers are device memory owned by the caller.  The library
 *    allocates nothing and keeps no state between calls.
 *  - Work is enqueued on `stream` and runs asynchronously; argument checks
 *    run synchronously on the host before anything is enqueued.  A call
 *    that returns an error has enqueued nothing, except MXQ_ERR_CUDA, which
 *    reports a failed launch (the CUDA error is consumed with
 *    cudaGetLastError()).
 *  - A tensor is viewed as `rows` rows of `K` elements, row r starting
 *    `ld` elements after row r-1 (ld >= K).  Leading dimensions are in
 *    elements.  Higher-rank tensors pass rows = prod(shape[:-1]).
 *  - `rows == 0` or `K == 0` is an empty tensor: MXQ_OK, nothing launched.
 *  - Pointers must be aligned to their element size.  Any stronger
 *    alignment (16 bytes for the vector path) is optional: misaligned
 *    views take a scalar path with identical results.
 *  - Only one 1x32 block layout exists: block j of a row covers elements
 *    [32j, min(32j+32, K)), so a row has nb = ceil(K/32) blocks and the
 *    last one may be shorter; it keeps its own scale.
 *  - Results are bit-exact: every rounding is round-to-nearest-even on an
 *    exact value, and the library gives the same bytes when built with
 *    --use_fast_math.
 *  - NaN results are the canonical quiet NaN (bf16 0x7FC0, fp32
 *    0x7FC00000).
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MXQ_VERSION 1

#if defined(__GNUC__)
#define MXQ_API __attribute__((visibility("default")))
#else
#define MXQ_API
#endif

typedef enum {
    MXQ_OK = 0,
    MXQ_ERR_INVALID_ARG = 1,       /* bad size, stride, pointer or enum value */
    MXQ_ERR_UNSUPPORTED_DTYPE = 2, /* fp16 (and any other dtype) */
    MXQ_ERR_NO_ROWWISE_DATA = 3,   /* export of a storage without row-scaled data */
    MXQ_ERR_BUFFER_TOO_SMALL = 4,  /* export copy needed but scale_out too small */
    MXQ_ERR_CUDA = 5               /* a kernel launch failed */
} mxq_status;

typedef enum {
    MXQ_BF16 = 0,
    MXQ_FP32 = 1,
    MXQ_FP16 = 2 /* always rejected: the MXFP4 grid p*2^e reaches 6*2^125,
                    far beyond fp16 (TE PR #3264 "MXFP4 weight QAT on MXFP8
                    and FP8 block-scaling recipes", Description: STE
                    paragraph; "Known limitations") */
} mxq_dtype;

typedef enum { MXQ_E4M3 = 0, MXQ_E5M2 = 1 } mxq_fp8;

/* Layout of UE8M0 scale bytes for an MXFP8 tensor of rows x K.
 *  COMPACT:  [rows, nb] row-major, nb = ceil(K/32).
 *  PADDED:   [Rp, Cp] row-major, Rp = ceil(rows/128)*128, Cp = ceil(nb/4)*4.
 *  SWIZZLED: the same Rp*Cp bytes in the cuBLAS block-scaling-factor layout
 *            used by MXFP8 GEMMs: 128x4 tiles of 512 bytes, tiles in
 *            row-major order, and scale (r, j) at byte
 *            ((r/128)*(Cp/4) + j/4)*512 + (r%32)*16 + ((r%128)/32)*4 + j%4.
 * Writers fill padding bytes with 0; readers never look at them.
 * (TE PR #3790 "MXFP8TensorStorage.export_components()", Description:
 * scales padded when ceil(K/32) is not a multiple of 4, or swizzled for
 * GEMM with optimize_for_gemm=True.) */
typedef enum { MXQ_SCALES_COMPACT = 0, MXQ_SCALES_PADDED = 1, MXQ_SCALES_SWIZZLED = 2 } mxq_scale_layout;

/* Bytes of a scale buffer of the given layout (0 for an empty tensor). */
MXQ_API size_t mxq_scale_bytes(int64_t rows, int64_t K, mxq_scale_layout lay);

/* Number of fp32 tile scales of the 128x128 blockwise form:
 * ceil(rows/128) * ceil(K/128). */
MXQ_API size_t mxq_tile_scale_count(int64_t rows, int64_t K);

/* MXFP4 projection ("fake quantization").
 * Source: TE PR #3264 "MXFP4 weight QAT on MXFP8 and FP8 block-scaling
 * recipes", Description, mode 1 (Projection).
 * For every 1x32 block: e = clamp(ceil(log2(amax/6)), -126, 125), read off
 * the amax bit pattern; each element becomes sign(x) * p * 2^e with p the
 * E2M1 grid point {0, 0.5, 1, 1.5, 2, 3, 4, 6} nearest |x|/2^e (ties to the
 * even code; beyond 6 it saturates to 6, so amax > 6*2^125 lands on
 * 6*2^125).  A block holding a NaN or an Inf is poisoned: all its outputs
 * are the canonical NaN.  The sign of zero is kept.
 *   x:   [rows, ldx] input, bf16 or fp32 (dt); y: [rows, ldy] output, same
 *        dtype.  y == x (same ld) projects in place; any other overlap is
 *        undefined.
 * Errors: INVALID_ARG (negative sizes, ld < K, NULL or misaligned pointers),
 * UNSUPPORTED_DTYPE (fp16). */
MXQ_API mxq_status mxq_fake_quant_mxfp4(const void* x, void* y, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                int64_t ldy, cudaStream_t stream);

/* Direct MXFP4 -> MXFP8 rowwise conversion (fixed-shift-6 lift).
 * Source: TE PR #3264, Description, mode 2 (Direct), "MXFP8 rowwise".
 * With e and p from the projection above: scale code = max(e + 121, 0)
 * (the UE8M0 code of 2^(e-6), clamped at code 0 = 2^-127), payload =
 * E4M3(sign * p * 2^(e + 127 - code)), which is exact: p*2^6 when the code
 * is not clamped, the payload absorbing the clamp otherwise.  Payload *
 * 2^(code-127) equals the projection bit for bit.  Poisoned blocks get
 * scale code 0xFF and payloads 0x7F (both decode to NaN).
 *   x:      [rows, ldx] bf16 or fp32.
 *   data:   [rows, K] E4M3 bytes, contiguous.
 *   scales: mxq_scale_bytes(rows, K, lay) bytes in layout `lay`
 *           (padding written as 0).
 * Errors: as mxq_fake_quant_mxfp4; INVALID_ARG for a bad layout. */
MXQ_API mxq_status mxq_mxfp8_row_direct(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* data,
                                uint8_t* scales, mxq_scale_layout lay, cudaStream_t stream);

/* Direct MXFP4 -> FP8 128x128 blockwise conversion (per-tile exponent
 * folding).  Source: TE PR #3264, Description, mode 2 (Direct),
 * "blockwise"; "Test results (B200)": exact through tile scale spread 2^14.
 * Tiles are 128x128 (the last tile row/column may be partial).  With e_b
 * the exponent of each finite 1x32 block of the tile, T = max(max_b e_b -
 * 6, -127); every payload is E4M3 round-to-nearest-even (subnormals
 * included) of sign * p * 2^(e_b - T).  Poisoned blocks give payloads 0x7F
 * and do not enter the maximum; a tile without a finite block has T = -127.
 * No device-side assert exists on any spread.
 *   x:              [rows, ldx] bf16 or fp32.
 *   data:           [rows, K] E4M3 bytes, contiguous.
 *   tile_scale_inv: [ceil(rows/128), ceil(K/128)] fp32, each 2^T exactly
 *                   (2^-127 is the fp32 subnormal 0x00400000).
 * Errors: as mxq_fake_quant_mxfp4. */
MXQ_API mxq_status mxq_fp8_block128_direct(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* data,
                                   float* tile_scale_inv, cudaStream_t stream);

/* Packed MXFP4, the deployment form of the projection (TE PR #3264,
 * Description: training sees exactly the deployment weight, E2M1 payloads
 * with 1x32 power-of-two UE8M0 scales; "Known limitations": above
 * amax = 6*2^125 packed deployment moves to the scale 2^126).
 * Block exponent e' = clamp(ceil(log2(amax/6)), -126, 126) -- the
 * projection's rule with the upper clamp at 126 -- stored as the UE8M0 code
 * e' + 127; each element is the E2M1 code nearest |x|/2^e' (ties to the even
 * code) with the sign in bit 3.  Element 2i is the low nibble of byte i of
 * its row, element 2i+1 the high nibble (a missing last element leaves 0).
 * Wherever amax <= 6*2^125 the packed weight decodes exactly to
 * mxq_fake_quant_mxfp4's output.  A poisoned block has scale code 0xFF and
 * zero nibbles.
 *   x:      [rows, ldx] bf16 or fp32.
 *   packed: [rows, ceil(K/2)] bytes, contiguous.
 *   scales: mxq_scale_bytes(rows, K, lay) bytes in layout `lay`.
 * Errors: as mxq_mxfp8_row_direct. */
MXQ_API mxq_status mxq_mxfp4_pack(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx, uint8_t* packed,
                                  uint8_t* scales, mxq_scale_layout lay, cudaStream_t stream);

/* Direct MXFP4 -> MXFP8 columnwise (32x1 blocks) of the projected weight.
 * Source: TE PR #3264, Description, mode 2: "MXFP8 columnwise = fresh 32x1
 * quantization with the host amax rule" (its bytes match quantizing the
 * mode-1 projection).  The pages do not state the host rule; it is read as
 * the round-up power of two of MXFP8 quantizers: for each 32x1 block (rows
 * 32i..32i+31 of column c, the last may be shorter) of y =
 * mxq_fake_quant_mxfp4(x), s = ceil(log2(max|y| / 448)) clamped to
 * [-127, 127] (a zero block gives -127), UE8M0 code s + 127, payloads
 * RTNE_E4M3(y / 2^s), subnormals included (never saturating).  A block
 * holding a NaN (from a poisoned 1x32 block) gets code 0xFF and payloads
 * 0x7F.
 *   x:      [rows, ldx] bf16 or fp32.
 *   data:   [rows, K] E4M3 bytes, contiguous (quantized along rows).
 *   scales: the column scales as the K x ceil(rows/32) matrix of the
 *           transposed tensor -- scale (c, i) at c*ceil(rows/32) + i when
 *           COMPACT -- in layout `lay`: mxq_scale_bytes(K, rows, lay) bytes.
 * Errors: as mxq_mxfp8_row_direct. */
MXQ_API mxq_status mxq_mxfp8_col_direct(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                        uint8_t* data, uint8_t* scales, mxq_scale_layout lay, cudaStream_t stream);

/* Skip-update variants of the converters, for cached weights updated inside
 * a captured CUDA graph (TE PR #3264, review: a direct cache-hit update must
 * honour the skip-update flag of CUDA-graph replays).  `skip` is a device
 * int32 read when the kernel runs; if it is nonzero the call writes nothing
 * (every output keeps its previous bytes).  skip == NULL behaves as the
 * plain entry point.  Arguments and errors otherwise as above. */
MXQ_API mxq_status mxq_fake_quant_mxfp4_update(const void* x, void* y, mxq_dtype dt, int64_t rows, int64_t K,
                                               int64_t ldx, int64_t ldy, const int32_t* skip, cudaStream_t stream);
MXQ_API mxq_status mxq_mxfp8_row_direct_update(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                               uint8_t* data, uint8_t* scales, mxq_scale_layout lay,
                                               const int32_t* skip, cudaStream_t stream);
MXQ_API mxq_status mxq_fp8_block128_direct_update(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                                  uint8_t* data, float* tile_scale_inv, const int32_t* skip,
                                                  cudaStream_t stream);
/* The columnwise copy of the same cached weight (the direct workspace holds
 * rowwise, columnwise and blockwise forms; TE PR #3264, review flowchart:
 * every part of the workspace refresh is gated by the skip flag) and the
 * packed MXFP4 deployment form.  A nonzero flag leaves the payload, the
 * scales and their padding untouched. */
MXQ_API mxq_status mxq_mxfp8_col_direct_update(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                               uint8_t* data, uint8_t* scales, mxq_scale_layout lay,
                                               const int32_t* skip, cudaStream_t stream);
MXQ_API mxq_status mxq_mxfp4_pack_update(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                         uint8_t* packed, uint8_t* scales, mxq_scale_layout lay, const int32_t* skip,
                                         cudaStream_t stream);

typedef enum {
    MXQ_QUANT_MXFP8_ROW = 0,
    MXQ_QUANT_FP8_BLOCK128 = 1,
    MXQ_QUANT_MXFP4 = 2,
    MXQ_QUANT_MXFP8_COL = 3 /* scales: the transposed K x ceil(rows/32) matrix in `lay` */
} mxq_quant_kind;

/* A quantized tensor of rows x K as read by mxq_dequantize. */
typedef struct {
    mxq_quant_kind kind;
    const uint8_t* data;         /* [rows, K] payload bytes, contiguous; MXFP4: [rows, ceil(K/2)] nibbles */
    int64_t rows, K;
    mxq_fp8 fp8;                 /* payload encoding; BLOCK128 takes E4M3 only; MXFP4 ignores it */
    const uint8_t* scales;       /* MXFP8_ROW, MXFP4: UE8M0 codes in layout `lay` */
    mxq_scale_layout lay;
    const float* tile_scale_inv; /* FP8_BLOCK128: [ceil(rows/128), ceil(K/128)] */
} mxq_quantized;

/* Dequantize to bf16 or fp32.  Sources: TE PR #3790, Description and tests
 * (the export decodes to dequantize() exactly); TE PR #3264, Description
 * (UE8M0 decode: code 0 is 2^-127, code 255 is NaN).
 * MXFP8_ROW: out = payload * 2^(code - 127); BLOCK128: out = payload *
 * tile_scale_inv; MXFP4: out = E2M1 value * 2^(code - 127); MXFP8_COL: out =
 * payload * 2^(code(c, r/32) - 127).  fp32 output is
 * that product rounded to nearest even (exact for power-of-two scales, Inf
 * on overflow, e.g. 4 * 2^126); bf16 output is one more
 * round-to-nearest-even of the fp32 value.
 *   out: [rows, K] contiguous, dtype out_dt (fp16 rejected).
 * Errors: INVALID_ARG, UNSUPPORTED_DTYPE. */
MXQ_API mxq_status mxq_dequantize(const mxq_quantized* q, void* out, mxq_dtype out_dt, cudaStream_t stream);

/* An MXFP8 tensor as a quantized storage holds it. */
typedef struct {
    const uint8_t* data;   /* rowwise payload [rows, K]; NULL = no row-scaled data */
    const uint8_t* scales; /* rowwise UE8M0 codes in layout `lay` */
    mxq_fp8 fp8;           /* how the payload bytes are to be read */
    mxq_scale_layout lay;
    int64_t rows, K;
} mxq_mxfp8_storage;

/* Export result: values plus compact (rows, ceil(K/32)) uint8 scales. */
typedef struct {
    const uint8_t* data;   /* always an alias of storage.data */
    mxq_fp8 fp8;           /* the dtype to view `data` as */
    const uint8_t* scales; /* compact [rows, scale_cols] */
    int64_t rows, K, scale_cols;
    int is_view;           /* 1: scales alias storage.scales; 0: copied into scale_out */
} mxq_mxfp8_components;

/* export_components.  Source: TE PR #3790 "MXFP8TensorStorage.
 * export_components()", Description.
 * `data` always aliases the storage's payload, so it changes when the
 * storage is updated in place (copy it to keep a snapshot).  The scales are
 * a view of the storage when they are already compact in memory (COMPACT,
 * or PADDED with nb a multiple of 4, whose first rows*nb bytes are the
 * compact matrix); otherwise (PADDED with nb % 4 != 0, SWIZZLED) one kernel
 * copies them into `scale_out`, dropping padding and undoing the swizzle.
 *   scale_out: device buffer of scale_out_bytes >= rows*nb, used only when
 *              a copy is needed (may be NULL otherwise).
 * Large swizzled copies stage 128-row tiles in shared memory through bulk
 * copies whose completion the kernel waits for at most about a second; a
 * tile whose copy has not arrived by then (a device fault, never expected)
 * has its compact rows written as 0xFF, the E8M0 NaN code, since the call
 * itself has already returned.
 * Errors: NO_ROWWISE_DATA if st->data is NULL (with rows*K > 0);
 * BUFFER_TOO_SMALL if a copy is needed and scale_out is NULL or too small;
 * INVALID_ARG otherwise.  `out` is written only on MXQ_OK. */
MXQ_API mxq_status mxq_export_mxfp8(const mxq_mxfp8_storage* st, uint8_t* scale_out, size_t scale_out_bytes,
                            mxq_mxfp8_components* out, cudaStream_t stream);

/* Export of several storages (per-expert export; TE PR #3790 lists the
 * per-expert export of a GroupedTensor as not covered there) in as few
 * launches as possible: every storage is exported as by mxq_export_mxfp8;
 * the ones that need a copy get consecutive regions of scale_out, in order,
 * and all copies run in one kernel launch per 128 storages.  Storages of
 * any size are accepted (each one's 128-row tiles are walked in a loop).
 *   st[count], out[count]: storages and their components.
 *   scale_out: device buffer for the copied scales, scale_out_bytes long.
 * Errors: as mxq_export_mxfp8 for any storage, and BUFFER_TOO_SMALL if the
 * copies do not fit -- both checked before anything is launched; MXQ_ERR_CUDA
 * if a launch fails, in which case the launches of earlier groups of 128
 * storages may already be enqueued. */
MXQ_API mxq_status mxq_export_mxfp8_grouped(const mxq_mxfp8_storage* st, int64_t count, uint8_t* scale_out,
                                            size_t scale_out_bytes, mxq_mxfp8_components* out, cudaStream_t stream);

/* Quantize and export in one call (TE issue #3644: "quantize weights for
 * inference, then extract the resulting values and scales"; TE PR #3790,
 * Description: a standalone function that quantizes a BF16 weight first).
 * Runs mxq_mxfp8_row_direct with COMPACT scales, which are already the
 * exported layout, and fills `out` (a view of data and scales).
 *   data: [rows, K] E4M3 bytes; scales: [rows, ceil(K/32)] bytes.
 * Errors: as mxq_mxfp8_row_direct; INVALID_ARG if out is NULL. */
MXQ_API mxq_status mxq_quantize_export_mxfp8(const void* x, mxq_dtype dt, int64_t rows, int64_t K, int64_t ldx,
                                             uint8_t* data, uint8_t* scales, mxq_mxfp8_components* out,
                                             cudaStream_t stream);

/* Static description of a status code. */
MXQ_API const char* mxq_status_string(mxq_status s);

/* MXQ_VERSION of the loaded library. */
MXQ_API int mxq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H */
