/*
 * fp4_quant.h -- C ABI of the online quantisation step that feeds the
 * block-scaled FP4 GEMM (include/fp4_gemm.h): fp32 or bf16 values become E2M1
 * codes packed two per byte plus one scale byte per block of vec values.
 *
 * The formats and block sizes are the GEMM's ("[BUG] Add FP4 TMA kernel
 * example for Blackwell in CuTe Python DSL", CUTLASS issue #2922, sections
 * "Scale Factor Granularity" and "Code Reference": Float8E4M3FN scales, one per
 * 16 values; "TMA Pipelines, Tensor Cores, and ctm-rs Interop", section 1:
 * Float8E8M0FNU scales, one per 32 values, for MXFP4). The pages do not say how
 * a scale is chosen; this library takes the usual absmax rule:
 *
 *   NVFP4  s = E4M3(amax / 6): the division in fp32, then round to nearest
 *          E4M3 (ties to the even code), saturating at 448;
 *   MXFP4  s = 2^(floor(log2 amax) - 2), exponent clamped to [-127, 127]; an
 *          all-zero block gets 2^-127 (byte 0);
 *   code   the E2M1 value nearest to q = x / s (q rounded to fp32 first), ties
 *          to the even code, |q| >= 6 saturating to 6, sign bit of x kept
 *          (-0 and negatives that round to zero give code 8). An NVFP4 block
 *          whose scale rounds to 0 gets all codes 0.
 *
 * Every decision is taken in fp32 and is exact: the codes and scale bytes are
 * a function of the input bits alone. Non-finite inputs are outside the
 * definition (their block's output is unspecified, nothing faults).
 *
 * Layouts (row-major, contiguous, device memory):
 *   X      [rows][K] fp32 or bf16 values.
 *   codes  [rows][K/2] bytes: element k = 2j in the low nibble of byte j, k = 2j + 1
 *          in the high nibble (the A / B operand layout of fp4_gemm).
 *   sf     FP4_SF_PLAIN: [rows][K/vec] bytes (the plain layout of fp4_gemm).
 *          FP4_SF_ATOM:  the 128x4 atom layout of fp4_scale_reorder, every byte
 *          of fp4_scale_atom_bytes(rows, K, vec) written (padding 0), ready for
 *          the _prepacked GEMM calls.
 *
 * Requirements: K % 32 == 0; X and codes 16-byte aligned; sf 16-byte aligned in
 * the atom layout (any alignment in the plain layout); no buffer overlaps
 * another. rows == 0 or K == 0 is a no-op.
 *
 * Ownership: the caller owns every buffer; nothing is allocated.
 * Errors: argument problems return a status synchronously and launch nothing
 * (rows above 2^31 - 1025, K above 2^31 - 1, or rows * K above 2^40:
 * FP4_ERR_UNSUPPORTED); a failed launch returns FP4_ERR_CUDA. The kernel's
 * waits are bounded (the limit of fp4_set_wait_limit_ms); one that runs out
 * leaves the outputs incomplete and is reported as FP4_ERR_TIMEOUT by
 * fp4_get_device_status. Asynchronous on `stream`, current device.
 */
#ifndef FP4_QUANT_H
#define FP4_QUANT_H

#include "fp4_gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FP4_IN_F32 = 0, FP4_IN_BF16 = 1 } fp4_in_dtype;
typedef enum { FP4_SF_PLAIN = 0, FP4_SF_ATOM = 1 } fp4_sf_layout;

/* Quantise X into E2M1 codes and NVFP4 (E4M3, vec 16) or MXFP4 (E8M0, vec 32) scales. */
fp4_status fp4_quantize(fp4_format fmt, const void *X, fp4_in_dtype in, int64_t rows, int64_t K,
                        void *codes, void *sf, fp4_sf_layout layout, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP4_QUANT_H */
