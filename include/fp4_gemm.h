/*
 * fp4_gemm.h -- C ABI of the GB300 (sm_103a) block-scaled FP4 GEMM.
 *
 *   D = alpha * ( decode(A, sfA) . decode(B, sfB)^T )
 *
 * The operation: a blockwise-scaled GEMM on E2M1 (Float4E2M1FN) operands,
 * computed by the block-scaled FP4 MMA ("[BUG] Add FP4 TMA kernel example for
 * Blackwell in CuTe Python DSL", CUTLASS issue #2922, sections "Summary",
 * "Background" and "What Works": MmaMXF4NVF4Op). Two scale formats:
 *   - NVFP4: one E4M3 scale per 16 K-elements (same issue, section "Scale
 *     Factor Granularity": sf_vec_size = 16, Float8E4M3FN scales);
 *   - MXFP4: one E8M0 scale per 32 K-elements ("TMA Pipelines, Tensor Cores,
 *     and ctm-rs Interop", section 1, "Block-Scaled MXFP4 GEMM in cute-rs
 *     (SM120a)": Float8E8M0FNU scales).
 * The block-scaled MMA consumes K = 64 FP4 elements per instruction (issue
 * #2922, section "MMA Instruction K Constraint").
 *
 * Layouts (all row-major, contiguous, on the device unless a call says host):
 *   A    [M][K/2] bytes. Two E2M1 codes per byte, K-major: element k = 2j is
 *        the low nibble of byte j, k = 2j + 1 the high nibble. ("Hopper GEMM
 *        in CUTLASS C++ and the CuTe DSL, part 1", section on the swapped
 *        operands, reason 3: both operands of the narrow GEMM are K-major.)
 *   B    [N][K/2] bytes, same packing (the GEMM uses B transposed).
 *   sfA  [M][K/vec] bytes, sfB [N][K/vec] bytes: plain row-major scale bytes
 *        (E4M3 for NVFP4, vec = 16; E8M0 for MXFP4, vec = 32). E4M3 scales are
 *        read as unsigned (sign bit must be 0); NaN scale bytes give
 *        unspecified output.
 *   "prepacked" scales: the same bytes in the 128x4 atom layout produced by
 *        fp4_scale_reorder (rows padded to 128, scale columns to 4; atom
 *        (rb, cb) at byte (rb * ceil(K/vec/4) + cb) * 512; row r, column c
 *        inside it at (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4); padding 0).
 *   D    [M][N], fp32 or bf16 (round to nearest even), overwritten. No C, no beta.
 *
 * Requirements: K % 32 == 0; A, B, sfA, sfB, D 16-byte aligned. M, N, K >= 0;
 * M == 0 or N == 0 is a no-op; K == 0 writes D = 0.
 *
 * Ownership: the caller owns every buffer; the library never frees them.
 * Calls taking plain scales reorder them into stream-ordered scratch
 * (cudaMallocAsync / cudaFreeAsync on `stream`); the partial sums of split-K
 * plans and of a split last wave (with its hand-off flags; only when
 * fp4_gemm_config.split_tail asks for it) use the same kind of scratch.
 * Nothing else is allocated per call.
 *
 * Errors: argument problems return a status synchronously and launch nothing.
 * Launch failures return FP4_ERR_CUDA. Every wait inside the kernels is
 * bounded; a wait that runs out records FP4_ERR_TIMEOUT in a per-device status
 * word that fp4_get_device_status reports. Calls are asynchronous with respect
 * to the host and run on the current device.
 *
 * Graphs: the GEMM, reorder and quantiser calls may be recorded by stream
 * capture into a CUDA graph, once a plain call of the same kind has run on the
 * device (it sets the kernels' attributes). Each replay repeats the captured
 * plan on the same buffers, alpha and (grouped calls) group offsets, and reads
 * whatever the input buffers hold at replay time. Scratch taken while capturing
 * becomes graph-owned memory. fp4_get_device_status synchronises the stream and
 * cannot be captured.
 */
#ifndef FP4_GEMM_H
#define FP4_GEMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP4_OK = 0,
    FP4_ERR_INVALID_ARG = 1,   /* null pointer, negative size, unknown enum */
    FP4_ERR_UNSUPPORTED = 2,   /* K % 32 != 0, size beyond the kernel's index range, bad config */
    FP4_ERR_MISALIGNED = 3,    /* a pointer not 16-byte aligned */
    FP4_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    FP4_ERR_TIMEOUT = 5,       /* a bounded device wait ran out (reported by fp4_get_device_status) */
    FP4_ERR_NO_DEVICE = 6,     /* no device, or not an sm_103 device */
    FP4_ERR_SCRATCH_LIMIT = 7  /* fp4_gemm_static_scratch: problem needs more than FP4_STATIC_SCRATCH_BYTES */
} fp4_status;

typedef enum { FP4_OUT_F32 = 0, FP4_OUT_BF16 = 1 } fp4_out_dtype;
typedef enum { FP4_FMT_NVFP4 = 0, FP4_FMT_MXFP4 = 1 } fp4_format;

/* Optional overrides of the launch plan (zero-initialise for "automatic").
 *   mode:      0 auto; 1 direct (A on the MMA's M side, D rows written in
 *              whole 32-byte sectors); 2 swap-AB (B on the M side, D^T tiles written with
 *              coalesced stores; the trick of "Hopper GEMM in CUTLASS C++ and
 *              the CuTe DSL, part 1", section on the swapped operands);
 *              3 the narrow-M CUDA-core kernel (M <= 4; it reads both scale
 *              layouts in place, so it launches no reorder and needs no
 *              scratch; sfB must be 2-byte aligned). Auto picks 3 for M == 1
 *              with plain scales (where it measured faster), when A's decoded
 *              row fits its shared staging (K + K/vec * 4 bytes, K rounded up
 *              to 4096, at most 200 KB) and sfB is 2-byte aligned; else 2 for
 *              M <= 256, else 1.
 *              The other fields apply to modes 1 and 2 only.
 *   bn:        0 auto; else the MMA N of a tile: 16, 32, 64, 128 or 256.
 *              Direct mode needs 128 or 256; so do several tiles on the N side.
 *   splits:    0 auto; else the number of K splits (swap-AB mode only).
 *   max_ctas:  0 = as many persistent CTAs as fit (one per SM); else a cap.
 *   cta_group: 0 auto; 1 = one CTA per 128-row MMA; 2 = a CTA pair (cluster
 *              of 2) per 256-row MMA (bn 128 or 256).
 *   stop_after: testing the bounded waits only, 0 otherwise. n > 0: every
 *              TMA producer of the GEMM kernel stops after filling n k-tile
 *              stages (it loads and signals nothing for stage n or later),
 *              so the MMA issuer's bounded wait for stage n runs out: the
 *              launch records FP4_ERR_TIMEOUT (read it with
 *              fp4_get_device_status), every role leaves its loop, the
 *              kernel waits for the copies and MMAs it did issue, frees its
 *              TMEM and returns. D is then unspecified. No MMA reads a stage
 *              that did not land. Modes 1 and 2 only.
 *   split_tail: direct mode. 0 = automatic, which is off: on this GPU every
 *              shape where it applied ran faster without it. 1 = when the
 *              last, partial wave of tiles fills at most half of the resident
 *              CTAs (or pairs), its tiles run as two K halves on two CTAs,
 *              the second adding the first's fp32 partial in a fixed order.
 *              Other values: FP4_ERR_INVALID_ARG.                           */
typedef struct {
    int32_t mode;
    int32_t bn;
    int32_t splits;
    int32_t max_ctas;
    int32_t cta_group;
    int32_t stop_after;
    int32_t split_tail;
} fp4_gemm_config;

/* What a call with these arguments would launch (no launch, nothing read):
 *   kernel:    0 the tcgen05 GEMM, 1 the narrow-M CUDA-core kernel;
 *   swap, bn, cta_group, splits: the tcgen05 plan (mode 1/2 semantics);
 *   launches:  kernels one call launches (scale reorders, GEMM, split-K
 *              reduce). Assumes 2-byte aligned scales. Needs an sm_103 device
 *              (the plan depends on its SM count);
 *   errors as the GEMM call's host validation. */
typedef struct {
    int32_t kernel;
    int32_t swap;
    int32_t bn;
    int32_t cta_group;
    int32_t splits;
    int32_t launches;
} fp4_plan_info;

fp4_status fp4_gemm_plan(fp4_format fmt, int scales_prepacked, int64_t M, int64_t N, int64_t K,
                         fp4_out_dtype out, int32_t act, const fp4_gemm_config *cfg,
                         fp4_plan_info *info);

/* NVFP4 GEMM (E4M3 scales, one per 16 K-elements), plain row-major scales. */
fp4_status fp4_gemm_nvfp4(const void *A, const void *sfA, const void *B, const void *sfB,
                          float alpha, void *D, int64_t M, int64_t N, int64_t K,
                          fp4_out_dtype out, cudaStream_t stream);

/* MXFP4 GEMM (E8M0 scales, one per 32 K-elements), plain row-major scales. */
fp4_status fp4_gemm_mxfp4(const void *A, const void *sfA, const void *B, const void *sfB,
                          float alpha, void *D, int64_t M, int64_t N, int64_t K,
                          fp4_out_dtype out, cudaStream_t stream);

/* Same GEMMs on scales already in the 128x4 atom layout (fp4_scale_reorder):
 * the weight-side reorder can be done once and hoisted out of the hot loop. */
fp4_status fp4_gemm_nvfp4_prepacked(const void *A, const void *sfA_atoms, const void *B,
                                    const void *sfB_atoms, float alpha, void *D, int64_t M,
                                    int64_t N, int64_t K, fp4_out_dtype out, cudaStream_t stream);
fp4_status fp4_gemm_mxfp4_prepacked(const void *A, const void *sfA_atoms, const void *B,
                                    const void *sfB_atoms, float alpha, void *D, int64_t M,
                                    int64_t N, int64_t K, fp4_out_dtype out, cudaStream_t stream);

/* General form of the four calls above, with an optional plan override (cfg may be NULL). */
fp4_status fp4_gemm(fp4_format fmt, int scales_prepacked, const void *A, const void *sfA,
                    const void *B, const void *sfB, float alpha, void *D, int64_t M, int64_t N,
                    int64_t K, fp4_out_dtype out, const fp4_gemm_config *cfg, cudaStream_t stream);

/* Fused epilogue of fp4_gemm_fused, applied to each element of the fp32
 * accumulator before the output cast (the pages name these elementwise
 * stages beside their block-scaled GEMMs: "TMA Pipelines, Tensor Cores, and
 * ctm-rs Interop", section "Where to Go Next" -- the SwiGLU elementwise
 * workload and the NVFP4 ReLU-squared MoE):
 *   z[m][n] = alpha * acc[m][n] + (bias ? bias[n] : 0)
 *   FP4_ACT_NONE    D[m][n] = z[m][n]
 *   FP4_ACT_RELU    D[m][n] = max(z[m][n], 0)
 *   FP4_ACT_RELU2   D[m][n] = max(z[m][n], 0)^2
 *   FP4_ACT_SWIGLU  D[m][j] = silu(z[m][2j]) * z[m][2j+1],  silu(x) = x / (1 + exp(-x)),
 *                   j < N/2: gate and up projections interleaved column by column
 *                   in B (gate rows 2j, up rows 2j+1), so D has N/2 columns.
 * The pages do not fix the SwiGLU column layout; interleaving keeps each
 * gate/up pair inside one accumulator tile. Arithmetic is fp32 (fmaf for z,
 * expf and an IEEE division for silu).
 *   bias: device, N floats (one per GEMM output column, before the SwiGLU
 *         pairing), 4-byte aligned; NULL for none. Owned by the caller.     */
typedef enum {
    FP4_ACT_NONE = 0,
    FP4_ACT_RELU = 1,
    FP4_ACT_RELU2 = 2,
    FP4_ACT_SWIGLU = 3
} fp4_activation;

typedef struct {
    int32_t act;          /* fp4_activation */
    const float *bias;    /* NULL or N floats on the device */
} fp4_epilogue;

/* fp4_gemm with a fused epilogue (epi may be NULL: then identical to fp4_gemm).
 * D is [M][N] (fp32 or bf16), or [M][N/2] for FP4_ACT_SWIGLU, which needs N even
 * (else FP4_ERR_UNSUPPORTED). A misaligned bias gives FP4_ERR_MISALIGNED, an
 * unknown act FP4_ERR_INVALID_ARG. K == 0 writes the epilogue of z = bias. */
fp4_status fp4_gemm_fused(fp4_format fmt, int scales_prepacked, const void *A, const void *sfA,
                          const void *B, const void *sfB, float alpha, const fp4_epilogue *epi,
                          void *D, int64_t M, int64_t N, int64_t K, fp4_out_dtype out,
                          const fp4_gemm_config *cfg, cudaStream_t stream);

/* Grouped GEMM (a mixture-of-experts layer): G independent GEMMs sharing N
 * and K. Group g owns rows offsets[g] .. offsets[g+1]-1 of A and of D and the
 * weight matrix B_g; for each g
 *   D[offsets[g] + i][n] = epi( alpha * sum_k a(offsets[g] + i, k) * b_g(n, k) + bias[g*N + n] )
 * (the NVFP4 ReLU-squared MoE of "TMA Pipelines, Tensor Cores, and ctm-rs
 * Interop", "Where to Go Next": each expert's weights applied to the tokens
 * routed to it, rows sorted by expert).
 *   offsets  HOST array of G+1 int64: offsets[0] = 0, non-decreasing (empty
 *            groups allowed), M_total = offsets[G]. Read during the call only.
 *   A        [M_total][K/2], sfA plain [M_total][K/vec].
 *   B        [G][N][K/2] (B_g contiguous); sfB plain [G][N][K/vec], or with
 *            FP4_GROUPED_B_ATOMS in scales_prepacked the G atom-layout copies
 *            of fp4_scale_reorder back to back (each fp4_scale_atom_bytes(N,
 *            K, vec) bytes; the same bytes as one reorder of all G*N rows
 *            when N % 128 == 0). With FP4_GROUPED_A_ATOMS, sfA is the output
 *            of fp4_scale_reorder_grouped for the same offsets.
 *   epi      as fp4_gemm_fused; bias, if given, is [G][N] floats (per group).
 *   D        [M_total][N] (or [M_total][N/2] for SwiGLU).
 * One launch covers every group: the persistent kernel's tiles are the groups'
 * tiles back to back, the groups' geometry passed in its parameter block (no
 * table upload, so the call never synchronises the host with the stream).
 * Plan: swap-AB (weights on the MMA's M side, one tile of a group's rows on
 * its N side) when every group has at most 256 rows or D's rows cannot take
 * 16-byte stores, else direct; no K split. Scratch: stream-ordered (the
 * reordered scales). Requirements and errors as fp4_gemm; offsets not
 * starting at 0 or decreasing give FP4_ERR_INVALID_ARG; G above 256, M_total
 * or G * N above 2^30, FP4_ERR_UNSUPPORTED. cfg may force mode 1 (direct) or
 * 2 (swap-AB). */
#define FP4_GROUPED_B_ATOMS 1   /* sfB: the G groups' atom-layout copies back to back */
#define FP4_GROUPED_A_ATOMS 2   /* sfA: the grouped atom layout of fp4_scale_reorder_grouped */
fp4_status fp4_gemm_grouped(fp4_format fmt, int scales_prepacked, int64_t G, const int64_t *offsets,
                            const void *A, const void *sfA, const void *B, const void *sfB, float alpha,
                            const fp4_epilogue *epi, void *D, int64_t N, int64_t K, fp4_out_dtype out,
                            const fp4_gemm_config *cfg, cudaStream_t stream);

/* The grouped atom layout of activation scales: each group's rows
 * (offsets as fp4_gemm_grouped) reordered like fp4_scale_reorder, every group
 * starting a fresh 128-row block; fp4_scale_atom_bytes_grouped gives its size
 * (0 for invalid arguments). Host offsets, G <= 256; errors as
 * fp4_scale_reorder. */
size_t fp4_scale_atom_bytes_grouped(int64_t G, const int64_t *offsets, int64_t k, int vec);
fp4_status fp4_scale_reorder_grouped(const void *sf_plain, void *sf_atom, int64_t G, const int64_t *offsets,
                                     int64_t k, int vec, cudaStream_t stream);

/* Host-buffer convenience form: A, sfA, B, sfB and D live in HOST memory
 * (pinned for asynchronous copies). The call copies the inputs to stream-ordered
 * device scratch, runs fp4_gemm, copies D back and returns; D is valid once
 * `stream` has been synchronised. Same layouts and errors as fp4_gemm. */
fp4_status fp4_gemm_host(fp4_format fmt, const void *A, const void *sfA, const void *B,
                         const void *sfB, float alpha, void *D, int64_t M, int64_t N, int64_t K,
                         fp4_out_dtype out, cudaStream_t stream);

/* Capacity of the library's static device scratch array (see fp4_gemm_static_scratch). */
#define FP4_STATIC_SCRATCH_BYTES (16u << 20)

/* The same GEMM as fp4_gemm_nvfp4 / fp4_gemm_mxfp4 (plain row-major scales),
 * for callers that must not allocate device memory: code running where
 * cudaMalloc / cudaMallocAsync are unavailable or forbidden, such as inside a
 * memory-pool owner, an allocator callback, or a process whose device memory
 * is entirely pre-reserved by another framework. The pages have no
 * counterpart; this entry point exists for such callers only.
 *
 * The reordered scales and any split-K partial sums go to one static
 * __device__ array of FP4_STATIC_SCRATCH_BYTES (16 MiB) that every device
 * loading the library holds until the process exits. The call takes the
 * automatic plan (no split last wave). A plan whose split-K partials would not
 * fit takes fewer K splits (down to none); problems whose scale atoms alone do
 * not fit (2 * ceil(rows/128) * ceil(K/vec/4) * 512 bytes) are rejected with
 * FP4_ERR_SCRATCH_LIMIT before anything is launched. The call allocates
 * nothing and calls no allocating library routine. Nothing in the array has to
 * start at zero: every byte a call reads was written earlier in the same call.
 * All calls on a device share the array, so calls whose kernels overlap on the
 * GPU (other streams, other threads) race: order them on one stream.
 * The first call on a device loads the library's device code there (CUDA's
 * lazy module loading), which is when the array is reserved, and looks up the
 * array's device address (cudaGetSymbolAddress) with that device current:
 * make that first call before the device's memory is handed to another owner,
 * and before any stream capture. Inputs, outputs and errors as fp4_gemm. */
fp4_status fp4_gemm_static_scratch(fp4_format fmt, const void *A, const void *sfA, const void *B,
                                   const void *sfB, float alpha, void *D, int64_t M, int64_t N,
                                   int64_t K, fp4_out_dtype out, cudaStream_t stream);

/* Bytes of the atom-layout copy of a rows x (k/vec) scale matrix (vec 16 or 32).
 * Returns 0 for invalid arguments. */
size_t fp4_scale_atom_bytes(int64_t rows, int64_t k, int vec);

/* Scale reorder kernel: plain row-major sf[rows][k/vec] -> 128x4 atom layout
 * (every byte of the fp4_scale_atom_bytes() output written, padding = 0).
 * Both buffers on the device; sf_atom must not overlap sf_plain. */
fp4_status fp4_scale_reorder(const void *sf_plain, void *sf_atom, int64_t rows, int64_t k,
                             int vec, cudaStream_t stream);

/* Both operands' scales of one GEMM in one launch (what the plain-scale calls
 * launch before the GEMM): sf_a -> atoms_a (rows_a rows), sf_b -> atoms_b
 * (rows_b rows), same k and vec; a side with 0 rows is skipped. As
 * fp4_scale_reorder otherwise. */
fp4_status fp4_scale_reorder2(const void *sf_a, void *atoms_a, int64_t rows_a, const void *sf_b, void *atoms_b,
                              int64_t rows_b, int64_t k, int vec, cudaStream_t stream);

/* Synchronises `stream`, then returns and clears the current device's status
 * word (FP4_OK, or FP4_ERR_TIMEOUT if a bounded wait ran out since the last call). */
fp4_status fp4_get_device_status(cudaStream_t stream);

/* Static description of a status code. */
const char *fp4_status_string(fp4_status s);

/* Bound on every device-side wait, in milliseconds (default 2000; also read once
 * from the FP4_GEMM_WAIT_LIMIT_MS environment variable). Values < 1 are clamped to 1. */
void fp4_set_wait_limit_ms(int64_t ms);

#ifdef __cplusplus
}
#endif

#endif /* FP4_GEMM_H */
