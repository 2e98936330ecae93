/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the block-scaled FP4 GEMM and
 * for the quantisation step that feeds it (the latter decides in fp32).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library. It shares no code, header,
 * table or constant with the CUDA path, and the product never calls it.
 *
 * What it computes (the plain definition, written out):
 *
 *   D[i][j] = alpha * sum_{k<K} e2m1(A[i][k]) * s(sfA[i][k/vec])
 *                              * e2m1(B[j][k]) * s(sfB[j][k/vec])
 *
 * - "[BUG] Add FP4 TMA kernel example for Blackwell in CuTe Python DSL"
 *   (CUTLASS issue #2922), Summary / Background: a blockwise (block-scaled)
 *   GEMM on Float4E2M1FN operands through the MmaMXF4NVF4Op block-scaled MMA
 *   atom; section "Scale Factor Granularity": FP4 takes one Float8E4M3FN scale
 *   per sf_vec_size = 16 K-elements (NVFP4).
 * - "TMA Pipelines, Tensor Cores, and ctm-rs Interop", section 1
 *   "Block-Scaled MXFP4 GEMM in cute-rs (SM120a)": the MXFP4 variant carries
 *   Float8E8M0FNU scales (one per 32 K-elements).
 * - "Hopper GEMM in CUTLASS C++ and the CuTe DSL, part 1", section "The
 *   operands are swapped", reason 3: both operands of the narrow-type GEMM are
 *   K-major. A is [M][K/2] bytes and B is [N][K/2] bytes; element k = 2j sits
 *   in the low nibble of byte j and k = 2j + 1 in the high nibble.
 *
 * Sums run in fp64 in k order. Every product of two decoded E2M1 values and
 * two decoded scales is exact in fp64 (at most 4 + 4 + 4 + 4 significant bits).
 * The decoders below follow the bit-field definitions of the three formats.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC oracle.c -o _oracle.so
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- element decoders ------------------------------------------------- */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa. No inf/NaN
 * ("FN" = finite). Exponent 0 is subnormal: 0.5 * m. */
double oracle_e2m1(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* E4M3 ("FN" variant): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa. Exponent 0 is subnormal (m * 2^-9). Only S.1111.111 is NaN; there
 * is no infinity, so the largest finite value is 1.75 * 2^8 = 448. */
double oracle_e4m3(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    if (e == 15u && m == 7u) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* E8M0: an unsigned power of two 2^(code - 127); code 255 is NaN. */
double oracle_e8m0(unsigned code)
{
    if (code == 255u) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* One K-block scale, by format: vec 16 -> E4M3 (NVFP4), vec 32 -> E8M0 (MXFP4). */
static double scale_value(unsigned code, int vec)
{
    return vec == 16 ? oracle_e4m3(code) : oracle_e8m0(code);
}

/* Code k of a K-major packed row (low nibble holds the even element). */
static unsigned nibble(const uint8_t *row, int64_t k)
{
    uint8_t byte = row[k >> 1];
    return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 0xF);
}

/* ---- the GEMM ----------------------------------------------------------- */

/* One output element: returns alpha * sum and, through *absdot, |alpha| * sum |a_k b_k|
 * (the scale of the tolerance the parity tests use). */
static double dot_one(const uint8_t *A, const uint8_t *sfA, const uint8_t *B, const uint8_t *sfB,
                      int64_t i, int64_t j, int64_t K, int vec, double alpha, double *absdot)
{
    const int64_t row_bytes = K / 2, ksf = K / vec;
    const uint8_t *a_row = A + i * row_bytes, *b_row = B + j * row_bytes;
    const uint8_t *sa_row = sfA + i * ksf, *sb_row = sfB + j * ksf;
    double sum = 0.0, abs_sum = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double a = oracle_e2m1(nibble(a_row, k)) * scale_value(sa_row[k / vec], vec);
        double b = oracle_e2m1(nibble(b_row, k)) * scale_value(sb_row[k / vec], vec);
        double p = a * b;
        sum += p;
        abs_sum += fabs(p);
    }
    if (absdot) *absdot = fabs(alpha) * abs_sum;
    return alpha * sum;
}

/*
 * Rows variant: D is nrows x N (fp64, before any output rounding), one row per
 * entry of rows[] (rows == NULL means every row 0..M-1, nrows = M).
 * absdot (same shape, may be NULL) receives |alpha| * sum_k |a_k b_k|.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gemm_rows(const uint8_t *A, const uint8_t *sfA, const uint8_t *B, const uint8_t *sfB,
                     int64_t M, int64_t N, int64_t K, int vec, double alpha,
                     const int64_t *rows, int64_t nrows, double *D, double *absdot, int nthreads)
{
    if (vec != 16 && vec != 32) return -1;
    if (M < 0 || N < 0 || K < 0 || K % vec != 0 || K % 2 != 0) return -1;
    if (rows == NULL) nrows = M;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) return -1;
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        for (int64_t j = 0; j < N; ++j) {
            double ad;
            D[r * N + j] = dot_one(A, sfA, B, sfB, i, j, K, vec, alpha, &ad);
            if (absdot) absdot[r * N + j] = ad;
        }
    }
    return 0;
}

/* Pairs variant: out[p] = D[ii[p]][jj[p]] for p < npairs (for sampled checks at
 * sizes where whole rows are too slow). */
int oracle_gemm_pairs(const uint8_t *A, const uint8_t *sfA, const uint8_t *B, const uint8_t *sfB,
                      int64_t M, int64_t N, int64_t K, int vec, double alpha,
                      const int64_t *ii, const int64_t *jj, int64_t npairs,
                      double *out, double *absdot, int nthreads)
{
    if (vec != 16 && vec != 32) return -1;
    if (M < 0 || N < 0 || K < 0 || K % vec != 0 || K % 2 != 0) return -1;
    for (int64_t p = 0; p < npairs; ++p)
        if (ii[p] < 0 || ii[p] >= M || jj[p] < 0 || jj[p] >= N) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t p = 0; p < npairs; ++p) {
        double ad;
        out[p] = dot_one(A, sfA, B, sfB, ii[p], jj[p], K, vec, alpha, &ad);
        if (absdot) absdot[p] = ad;
    }
    return 0;
}

/* ---- output rounding ---------------------------------------------------- */

/* fp64 -> fp32, round to nearest even (the C conversion under the default mode). */
float oracle_round_f32(double x) { return (float)x; }

/* fp64 -> bf16 bits, one rounding, to nearest with ties to even. bf16 keeps 8
 * significant bits and fp32's exponent range (normal down to 2^-126,
 * subnormal quantum 2^-133); overflow goes to infinity. */
uint16_t oracle_round_bf16(double x)
{
    if (isnan(x)) return 0x7FC0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1): leading bit 2^(e-1) */
    int q_exp = (e - 1) - 7;       /* weight of the last kept bit */
    if (q_exp < -133) q_exp = -133;
    double q = nearbyint(ldexp(a, -q_exp)); /* ties to even under the default mode */
    double v = ldexp(q, q_exp);
    if (v >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)v;            /* exact: v has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* Round a whole array (n values) to bf16 bits. */
void oracle_round_bf16_array(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t p = 0; p < n; ++p) out[p] = oracle_round_bf16(x[p]);
}

/* ---- scale-factor atom layout ------------------------------------------- */

/* Bytes of the atom-layout copy of a rows x ksf scale matrix: rows padded to
 * 128, scale columns padded to 4 (one 512-byte atom per 128 x 4 block). */
int64_t oracle_scale_atom_bytes(int64_t rows, int64_t ksf)
{
    int64_t rb = (rows + 127) / 128, cb = (ksf + 3) / 4;
    return rb * cb * 512;
}

/*
 * Plain row-major sf[rows][ksf] -> 128x4 atom layout:
 *   atom (rb, cb) = rows 128rb..128rb+127, scale columns 4cb..4cb+3, stored at
 *   (rb * ceil(ksf/4) + cb) * 512; inside an atom, row r and column c sit at
 *   (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4). Padding bytes are zero.
 * This is the reading of the "128x4 scale atom" used throughout: the pages
 * name the atom (load_scale_atom_128 in "TMA Pipelines, Tensor Cores, and
 * ctm-rs Interop", section 1) but print no byte layout.
 */
void oracle_scale_reorder(const uint8_t *sf, int64_t rows, int64_t ksf, uint8_t *out)
{
    int64_t kc4 = (ksf + 3) / 4;
    memset(out, 0, (size_t)oracle_scale_atom_bytes(rows, ksf));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < ksf; ++c) {
            int64_t atom = (r / 128) * kc4 + c / 4;
            int64_t off = (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);
            out[atom * 512 + off] = sf[r * ksf + c];
        }
}

/* ---- online quantisation: values -> E2M1 codes + one scale per block ------ */
/*
 * The step before the GEMM: an activation row of K values becomes K E2M1
 * codes packed two per byte (low nibble = even k) and one scale byte per
 * block of vec values. The pages fix the formats and the block sizes
 * ("[BUG] Add FP4 TMA kernel example for Blackwell in CuTe Python DSL",
 * "Scale Factor Granularity" and "Code Reference": Float8E4M3FN scales, one per
 * 16 values; "TMA Pipelines, Tensor Cores, and ctm-rs Interop", section 1:
 * Float8E8M0FNU scales for MXFP4) but not how a scale is chosen. The reading
 * taken here:
 *   NVFP4: s = E4M3(amax / 6), the division in fp32, then round to nearest
 *          E4M3 (ties to the even code, saturating at 448);
 *   MXFP4: s = 2^(floor(log2 amax) - 2), exponent clamped to [-127, 127]; an
 *          all-zero block gets 2^-127 (byte 0);
 *   code = E2M1 value nearest to q = x / s, with q rounded to fp32 first; ties
 *          to the even code; |q| >= 6 saturates to 6; the sign bit of x is
 *          kept (so -0 and negatives that round to 0 give code 8). An NVFP4
 *          block whose scale is 0 gets all codes 0.
 * Every decision above is taken in fp32, the precision the kernel works in.
 */

/* Nearest E2M1 code to q: search the eight magnitudes, a tie keeps the even code. */
unsigned oracle_e2m1_encode(float q)
{
    const unsigned sign = signbit(q) ? 8u : 0u;
    const double a = fabs((double)q);
    if (a >= 6.0) return sign | 7u;
    unsigned best = 0;
    for (unsigned c = 1; c < 8; ++c) {
        const double dc = fabs(a - oracle_e2m1(c)), db = fabs(a - oracle_e2m1(best));
        if (dc < db || (dc == db && c % 2 == 0)) best = c;
    }
    return sign | best;
}

/* Nearest E4M3 code to v >= 0 among the finite non-negative codes 0x00..0x7E
 * (a tie keeps the even code); v >= 448 saturates to 448 (0x7E). */
unsigned oracle_e4m3_encode(float v)
{
    if (v >= 448.0f) return 0x7Eu;
    unsigned best = 0;
    for (unsigned c = 1; c <= 0x7Eu; ++c) {
        const double dc = fabs((double)v - oracle_e4m3(c)), db = fabs((double)v - oracle_e4m3(best));
        if (dc < db || (dc == db && c % 2 == 0)) best = c;
    }
    return best;
}

/* One input value as fp32: bf16 bits widen exactly (they are fp32's top half). */
static float load_value(const void *X, int in_bf16, int64_t idx)
{
    if (!in_bf16) return ((const float *)X)[idx];
    uint32_t u = (uint32_t)((const uint16_t *)X)[idx] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * X: rows x K values (fp32, or bf16 bits when in_bf16), row-major.
 * codes: rows x K/2 bytes; sf: rows x K/vec scale bytes, plain row-major.
 * Returns 0, or -1 on a bad argument. Non-finite inputs are outside the
 * definition.
 */
int oracle_quantize(const void *X, int in_bf16, int64_t rows, int64_t K, int vec, uint8_t *codes, uint8_t *sf)
{
    if (vec != 16 && vec != 32) return -1;
    if (rows < 0 || K < 0 || K % vec != 0) return -1;
    const int64_t nb = K / vec;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            float x[32];
            float amax = 0.0f;
            for (int i = 0; i < vec; ++i) {
                x[i] = load_value(X, in_bf16, r * K + b * vec + i);
                amax = fmaxf(amax, fabsf(x[i]));
            }
            unsigned scode;
            float s;
            if (vec == 16) {
                const float t = amax / 6.0f;
                scode = oracle_e4m3_encode(t);
                s = (float)oracle_e4m3(scode);
            } else {
                int e2 = -127;
                if (amax > 0.0f) {
                    int e;
                    (void)frexpf(amax, &e);          /* amax = f * 2^e, f in [0.5, 1) */
                    e2 = (e - 1) - 2;
                    if (e2 < -127) e2 = -127;
                    if (e2 > 127) e2 = 127;
                }
                scode = (unsigned)(e2 + 127);
                s = ldexpf(1.0f, e2);
            }
            sf[r * nb + b] = (uint8_t)scode;
            for (int i = 0; i < vec; i += 2) {
                unsigned lo = 0, hi = 0;
                if (s != 0.0f) {
                    lo = oracle_e2m1_encode(x[i] / s);
                    hi = oracle_e2m1_encode(x[i + 1] / s);
                }
                codes[r * (K / 2) + (b * vec + i) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return 0;
}

/* ---- fused epilogues --------------------------------------------------------- */
/*
 * Applied to the GEMM's unrounded result y[m][n] = alpha * sum_k a_k b_k (the
 * rows of oracle_gemm_rows): z = y + bias[n] (bias may be NULL), then
 *   op 0: z;  op 1: max(z, 0);  op 2: max(z, 0)^2 (squared ReLU);
 *   op 3: SwiGLU over interleaved columns, out[m][j] = silu(z[m][2j]) * z[m][2j+1]
 *         with silu(x) = x / (1 + exp(-x)), for j < N/2.
 * The pages list these as the elementwise work around the GEMM ("TMA Pipelines,
 * Tensor Cores, and ctm-rs Interop", "Where to Go Next": SwiGLU elementwise;
 * the NVFP4 ReLU^2 MoE). Reading: bias before the activation; the gate is the
 * even column of each pair. fp64 throughout (exp from the C library).
 * out has rows x N (ops 0-2) or rows x N/2 (op 3) entries. Returns 0, or -1.
 */
int oracle_epilogue(const double *y, int64_t rows, int64_t N, const float *bias, int op, double *out)
{
    if (rows < 0 || N < 0 || op < 0 || op > 3) return -1;
    if (op == 3 && N % 2 != 0) return -1;
    for (int64_t m = 0; m < rows; ++m) {
        if (op == 3) {
            for (int64_t j = 0; j < N / 2; ++j) {
                double g = y[m * N + 2 * j], u = y[m * N + 2 * j + 1];
                if (bias) {
                    g += (double)bias[2 * j];
                    u += (double)bias[2 * j + 1];
                }
                out[m * (N / 2) + j] = g / (1.0 + exp(-g)) * u;
            }
            continue;
        }
        for (int64_t n = 0; n < N; ++n) {
            double z = y[m * N + n] + (bias ? (double)bias[n] : 0.0);
            if (op >= 1 && z < 0.0) z = 0.0;
            if (op == 2) z = z * z;
            out[m * N + n] = z;
        }
    }
    return 0;
}
