// fp4_quant.cu -- online quantisation for the block-scaled FP4 GEMM on GB300
// (sm_103a) behind the C ABI of include/fp4_quant.h.
//
// Rows of fp32 or bf16 values become E2M1 codes (two per byte, low nibble =
// even element) plus one scale per block: NVFP4 (E4M3, 16 values; "[BUG] Add
// FP4 TMA kernel example for Blackwell in CuTe Python DSL", sections "Scale
// Factor Granularity" and "Code Reference") or MXFP4 (E8M0, 32 values; "TMA
// Pipelines, Tensor Cores, and ctm-rs Interop", section 1). The scale rule is
// the absmax rule stated in the header.
//
// The step is bound by HBM: about 2.6 bytes move per value (bf16 in, half a
// byte of code and 1/16 or 1/32 byte of scale out). Work unit = one "chunk" of
// 128 rows x 4 scale blocks, which is exactly one 512-byte 128x4 scale atom.
// A CTA of 128 threads takes a chunk; lanes run along K (a 16-byte piece each,
// whole 128-byte lines per warp-wide load), the block maximum is reduced over
// the block's 2-8 lanes with shuffles, and each lane stores the codes of its
// piece (2 or 4 bytes, whole 32-byte sectors per row). The first lane of each
// block writes the scale byte into the plain row-major matrix or into a
// 512-byte shared staging atom that one warp writes out with 16-byte stores.
// The grid is persistent (the SM count times the CTAs that fit on one SM) and
// walks chunks along K inside each 128-row band.
//
// Exactness. Every decision is the one the fp32 definition makes:
//   - NVFP4 scale: RN(amax / 6) (by the residual step below, which gives the
//     correctly rounded quotient), then the hardware conversion
//     cvt.rn.satfinite.e4m3x2.f32 (round to nearest even, saturate at 448);
//   - MXFP4 scale: the exponent field of amax (subnormals through the count of
//     leading zeros), so floor(log2 amax) is exact;
//   - q = x / s rounded to fp32: for MXFP4 s is a power of two and x * 2^-e is
//     exact; for NVFP4 the quotient is x * RN(1/s) refined by one residual
//     step, r = fma(-q0, s, x), q = fma(r, RN(1/s), q0), which gives the
//     correctly rounded quotient (P. Markstein, "Computation of elementary
//     functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34,
//     1990: a correctly rounded reciprocal and one such correction yield the
//     correctly rounded quotient);
//   - the code: cvt.rn.satfinite.e2m1x2.f32 on q (round to nearest even,
//     saturate at +-6, sign kept, so -0 gives code 8), with the sign bit of x
//     copied onto q first because the residual step turns -0 into +0.
//   - RN(1/s) for the 127 finite E4M3 values comes from a per-CTA table filled
//     with the correctly rounded reciprocal at kernel start.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "fp4_quant.h"

namespace fp4q {

constexpr int kChunkRows = 128;    // rows per chunk = rows of one scale atom
constexpr int kChunkBlocks = 4;    // scale blocks per chunk = columns of one scale atom
constexpr int kAtomBytes = 512;

// Four E2M1 bytes from eight values (round to nearest even, saturating at +-6,
// the sign kept: -0 and negatives that round to zero give code 8); byte j
// holds value 2j in its low nibble and 2j + 1 in its high nibble.
__device__ __forceinline__ uint32_t e2m1x8(const float (&q)[8])
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
    return r;
}

// Non-negative fp32 -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_code(float t)
{
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(t));
    return h & 0xFFu;
}

// E4M3 byte (sign 0, not NaN) -> its value: bias 7; exponent 0 is m * 2^-9.
__device__ __forceinline__ float e4m3_value(uint32_t c)
{
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    if (e == 0) return static_cast<float>(m) * 0.001953125f;
    return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// RN(a / 6) for finite a >= 0: a * RN(1/6), then one residual step (the same
// correctly rounded quotient as the division, by the theorem cited above).
__device__ __forceinline__ float div6(float a)
{
    const float y = 0.16666667163372039794921875f;          // RN(1/6)
    const float q0 = a * y;
    const float r = fmaf(-q0, 6.0f, a);
    return fmaf(r, y, q0);
}

// q with the sign bit of x (the residual step of the quotient loses the sign of -0).
__device__ __forceinline__ float with_sign_of(float q, float x)
{
    return __uint_as_float((__float_as_uint(q) & 0x7FFFFFFFu) | (__float_as_uint(x) & 0x80000000u));
}

// Lane geometry of one chunk (128 rows x 4 scale blocks). A lane owns a
// 16-byte piece of a row (8 bf16 or 4 fp32 values); L consecutive lanes hold
// one scale block, P consecutive lanes one chunk row, so every warp-wide load
// reads whole 128-byte lines (32 / P rows of the chunk, P x 16 contiguous
// bytes each). A pass covers 128 / P rows; 8 passes are a step, whose 8 loads
// a thread issues before it quantises any of them.
template <bool MX, bool BF16>
struct Geo {
    static constexpr int VEC = MX ? 32 : 16;
    static constexpr int ESIZE = BF16 ? 2 : 4;
    static constexpr int EPL = 16 / ESIZE;                 // values per lane piece: 8 or 4
    static constexpr int L = VEC / EPL;                    // lanes per scale block: 2, 4 or 8
    static constexpr int P = kChunkBlocks * L;             // lanes per chunk row: 8, 16 or 32
    static constexpr int RPP = kChunkRows / P;             // chunk rows per pass (128 threads)
    static constexpr int NSTEP = P / 8;                    // steps per chunk (P passes of RPP rows)
    static_assert(P <= 32 && kChunkRows % P == 0, "lane geometry");
};

// The piece's values as fp32.
template <bool BF16, int EPL>
__device__ __forceinline__ void unpack(const uint4 &raw, float (&v)[EPL])
{
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            v[i] = __uint_as_float(w[i]);
        }
    }
}

// Quantises one lane piece: `amax` is the block's (already reduced over its
// lanes); s_val / s_rcp hold each E4M3 byte's value and RN(1 / value). Returns
// the scale byte; `out` gets EPL / 2 code bytes (low byte first).
template <bool MX, int EPL>
__device__ __forceinline__ uint32_t quant_piece(const float (&v)[EPL], float amax, const float *s_val,
                                                const float *s_rcp, uint32_t &out)
{
    uint32_t sc;
    float s, rcp;
    if constexpr (MX) {
        const uint32_t bits = __float_as_uint(amax);
        const int ex = static_cast<int>(bits >> 23);
        int fl = ex - 127;                                              // floor(log2 amax), normal amax
        if (ex == 0) fl = (31 - __clz(static_cast<int>(bits))) - 149;   // subnormal amax
        const int e2 = amax == 0.0f ? -127 : max(fl - 2, -127);          // at most 125 for finite amax
        sc = static_cast<uint32_t>(e2 + 127);
        s = 1.0f;                                                        // unused: q = x * 2^-e2 exactly
        rcp = __uint_as_float(static_cast<uint32_t>(127 - e2) << 23);
    } else {
        sc = e4m3_code(div6(amax));
        s = s_val[sc];
        if (s == 0.0f) {                                                 // zero scale: all codes 0
            out = 0;
            return sc;
        }
        rcp = s_rcp[sc];
    }
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < EPL) {
            const float x = v[i];
            if constexpr (MX) {
                q[i] = x * rcp;
            } else {
                const float q0 = x * rcp;
                const float r = fmaf(-q0, s, x);
                q[i] = with_sign_of(fmaf(r, rcp, q0), x);
            }
        } else {
            q[i] = 0.0f;
        }
    }
    out = e2m1x8(q);
    return sc;
}

// Per-thread work of one step: the 8 pieces (8 x 16 bytes) of passes
// 8 * st .. 8 * st + 7 of chunk c.
template <bool MX, bool BF16>
struct Work {
    using G = Geo<MX, BF16>;
    const uint8_t *__restrict__ X;
    uint8_t *__restrict__ codes;
    uint8_t *__restrict__ sf;
    int64_t rows, K, nb, kc4;
    int atom_layout;

    __device__ __forceinline__ void load(int64_t c, int st, uint4 (&raw)[8]) const
    {
        const int t = threadIdx.x, piece = t % G::P;
        const int64_t rb = c / kc4, b0 = (c - rb * kc4) * kChunkBlocks;
        const bool col_ok = b0 + piece / G::L < nb;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int64_t r = rb * kChunkRows + (st * 8 + q) * G::RPP + t / G::P;
            raw[q] = make_uint4(0, 0, 0, 0);
            if (r < rows && col_ok)
                raw[q] = __ldg(reinterpret_cast<const uint4 *>(X + (r * K + b0 * G::VEC) * G::ESIZE) + piece);
        }
    }

    __device__ __forceinline__ void quantise(int64_t c, int st, const uint4 (&raw)[8], uint8_t *staging,
                                             const float *s_val, const float *s_rcp) const
    {
        const int t = threadIdx.x, piece = t % G::P, j = piece / G::L;
        const bool leader = piece % G::L == 0;                  // writes the block's scale byte
        const int64_t rb = c / kc4, b0 = (c - rb * kc4) * kChunkBlocks;
        const bool col_ok = b0 + j < nb;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int rr = (st * 8 + q) * G::RPP + t / G::P;     // row within the chunk
            const int64_t r = rb * kChunkRows + rr;
            const bool ok = r < rows && col_ok;
            float v[G::EPL];
            unpack<BF16, G::EPL>(raw[q], v);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < G::EPL; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
            for (int o = 1; o < G::L; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            uint32_t out;
            const uint32_t sc = quant_piece<MX, G::EPL>(v, amax, s_val, s_rcp, out);
            if (ok) {
                uint8_t *dst = codes + r * (K / 2) + (b0 * G::VEC) / 2 + piece * (G::EPL / 2);
                if constexpr (BF16)
                    *reinterpret_cast<uint32_t *>(dst) = out;
                else
                    *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(out);
            }
            if (leader) {
                if (atom_layout)
                    staging[(rr & 31) * 16 + (rr >> 5) * 4 + j] = ok ? static_cast<uint8_t>(sc) : 0;
                else if (ok)
                    sf[r * nb + b0 + j] = static_cast<uint8_t>(sc);
            }
        }
    }

    // After a chunk's last step: the staged atom goes out in 16-byte stores.
    __device__ __forceinline__ void finish(int64_t c, const uint8_t *staging) const
    {
        if (!atom_layout) return;
        __syncthreads();
        if (threadIdx.x < 32)
            reinterpret_cast<uint4 *>(sf + c * kAtomBytes)[threadIdx.x] = reinterpret_cast<const uint4 *>(staging)[threadIdx.x];
        __syncthreads();
    }
};

// Persistent loop over chunks; each step's 8 loads are issued together before
// the step is quantised (more resident CTAs, not a second register buffer,
// keep the loads of other CTAs in flight meanwhile).
template <bool MX, bool BF16>
__global__ void __launch_bounds__(kChunkRows) quantize_kernel(const uint8_t *__restrict__ X,
                                                              uint8_t *__restrict__ codes,
                                                              uint8_t *__restrict__ sf, int64_t rows,
                                                              int64_t K, int64_t nb, int64_t kc4,
                                                              int64_t chunks, int atom_layout)
{
    using G = Geo<MX, BF16>;
    __shared__ __align__(16) uint8_t staging[kAtomBytes];    // one scale atom
    __shared__ float s_val[128], s_rcp[128];                  // E4M3 byte -> value, RN(1 / value)
    if (!MX) {
        const float val = e4m3_value(threadIdx.x);
        s_val[threadIdx.x] = val;
        s_rcp[threadIdx.x] = val != 0.0f ? __frcp_rn(val) : 0.0f;
        __syncthreads();
    }
    const Work<MX, BF16> w{X, codes, sf, rows, K, nb, kc4, atom_layout};
    for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x) {
#pragma unroll 1
        for (int st = 0; st < G::NSTEP; ++st) {
            uint4 raw[8];
            w.load(c, st, raw);
            w.quantise(c, st, raw, staging, s_val, s_rcp);
        }
        w.finish(c, staging);
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace fp4q

extern "C" fp4_status fp4_quantize(fp4_format fmt, const void *X, fp4_in_dtype in, int64_t rows, int64_t K,
                                   void *codes, void *sf, fp4_sf_layout layout, cudaStream_t stream)
{
    using namespace fp4q;
    if (fmt != FP4_FMT_NVFP4 && fmt != FP4_FMT_MXFP4) return FP4_ERR_INVALID_ARG;
    if (in != FP4_IN_F32 && in != FP4_IN_BF16) return FP4_ERR_INVALID_ARG;
    if (layout != FP4_SF_PLAIN && layout != FP4_SF_ATOM) return FP4_ERR_INVALID_ARG;
    if (rows < 0 || K < 0) return FP4_ERR_INVALID_ARG;
    if (K % 32 != 0) return FP4_ERR_UNSUPPORTED;
    if (rows == 0 || K == 0) return FP4_OK;
    if (!X || !codes || !sf) return FP4_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(codes) || (layout == FP4_SF_ATOM && !aligned16(sf))) return FP4_ERR_MISALIGNED;
    if (rows > (int64_t(1) << 40) / K) return FP4_ERR_UNSUPPORTED;      // element index range
    const bool mx = fmt == FP4_FMT_MXFP4;
    const int64_t vec = mx ? 32 : 16;
    const int64_t nb = K / vec;
    const int64_t kc4 = (nb + kChunkBlocks - 1) / kChunkBlocks;
    const int64_t chunks = (rows + kChunkRows - 1) / kChunkRows * kc4;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return FP4_ERR_NO_DEVICE;
    using Kernel = void (*)(const uint8_t *, uint8_t *, uint8_t *, int64_t, int64_t, int64_t, int64_t, int64_t, int);
    const Kernel kern = mx ? (in == FP4_IN_BF16 ? quantize_kernel<true, true> : quantize_kernel<true, false>)
                           : (in == FP4_IN_BF16 ? quantize_kernel<false, true> : quantize_kernel<false, false>);
    // persistent grid: every SM filled to the kernel's occupancy
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kChunkRows, 0) != cudaSuccess || per_sm <= 0) {
        cudaGetLastError();
        per_sm = 4;
    }
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>(chunks, int64_t(sms) * per_sm));
    const int atom = layout == FP4_SF_ATOM;
    kern<<<blocks, kChunkRows, 0, stream>>>(static_cast<const uint8_t *>(X), static_cast<uint8_t *>(codes),
                                            static_cast<uint8_t *>(sf), rows, K, nb, kc4, chunks, atom);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}
