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
// 128 rows x 4 scale blocks, which is exactly one 512-byte 128x4 scale atom:
// a CTA of 128 threads takes a chunk, thread t owns row t of it, loads its four
// blocks with 16-byte loads (all issued before any arithmetic), writes its
// codes with 8- or 16-byte stores and its four scale bytes either into the
// plain row-major matrix or into a 512-byte shared staging atom that one warp
// writes out with 16-byte stores. The grid is persistent (the SM count times
// the CTAs that fit on one SM) and walks chunks along K inside each 128-row band.
//
// Exactness. Every decision is the one the fp32 definition makes:
//   - NVFP4 scale: amax / 6 with IEEE division, then the hardware conversion
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
//   - the code: cvt.rn.satfinite.e2m1x2.f32 on |q| (round to nearest even,
//     saturate at 6) with the sign bit of x put back by hand.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "fp4_quant.h"

namespace fp4q {

constexpr int kChunkRows = 128;    // rows per chunk = rows of one scale atom
constexpr int kChunkBlocks = 4;    // scale blocks per chunk = columns of one scale atom
constexpr int kAtomBytes = 512;

// Four E2M1 bytes from eight non-negative values (round to nearest even, saturating at 6);
// byte j holds value 2j in its low nibble and 2j + 1 in its high nibble.
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

// Sign bits of eight values placed where their codes' sign bits go.
__device__ __forceinline__ uint32_t sign_bits8(const float (&v)[8])
{
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s |= (__float_as_uint(v[2 * j]) >> 31) << (8 * j + 3);
        s |= (__float_as_uint(v[2 * j + 1]) >> 31) << (8 * j + 7);
    }
    return s;
}

// The block's values as fp32 (LINES 16-byte words of raw input).
template <bool BF16, int VEC, int LINES>
__device__ __forceinline__ void unpack(const uint4 (&raw)[LINES], float (&v)[VEC])
{
#pragma unroll
    for (int l = 0; l < LINES; ++l) {
        const uint32_t w[4] = {raw[l].x, raw[l].y, raw[l].z, raw[l].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (BF16) {
                v[8 * l + 2 * i] = __uint_as_float(w[i] << 16);
                v[8 * l + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            } else {
                v[4 * l + i] = __uint_as_float(w[i]);
            }
        }
    }
}

// One block: returns its scale byte and writes VEC / 8 words of codes.
template <bool MX, bool BF16, int VEC, int LINES>
__device__ __forceinline__ uint32_t quant_block(const uint4 (&raw)[LINES], uint32_t (&codes)[VEC / 8])
{
    float v[VEC];
    unpack<BF16, VEC, LINES>(raw, v);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) amax = fmaxf(amax, fabsf(v[i]));

    uint32_t sc;
    float s, rcp;
    if constexpr (MX) {
        const uint32_t bits = __float_as_uint(amax);
        const int ex = static_cast<int>(bits >> 23);
        int fl = ex - 127;                                        // floor(log2 amax), normal amax
        if (ex == 0) fl = (31 - __clz(static_cast<int>(bits))) - 149;   // subnormal amax
        const int e2 = amax == 0.0f ? -127 : max(fl - 2, -127);    // at most 125 for finite amax
        sc = static_cast<uint32_t>(e2 + 127);
        s = 1.0f;                                                  // unused: q = x * 2^-e2 exactly
        rcp = __uint_as_float(static_cast<uint32_t>(127 - e2) << 23);
    } else {
        sc = e4m3_code(amax / 6.0f);
        s = e4m3_value(sc);
        if (s == 0.0f) {
#pragma unroll
            for (int w = 0; w < VEC / 8; ++w) codes[w] = 0;        // zero scale: all codes 0
            return sc;
        }
        rcp = __frcp_rn(s);
    }
#pragma unroll
    for (int w = 0; w < VEC / 8; ++w) {
        float q[8], x8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float a = fabsf(v[8 * w + i]);
            x8[i] = v[8 * w + i];
            if constexpr (MX) {
                q[i] = a * rcp;
            } else {
                const float q0 = a * rcp;
                const float r = fmaf(-q0, s, a);
                q[i] = fmaf(r, rcp, q0);
            }
        }
        codes[w] = e2m1x8(q) | sign_bits8(x8);
    }
    return sc;
}

template <bool MX, bool BF16>
__global__ void __launch_bounds__(kChunkRows) quantize_kernel(const uint8_t *__restrict__ X,
                                                              uint8_t *__restrict__ codes,
                                                              uint8_t *__restrict__ sf, int64_t rows,
                                                              int64_t K, int64_t nb, int64_t kc4,
                                                              int64_t chunks, int atom_layout, int plain_words)
{
    constexpr int VEC = MX ? 32 : 16;
    constexpr int ESIZE = BF16 ? 2 : 4;
    constexpr int LINES = VEC * ESIZE / 16;            // 16-byte input words per block
    __shared__ uint32_t staging[kChunkRows];            // one scale atom
    const int t = threadIdx.x;
    for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x) {
        const int64_t rb = c / kc4, cb = c - rb * kc4;
        const int64_t r = rb * kChunkRows + t;
        const int64_t b0 = cb * kChunkBlocks;
        const int nblk = nb - b0 < kChunkBlocks ? static_cast<int>(nb - b0) : kChunkBlocks;
        uint32_t scales = 0;
        if (r < rows) {
            const uint4 *src = reinterpret_cast<const uint4 *>(X + (r * K + b0 * VEC) * ESIZE);
            uint4 raw[kChunkBlocks][LINES];
#pragma unroll
            for (int j = 0; j < kChunkBlocks; ++j)
                if (j < nblk)
#pragma unroll
                    for (int l = 0; l < LINES; ++l) raw[j][l] = __ldg(src + j * LINES + l);
            uint8_t *dst = codes + r * (K / 2) + b0 * (VEC / 2);
#pragma unroll
            for (int j = 0; j < kChunkBlocks; ++j) {
                if (j < nblk) {
                    uint32_t w[VEC / 8];
                    scales |= quant_block<MX, BF16, VEC, LINES>(raw[j], w) << (8 * j);
                    if constexpr (MX)
                        *reinterpret_cast<uint4 *>(dst + j * 16) = make_uint4(w[0], w[1], w[2], w[3]);
                    else
                        *reinterpret_cast<uint2 *>(dst + j * 8) = make_uint2(w[0], w[1]);
                }
            }
        }
        if (atom_layout) {
            // row t of the atom: line t % 32, byte group t / 32 (columns in byte order)
            staging[(t & 31) * 4 + (t >> 5)] = scales;
            __syncthreads();
            if (t < 32)
                reinterpret_cast<uint4 *>(sf + c * kAtomBytes)[t] = reinterpret_cast<const uint4 *>(staging)[t];
            __syncthreads();
        } else if (r < rows) {
            uint8_t *row = sf + r * nb + b0;
            if (plain_words && nblk == kChunkBlocks) {
                *reinterpret_cast<uint32_t *>(row) = scales;
            } else {
                for (int j = 0; j < nblk; ++j) row[j] = static_cast<uint8_t>(scales >> (8 * j));
            }
        }
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
    using Kernel = void (*)(const uint8_t *, uint8_t *, uint8_t *, int64_t, int64_t, int64_t, int64_t, int64_t,
                            int, int);
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
    const int words = (nb % 4 == 0) && ((reinterpret_cast<uintptr_t>(sf) & 3u) == 0);
    kern<<<blocks, kChunkRows, 0, stream>>>(static_cast<const uint8_t *>(X), static_cast<uint8_t *>(codes),
                                            static_cast<uint8_t *>(sf), rows, K, nb, kc4, chunks, atom, words);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}
