// fp4_gemv.cu -- the block-scaled FP4 GEMM for one to four rows of A, on CUDA
// cores.
//
// With M <= 4 the GEMM is a matrix-vector product: every byte of B is read
// once and used M times, so the time is the stream of B from HBM and the
// tensor cores have nothing to add (the MXFP4 GEMV workload of "TMA Pipelines,
// Tensor Cores, and ctm-rs Interop", "Where to Go Next"). The arithmetic is
// the block-scaled dot product of "[BUG] Add FP4 TMA kernel example for
// Blackwell in CuTe Python DSL" (CUTLASS issue #2922): per scale block (16
// elements with an E4M3 scale, or 32 with an E8M0 scale), sum the E2M1
// products and multiply by both scales.
//
// Twice an E2M1 value is an integer (magnitudes 0, 1, 2, 3, 4, 6, 8, 12), so
// one block's sum of doubled products is an exact int32, computed with 4-way
// byte dot products (dp4a); it is then multiplied in fp32 by sA * sB / 4 and
// accumulated. A's rows are decoded once per CTA into shared memory as signed
// doubled int8 values. B's codes are decoded in registers: a byte permute of a
// table of the eight doubled magnitudes, with the code's sign bit used as the
// permute's sign-replicate flag, yields the magnitudes of the non-negative
// codes (negative codes give 0); with the sign bit flipped it yields those of
// the negative codes. Two dp4a per four codes then give the positive and the
// negative part of the sum.
//
// Work split: a warp owns two adjacent rows of B (so a SwiGLU gate/up pair
// stays in one warp) and walks K in units of 4096 codes, lane l taking the 128
// codes at 128l of each unit with four 16-byte loads per row; two units live in
// registers, so the next unit's loads are in flight while the current one is
// computed. The grid is sized so that every warp gets the same number of row
// pairs.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "epilogue.cuh"
#include "fp4_gemm.h"
#include "fp4_gemv.cuh"

namespace fp4 {
namespace {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kChunk = 4096;                // codes of a row per unit of a warp's work: 32 lanes x 128 codes
constexpr uint32_t kMagLo = 0x03020100u;    // doubled E2M1 magnitudes of codes 0..3 (bytes 0..3)
constexpr uint32_t kMagHi = 0x0C080604u;    // ... of codes 4..7 (bytes 4..7)
constexpr size_t kGemvSmemLimit = 200 * 1024;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Doubled magnitudes of the four codes in the low 16 bits of `sel`: non-negative
// codes (sign flag clear) in `pos`, negative ones in `neg`, 0 elsewhere.
__device__ __forceinline__ void magnitudes(uint32_t sel, uint32_t &pos, uint32_t &neg)
{
    pos = prmt(kMagLo, kMagHi, sel);
    neg = prmt(kMagLo, kMagHi, sel ^ 0x8888u);
}

// Eight codes (one word, element k in nibble k) dotted with eight int8 values
// (a_lo: elements 0..3, a_hi: 4..7), added to the positive / negative sums.
__device__ __forceinline__ void dot8(uint32_t w, uint32_t a_lo, uint32_t a_hi, int &sp, int &sn)
{
    uint32_t p, n;
    magnitudes(w, p, n);
    sp = __dp4a(static_cast<int>(p), static_cast<int>(a_lo), sp);
    sn = __dp4a(static_cast<int>(n), static_cast<int>(a_lo), sn);
    magnitudes(w >> 16, p, n);
    sp = __dp4a(static_cast<int>(p), static_cast<int>(a_hi), sp);
    sn = __dp4a(static_cast<int>(n), static_cast<int>(a_hi), sn);
}

// Four codes -> four signed doubled values as int8 bytes: (pos + 128 - neg) per
// byte stays in [116, 140] (no borrow between bytes); flipping bit 7 gives the
// two's complement of pos - neg.
__device__ __forceinline__ uint32_t signed_bytes(uint32_t sel)
{
    uint32_t p, n;
    magnitudes(sel, p, n);
    return ((p | 0x80808080u) - n) ^ 0x80808080u;
}

// Scale bytes as values (the sign bit of an E4M3 scale is not read).
__device__ __forceinline__ float e4m3_value(uint32_t b)
{
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    if (e == 0) return static_cast<float>(m) * 0x1p-9f;                  // subnormal: m * 2^-9
    return static_cast<float>(8u + m) * __uint_as_float((e + 117u) << 23);   // (8 + m) * 2^(e - 10)
}

__device__ __forceinline__ float e8m0_value(uint32_t b)
{
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);    // 2^(b - 127); b = 0: 2^-127
}

// Two E4M3 scale bytes (first in bits 0..7) -> their values, by the hardware
// conversion to f16 (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ float2 e4m3x2_values(uint32_t two)
{
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(two));
    __half2 v;
    memcpy(&v, &h, 4);
    return __half22float2(v);
}

// Byte offset of scale (row r, column c) in the plain or the atom layout.
__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t ksf, int64_t kc4, bool atoms)
{
    if (!atoms) return r * ksf + c;
    return ((r >> 7) * kc4 + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

__device__ __forceinline__ uint4 ld_stream16(const uint8_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void store_out(const GemvParams &p, int m, int64_t col, float v)
{
    if (p.bf16)
        static_cast<__nv_bfloat16 *>(p.D)[m * p.ldd + col] = __float2bfloat16_rn(v);
    else
        static_cast<float *>(p.D)[m * p.ldd + col] = v;
}

// Loads of one unit of a warp's work: a 4096-code chunk of two adjacent B rows;
// lane l holds codes 128l .. 128l + 127 of the chunk as four 32-code pieces.
struct Unit {
    uint4 b[2][4];        // [row][piece] codes
    uint32_t s[2][4];     // [row][piece] scale bytes (NVFP4: two, low byte first; MXFP4: one)
};

template <int MR, bool MX, bool ATOMS>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const GemvParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int VEC = MX ? 32 : 16;
    constexpr int SPC = kChunk / VEC;                   // scale columns per chunk
    const int K = p.K;
    const int kp = (K + kChunk - 1) / kChunk * kChunk;  // staged codes per row
    const int ksf = K / VEC;
    const int ksfp = kp / VEC;                          // staged scales per row
    const int kc4 = (ksf + 3) / 4;
    uint8_t *const a8 = smem;                                       // [MR][kp] int8
    float *const sa = reinterpret_cast<float *>(smem + MR * kp);    // [MR][ksfp]: sA / 4

    // ---- A, once per CTA: doubled signed int8 values and sA / 4, laid out so
    // that lane l's loads for piece j of chunk t are contiguous across the warp:
    // codes of 16-code group q (0..7) of lane l at t*4096 + 512q + 16l; NVFP4
    // scale pair of piece j at t*256 + 64j + 2l, MXFP4 scale at t*128 + 32j + l
    const int groups = K / 16;
    for (int i = threadIdx.x; i < MR * groups; i += kGemvThreads) {
        const int m = i / groups, g = i - m * groups;
        const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(p.A + static_cast<int64_t>(m) * (K / 2)) + g);
        const uint4 v = make_uint4(signed_bytes(raw.x), signed_bytes(raw.x >> 16), signed_bytes(raw.y),
                                   signed_bytes(raw.y >> 16));
        const int k = 16 * g, t = k / kChunk, kk = k % kChunk;
        *reinterpret_cast<uint4 *>(a8 + m * kp + t * kChunk + ((kk & 127) >> 4) * 512 + (kk >> 7) * 16) = v;
    }
    for (int i = threadIdx.x; i < MR * ksf; i += kGemvThreads) {
        const int m = i / ksf, c = i - m * ksf;
        const uint32_t b = __ldg(p.sfA + sf_offset(m, c, ksf, kc4, ATOMS));
        const int t = c / SPC, cc = c % SPC;
        const int at = MX ? t * SPC + (cc & 3) * 32 + (cc >> 2)
                          : t * SPC + ((cc & 7) >> 1) * 64 + (cc >> 3) * 2 + (cc & 1);
        sa[m * ksfp + at] = (MX ? e8m0_value(b) : e4m3_value(b)) * 0.25f;
    }
    __syncthreads();

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int pairs = (p.N + 1) / 2;
    const int chunks = kp / kChunk;
    const int64_t row_bytes = K / 2;
    const int stride = gridDim.x * kGemvWarps;
    const int first = blockIdx.x * kGemvWarps + warp;
    const int my_pairs = first < pairs ? (pairs - first + stride - 1) / stride : 0;
    const int units = my_pairs * chunks;

    auto load = [&](Unit &u, int idx) {
        const int r0 = 2 * (first + (idx / chunks) * stride), t = idx % chunks;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int64_t row = r0 + r;
            const bool row_ok = row < p.N;
            const uint8_t *bp = p.B + row * row_bytes + t * (kChunk / 2) + 64 * lane;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                u.b[r][j] = make_uint4(0u, 0u, 0u, 0u);
                u.s[r][j] = 0u;
                if (row_ok && t * kChunk + 128 * lane + 32 * j < K) {
                    u.b[r][j] = ld_stream16(bp + 16 * j);
                    if (MX) {
                        u.s[r][j] = __ldg(p.sfB + sf_offset(row, t * SPC + 4 * lane + j, ksf, kc4, ATOMS));
                    } else {
                        // the pair of scales is adjacent (and 2-byte aligned) in both layouts
                        u.s[r][j] = __ldg(reinterpret_cast<const uint16_t *>(
                            p.sfB + sf_offset(row, t * SPC + 8 * lane + 2 * j, ksf, kc4, ATOMS)));
                    }
                }
            }
        }
    };

    float acc[MR][2];
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m][0] = acc[m][1] = 0.0f;

    auto consume = [&](const Unit &u, int idx) {
        const int pr = first + (idx / chunks) * stride, t = idx % chunks;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (t * kChunk + 128 * lane + 32 * j < K) {
                float2 sb[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (MX) {
                        sb[r].x = e8m0_value(u.s[r][j]);
                        sb[r].y = 0.0f;
                    } else {
                        sb[r] = e4m3x2_values(u.s[r][j]);
                    }
                }
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    const uint8_t *am = a8 + m * kp + t * kChunk + 1024 * j + 16 * lane;
                    const uint4 alo = *reinterpret_cast<const uint4 *>(am);          // codes 0..15 of the piece
                    const uint4 ahi = *reinterpret_cast<const uint4 *>(am + 512);    // codes 16..31
                    if (MX) {
                        const float s_a = sa[m * ksfp + t * SPC + 32 * j + lane];
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            int sp = 0, sn = 0;
                            dot8(u.b[r][j].x, alo.x, alo.y, sp, sn);
                            dot8(u.b[r][j].y, alo.z, alo.w, sp, sn);
                            dot8(u.b[r][j].z, ahi.x, ahi.y, sp, sn);
                            dot8(u.b[r][j].w, ahi.z, ahi.w, sp, sn);
                            acc[m][r] = fmaf(static_cast<float>(sp - sn), s_a * sb[r].x, acc[m][r]);
                        }
                    } else {
                        const float2 s_a = *reinterpret_cast<const float2 *>(sa + m * ksfp + t * SPC + 64 * j + 2 * lane);
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            int sp0 = 0, sn0 = 0, sp1 = 0, sn1 = 0;
                            dot8(u.b[r][j].x, alo.x, alo.y, sp0, sn0);
                            dot8(u.b[r][j].y, alo.z, alo.w, sp0, sn0);
                            dot8(u.b[r][j].z, ahi.x, ahi.y, sp1, sn1);
                            dot8(u.b[r][j].w, ahi.z, ahi.w, sp1, sn1);
                            acc[m][r] = fmaf(static_cast<float>(sp0 - sn0), s_a.x * sb[r].x, acc[m][r]);
                            acc[m][r] = fmaf(static_cast<float>(sp1 - sn1), s_a.y * sb[r].y, acc[m][r]);
                        }
                    }
                }
            }
        }
        if (t != chunks - 1) return;
        // the pair is complete: warp sums (fixed butterfly order), the fused
        // epilogue on lane 0, and fresh accumulators
        const int r0 = 2 * pr;
        const bool has1 = r0 + 1 < p.N;
#pragma unroll
        for (int m = 0; m < MR; ++m)
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[m][r] += __shfl_xor_sync(0xFFFFFFFFu, acc[m][r], o);
        if (lane == 0) {
            const float b0 = p.bias ? p.bias[r0] : 0.0f;
            const float b1 = (p.bias && has1) ? p.bias[r0 + 1] : 0.0f;
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                const float z0 = p.bias ? fmaf(acc[m][0], p.alpha, b0) : acc[m][0] * p.alpha;
                const float z1 = p.bias ? fmaf(acc[m][1], p.alpha, b1) : acc[m][1] * p.alpha;
                if (p.act == FP4_ACT_SWIGLU) {
                    store_out(p, m, r0 / 2, silu(z0) * z1);
                } else {
                    store_out(p, m, r0, activate(z0, p.act));
                    if (has1) store_out(p, m, r0 + 1, activate(z1, p.act));
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[m][0] = acc[m][1] = 0.0f;
    };

    // two units in registers: the next one's loads are in flight while the
    // current one is computed
    Unit u0, u1;
    if (units > 0) load(u0, 0);
    for (int idx = 0; idx < units; idx += 2) {
        if (idx + 1 < units) load(u1, idx + 1);
        consume(u0, idx);
        if (idx + 1 >= units) break;
        if (idx + 2 < units) load(u0, idx + 2);
        consume(u1, idx + 1);
    }
}

template <int MR, bool MX, bool ATOMS>
cudaError_t launch(const GemvParams &p, int sms, size_t smem, cudaStream_t stream)
{
    auto kern = gemv_kernel<MR, MX, ATOMS>;
    // the shared-memory opt-in is raised to the largest size seen (per process;
    // one device family), the occupancy looked up again only when smem changes
    static std::atomic<size_t> opted{0};
    static std::atomic<uint64_t> occ{0};     // smem << 8 | CTAs per SM
    cudaError_t e;
    if (smem > opted.load()) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kGemvSmemLimit));
        if (e != cudaSuccess) return e;
        opted.store(kGemvSmemLimit);
    }
    int per_sm = 0;
    const uint64_t o = occ.load();
    if (o >> 8 == smem && (o & 255u)) {
        per_sm = static_cast<int>(o & 255u);
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGemvThreads, smem);
        if (e != cudaSuccess) return e;
        per_sm = std::min(std::max(per_sm, 1), 255);
        occ.store((static_cast<uint64_t>(smem) << 8) | static_cast<uint64_t>(per_sm));
    }
    // every warp gets the same number of row pairs: rounds = ceil(pairs / resident warps)
    const int64_t pairs = (static_cast<int64_t>(p.N) + 1) / 2;
    const int64_t resident = static_cast<int64_t>(sms) * per_sm * kGemvWarps;
    const int64_t rounds = (pairs + resident - 1) / resident;
    const int64_t warps = (pairs + rounds - 1) / rounds;
    const int64_t blocks = (warps + kGemvWarps - 1) / kGemvWarps;
    kern<<<static_cast<unsigned>(blocks), kGemvThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t gemv_smem_bytes(int64_t M, int64_t K, bool mx)
{
    if (M < 1 || M > kGemvMaxM || K <= 0) return 0;
    const int64_t kp = (K + kChunk - 1) / kChunk * kChunk;
    const size_t bytes = static_cast<size_t>(M * kp + M * (kp / (mx ? 32 : 16)) * 4);
    return bytes <= kGemvSmemLimit ? bytes : 0;
}

cudaError_t launch_gemv(const GemvParams &p, int sms, cudaStream_t stream)
{
    const size_t smem = gemv_smem_bytes(p.M, p.K, p.mx != 0);
    if (!smem) return cudaErrorInvalidValue;
    const int sel = (p.M - 1) * 4 + (p.mx ? 2 : 0) + (p.atoms ? 1 : 0);
    switch (sel) {
#define FP4_GEMV_CASE(MR_, MX_, AT_) \
    case (MR_ - 1) * 4 + (MX_ ? 2 : 0) + (AT_ ? 1 : 0): return launch<MR_, MX_, AT_>(p, sms, smem, stream);
#define FP4_GEMV_ROWS(MR_) \
    FP4_GEMV_CASE(MR_, false, false) FP4_GEMV_CASE(MR_, false, true) FP4_GEMV_CASE(MR_, true, false) \
    FP4_GEMV_CASE(MR_, true, true)
        FP4_GEMV_ROWS(1) FP4_GEMV_ROWS(2) FP4_GEMV_ROWS(3) FP4_GEMV_ROWS(4)
#undef FP4_GEMV_ROWS
#undef FP4_GEMV_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fp4
