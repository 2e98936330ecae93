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
// 256 rows x 4 scale blocks: two 128-row bands, each exactly one 512-byte 128x4
// scale atom (one band when a row of the chunk is 512 bytes, fp32 MXFP4).
// One persistent CTA per SM: a producer thread streams the CTA's chunks into a
// ring of shared-memory stages with tensor-map (TMA) copies, so that the input
// keeps flowing from HBM while sixteen consumer warps convert what has landed.
// Every consumer warp takes 8 rows of each band of every chunk and each of its
// lanes one whole scale block of one row (16 or 32 values, 32 to 128 bytes), so the
// block maximum, the scale and its reciprocal are worked out once per block by
// the lane that converts it; a lane stores its block's codes in one 8- or
// 16-byte store (a warp writes whole 32-byte sectors) and its scale byte into
// the plain row-major matrix or at its place in the chunk's atom. Rows and
// blocks past the matrix arrive as zeros (the copy's fill) and are not stored,
// except as the atom's zero padding.
//
// Exactness. Every decision is the one the fp32 definition makes:
//   - NVFP4 scale: RN(amax / 6) (by the residual step below, which gives the
//     correctly rounded quotient), then the hardware conversion
//     cvt.rn.satfinite.e4m3x2.f32 (round to nearest even, saturate at 448);
//   - MXFP4 scale: the exponent field of amax (subnormals through the count of
//     leading zeros), so floor(log2 amax) is exact;
//   - q = x / s rounded to fp32: for MXFP4 s is a power of two and x * 2^-e is
//     exact; for NVFP4 the quotient is q0 = x * RN(1/s) refined by one residual
//     step, e = fma(q0, s, -x), q = fma(-e, RN(1/s), q0), which gives the
//     correctly rounded quotient (P. Markstein, "Computation of elementary
//     functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34,
//     1990: a correctly rounded reciprocal and one such correction yield the
//     correctly rounded quotient). Written with the residual's sign flipped
//     (q0 s - x rather than x - q0 s), the step also keeps the sign of a zero
//     quotient: x = -0 gives e = +0 and q = (-0) + (-0) = -0;
//   - the code: cvt.rn.satfinite.e2m1x2.f32 on q (round to nearest even,
//     saturate at +-6, sign kept, so -0 gives code 8).
//   - RN(1/s) for the 127 finite E4M3 values comes from a per-CTA table filled
//     with the correctly rounded reciprocal at kernel start.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "fp4_quant.h"
#include "ptx.cuh"

namespace fp4q {

constexpr int kBandRows = 128;     // rows of one scale atom
constexpr int kChunkBlocks = 4;    // scale blocks per chunk = columns of one scale atom
constexpr int kAtomBytes = 512;
constexpr int kConsumerWarps = 16;                   // each takes 8 rows of every chunk
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + the producer warp
constexpr int kRingBytes = 192 * 1024;              // shared memory for the stages
constexpr int kMaxStages = 12;

// The first error of a quantiser launch on this device (0 = none); read and
// cleared by fp4::quant_take_device_status() (part of fp4_get_device_status).
__device__ int g_quant_status;

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

// Geometry of one chunk: ROWS rows x 4 scale blocks, ROWS = 256 (two 128-row
// bands, i.e. two scale atoms) while a row of the chunk is at most 256 bytes,
// else 128. The stage holds the chunk as SLABS column slabs of ROWS rows x 128
// bytes each (one copy per slab), stored with the 128-byte swizzle: the
// 16-byte unit u of row r sits at unit u ^ (r % 8) of that row. A lane owns one
// whole scale block in each band of the chunk (CPL 16-byte units); the eight
// lanes of a quarter-warp hold the same block of eight consecutive rows, so
// each of their shared-memory loads hits eight different bank groups.
template <bool MX, bool BF16>
struct Geo {
    static constexpr int VEC = MX ? 32 : 16;
    static constexpr int ESIZE = BF16 ? 2 : 4;
    static constexpr int EPU = 16 / ESIZE;                 // values per 16-byte unit: 8 or 4
    static constexpr int CPL = VEC / EPU;                  // units per block (per lane): 2, 4 or 8
    static constexpr int ROW_BYTES = kChunkBlocks * VEC * ESIZE;     // 128, 256 or 512
    static constexpr int BANDS = ROW_BYTES <= 256 ? 2 : 1;           // 128-row bands per chunk
    static constexpr int ROWS = BANDS * kBandRows;
    static constexpr int SLABS = ROW_BYTES / 128;                    // 1, 2 or 4
    static constexpr int SLAB_ELEMS = 128 / ESIZE;                   // values across one slab
    static constexpr int SLAB_BYTES = ROWS * 128;
    static constexpr int CHUNK_BYTES = SLABS * SLAB_BYTES;          // one stage: 32, 64 or 64 KB
    static constexpr int STAGES = kRingBytes / CHUNK_BYTES < kMaxStages ? kRingBytes / CHUNK_BYTES : kMaxStages;
    static constexpr int SMEM_BYTES = STAGES * CHUNK_BYTES + 1024;  // + alignment slack
    static_assert(kBandRows / kConsumerWarps == 8 && kChunkBlocks == 4, "a warp = 8 rows x 4 blocks per band");
    static_assert(STAGES >= 3, "ring depth");
};

// Converts one block: `raw` holds its VEC values in order; `out` gets the
// VEC / 2 code bytes (low byte first) and the scale byte is returned. s_val /
// s_rcp hold each E4M3 byte's value and RN(1 / value).
template <bool MX, bool BF16>
__device__ __forceinline__ uint32_t quant_block(const uint4 (&raw)[Geo<MX, BF16>::CPL], const float *s_val,
                                                const float *s_rcp, uint32_t (&out)[Geo<MX, BF16>::VEC / 8])
{
    using G = Geo<MX, BF16>;
    float v[G::VEC];
#pragma unroll
    for (int u = 0; u < G::CPL; ++u) {
        const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (BF16) {
                v[u * 8 + 2 * i] = __uint_as_float(w[i] << 16);
                v[u * 8 + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            } else {
                v[u * 4 + i] = __uint_as_float(w[i]);
            }
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < G::VEC; ++i) amax = fmaxf(amax, fabsf(v[i]));
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
        rcp = s_rcp[sc];                                                 // 0 for the zero scale
    }
#pragma unroll
    for (int g = 0; g < G::VEC / 8; ++g) {
        float q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float x = v[8 * g + i];
            if constexpr (MX) {
                q[i] = x * rcp;
            } else {
                const float q0 = x * rcp;
                const float e = fmaf(q0, s, -x);
                q[i] = fmaf(-e, rcp, q0);
            }
        }
        out[g] = e2m1x8(q);
        if constexpr (!MX) out[g] = s == 0.0f ? 0u : out[g];             // zero scale: all codes 0
    }
    return sc;
}

// Bounded wait on a barrier of this CTA: false when the time bound runs out
// (the error is recorded and the CTA's abort flag raised) or when another role
// of the CTA already gave up. The teardown wait passes no flag.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                       volatile uint32_t *abort_flag)
{
    const uint64_t t0 = fp4::global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (fp4::mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (abort_flag && *abort_flag != 0) return false;
            if (fp4::global_timer_ns() - t0 > limit_ns) {
                atomicCAS(&g_quant_status, 0, static_cast<int>(FP4_ERR_TIMEOUT));
                if (abort_flag) *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile uint32_t *abort_flag)
{
    if (fp4::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, limit_ns, abort_flag);
}

struct QArgs {
    uint8_t *codes;
    uint8_t *sf;
    int rows, K;
    int nb, kc4;                  // scale blocks per row; chunks (and atoms) per band of rows
    int chunks;
    int atom_layout;
    uint64_t wait_ns;
};

// The chunk a CTA works on, advanced by the grid size without a division:
// chunk row cr (ROWS rows), chunk column cb (4 scale blocks).
struct ChunkPos {
    int cr, cb;
    int step_cr, step_cb;         // gridDim.x as whole chunk rows and the rest

    __device__ __forceinline__ void start(int kc4)
    {
        cr = static_cast<int>(blockIdx.x) / kc4;
        cb = static_cast<int>(blockIdx.x) - cr * kc4;
        step_cr = static_cast<int>(gridDim.x) / kc4;
        step_cb = static_cast<int>(gridDim.x) - step_cr * kc4;
    }
    __device__ __forceinline__ void next(int kc4)
    {
        cr += step_cr;
        cb += step_cb;
        if (cb >= kc4) {
            cb -= kc4;
            ++cr;
        }
    }
};

// Per-lane constants: in band h of a chunk the lane converts block p of row
// 128 h + rr (rr = 8 warp + lane % 8, p = lane / 8); where its units sit in a
// stage does not depend on the chunk.
template <bool MX, bool BF16>
struct LaneGeo {
    using G = Geo<MX, BF16>;
    int p, rr;
    uint32_t unit[G::CPL];        // byte offset of each 16-byte unit of the band-0 block in a stage

    __device__ __forceinline__ void init(int warp, int lane)
    {
        p = lane >> 3;
        rr = warp * 8 + (lane & 7);
#pragma unroll
        for (int u = 0; u < G::CPL; ++u) {
            const int lu = p * G::CPL + u;                   // unit index along the row
            unit[u] = static_cast<uint32_t>((lu >> 3) * G::SLAB_BYTES + rr * 128 + (((lu & 7) ^ (rr & 7)) << 4));
        }
    }
};

// The lane's blocks of chunk `pos`, read from the stage at `stage` (a
// shared-window address).
template <bool MX, bool BF16>
__device__ __forceinline__ void quantise_blocks(const QArgs &a, const ChunkPos &pos, const LaneGeo<MX, BF16> &lg,
                                                uint32_t stage, const float *s_val, const float *s_rcp)
{
    using G = Geo<MX, BF16>;
    uint4 raw[G::BANDS][G::CPL];
#pragma unroll
    for (int h = 0; h < G::BANDS; ++h)
#pragma unroll
        for (int u = 0; u < G::CPL; ++u)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(raw[h][u].x), "=r"(raw[h][u].y), "=r"(raw[h][u].z), "=r"(raw[h][u].w)
                         : "r"(stage + lg.unit[u] + h * kBandRows * 128));   // (row + 128: same swizzle)
    const int blk = pos.cb * kChunkBlocks + lg.p;          // the block's index along the row
    const bool col_ok = blk < a.nb;
#pragma unroll
    for (int h = 0; h < G::BANDS; ++h) {
        uint32_t out[G::VEC / 8];
        const uint32_t sc = quant_block<MX, BF16>(raw[h], s_val, s_rcp, out);
        const int band = pos.cr * G::BANDS + h;
        const int row = band * kBandRows + lg.rr;
        const bool ok = row < a.rows && col_ok;
        if (ok) {
            uint8_t *dst = a.codes + static_cast<int64_t>(row) * (a.K / 2) + blk * (G::VEC / 2);
            if constexpr (G::VEC == 16)
                *reinterpret_cast<uint2 *>(dst) = make_uint2(out[0], out[1]);
            else
                *reinterpret_cast<uint4 *>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
        }
        if (a.atom_layout) {
            // every byte of an atom is written: rows and blocks past the matrix
            // arrived as zeros, whose scale byte is 0 in both formats; a band
            // wholly past the matrix has no atom
            if (band * kBandRows < a.rows)
                a.sf[(static_cast<int64_t>(band) * a.kc4 + pos.cb) * kAtomBytes + (lg.rr & 31) * 16 +
                     (lg.rr >> 5) * 4 + lg.p] = static_cast<uint8_t>(sc);
        } else if (ok) {
            a.sf[static_cast<int64_t>(row) * a.nb + blk] = static_cast<uint8_t>(sc);
        }
    }
}

// Persistent: CTA b takes chunks b, b + grid, ... The producer (warp 16, one
// lane) fills stage i % STAGES with the CTA's i-th chunk once all sixteen
// consumer warps have released the stage's previous chunk; every consumer warp
// takes every chunk in order, so each barrier phase a warp waits for is the one
// after the last it saw.
template <bool MX, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) quantize_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                                               const QArgs a)
{
    using G = Geo<MX, BF16>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ float s_val[128], s_rcp[128];                  // E4M3 byte -> value, RN(1 / value)
    __shared__ __align__(8) uint64_t bars[2 * G::STAGES];     // full, then empty
    __shared__ uint32_t abort_flag;
    const uint32_t ring = (fp4::smem_u32(smem_raw) + 1023u) & ~1023u;   // (the swizzle's 1024-byte period)
    const uint32_t full0 = fp4::smem_u32(bars), empty0 = full0 + 8 * G::STAGES;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (!MX && threadIdx.x < 128) {
        const float val = e4m3_value(threadIdx.x);
        s_val[threadIdx.x] = val;
        s_rcp[threadIdx.x] = val != 0.0f ? __frcp_rn(val) : 0.0f;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < G::STAGES; ++s) {
            fp4::mbar_init(full0 + 8 * s, 1);
            fp4::mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        abort_flag = 0;
        fp4::fence_mbarrier_init();
    }
    if (threadIdx.x == 32 * kConsumerWarps) fp4::prefetch_tensormap(&tmap_x);
    __syncthreads();
    const int mine = a.chunks > static_cast<int>(blockIdx.x)
                         ? (a.chunks - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                         : 0;
    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            ChunkPos pos;
            pos.start(a.kc4);
            int s = 0;
            uint32_t phase = 0;
            for (int i = 0; i < mine; ++i) {
                if (i >= G::STAGES && !wait(empty0 + 8 * s, phase ^ 1u, a.wait_ns, &abort_flag)) break;
                fp4::mbar_arrive_expect_tx(full0 + 8 * s, G::CHUNK_BYTES);
                // x: the slab's first value (a multiple of 32 or 64 values, so 16-byte
                // aligned); y: the chunk's first row. Parts past the matrix fill with 0.
#pragma unroll
                for (int sl = 0; sl < G::SLABS; ++sl)
                    fp4::tma_load_2d<1>(ring + s * G::CHUNK_BYTES + sl * G::SLAB_BYTES, &tmap_x, full0 + 8 * s,
                                        pos.cb * kChunkBlocks * G::VEC + sl * G::SLAB_ELEMS, pos.cr * G::ROWS);
                issued = i + 1;
                pos.next(a.kc4);
                if (++s == G::STAGES) {
                    s = 0;
                    phase ^= 1u;
                }
            }
            // every copy issued lands before the CTA exits
            for (int i = issued > G::STAGES ? issued - G::STAGES : 0; i < issued; ++i)
                wait(full0 + 8 * (i % G::STAGES), static_cast<uint32_t>(i / G::STAGES) & 1u, a.wait_ns, nullptr);
        }
    } else {
        // ------------------------------------------------------------ consumers
        LaneGeo<MX, BF16> lg;
        lg.init(warp, lane);
        ChunkPos pos;
        pos.start(a.kc4);
        int s = 0;
        uint32_t phase = 0;
        for (int i = 0; i < mine; ++i) {
            // every lane waits (the stage's bytes are visible to the lanes that saw
            // it complete); the warp leaves together if any lane gave up
            const bool landed = wait(full0 + 8 * s, phase, a.wait_ns, &abort_flag);
            if (!__all_sync(0xFFFFFFFFu, landed)) break;
            quantise_blocks<MX, BF16>(a, pos, lg, ring + s * G::CHUNK_BYTES, s_val, s_rcp);
            __syncwarp();
            if (lane == 0) fp4::mbar_arrive(empty0 + 8 * s);   // this warp is done with the stage
            pos.next(a.kc4);
            if (++s == G::STAGES) {
                s = 0;
                phase ^= 1u;
            }
        }
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using Kernel = void (*)(const CUtensorMap, const QArgs);

// Per device: whether the four kernel variants may use their shared memory.
struct DeviceState {
    bool probed = false;
    bool ok = false;
    int sms = 0;
};
std::mutex g_mu;
DeviceState g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <bool MX, bool BF16>
bool allow_smem()
{
    return cudaFuncSetAttribute(quantize_kernel<MX, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Geo<MX, BF16>::SMEM_BYTES) == cudaSuccess;
}

fp4_status device_state(int &sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP4_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.probed) {
        d.probed = true;
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                    cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        int n = 0;
        d.ok = g_encode && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0 &&
               allow_smem<false, false>() && allow_smem<false, true>() && allow_smem<true, false>() &&
               allow_smem<true, true>();
        d.sms = n;
        if (!d.ok) (void)cudaGetLastError();
    }
    sms = d.sms;
    return d.ok ? FP4_OK : FP4_ERR_NO_DEVICE;
}

}  // namespace fp4q

namespace fp4 {
uint64_t library_wait_limit_ns();     // the GEMM library's bounded-wait limit (fp4_set_wait_limit_ms)

// The quantiser's device status word, read and cleared (part of fp4_get_device_status).
int quant_take_device_status()
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, fp4q::g_quant_status, sizeof v) != cudaSuccess) return FP4_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(fp4q::g_quant_status, &zero, sizeof zero) != cudaSuccess) return FP4_ERR_CUDA;
    }
    return v;
}
}  // namespace fp4

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
    if (rows > INT32_MAX - 1024 || K > INT32_MAX) return FP4_ERR_UNSUPPORTED;   // 32-bit rows and copy coordinates
    const bool mx = fmt == FP4_FMT_MXFP4, bf16 = in == FP4_IN_BF16;
    int sms = 0;
    if (const fp4_status st = device_state(sms)) return st;
    const int64_t vec = mx ? 32 : 16, esize = bf16 ? 2 : 4;
    const int chunk_rows = mx ? (bf16 ? Geo<true, true>::ROWS : Geo<true, false>::ROWS)
                              : (bf16 ? Geo<false, true>::ROWS : Geo<false, false>::ROWS);
    QArgs a;
    a.codes = static_cast<uint8_t *>(codes);
    a.sf = static_cast<uint8_t *>(sf);
    a.rows = static_cast<int>(rows);
    a.K = static_cast<int>(K);
    a.nb = static_cast<int>(K / vec);
    a.kc4 = (a.nb + kChunkBlocks - 1) / kChunkBlocks;
    const int64_t chunks = (rows + chunk_rows - 1) / chunk_rows * a.kc4;
    if (chunks > INT32_MAX) return FP4_ERR_UNSUPPORTED;
    a.chunks = static_cast<int>(chunks);
    a.atom_layout = layout == FP4_SF_ATOM;
    a.wait_ns = fp4::library_wait_limit_ns();
    // X as [rows][K] values; one box = one 128-byte column slab of a chunk (128
    // or 256 rows), 128-byte swizzle; what lies past the matrix reads as 0
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * esize)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(chunk_rows)};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(&map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                 const_cast<void *>(X), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return FP4_ERR_CUDA;
    const Kernel kern = mx ? (bf16 ? quantize_kernel<true, true> : quantize_kernel<true, false>)
                           : (bf16 ? quantize_kernel<false, true> : quantize_kernel<false, false>);
    const int smem = mx ? (bf16 ? Geo<true, true>::SMEM_BYTES : Geo<true, false>::SMEM_BYTES)
                        : (bf16 ? Geo<false, true>::SMEM_BYTES : Geo<false, false>::SMEM_BYTES);
    // persistent grid: one CTA per SM (the ring fills its shared memory)
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>(a.chunks, sms));
    kern<<<blocks, kThreads, smem, stream>>>(map, a);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}
