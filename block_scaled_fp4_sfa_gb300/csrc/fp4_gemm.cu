// fp4_gemm.cu -- block-scaled FP4 GEMM for GB300 (sm_103a) behind the C ABI of
// include/fp4_gemm.h.
//
//   D = alpha * decode(A, sfA) . decode(B, sfB)^T
//
// The operation is the block-scaled FP4 GEMM of "[BUG] Add FP4 TMA kernel
// example for Blackwell in CuTe Python DSL" (CUTLASS issue #2922): E2M1
// operands, K = 64 per block-scaled MMA ("MMA Instruction K Constraint"), one
// E4M3 scale per 16 elements ("Scale Factor Granularity") or, for MXFP4, one
// E8M0 scale per 32 ("TMA Pipelines, Tensor Cores, and ctm-rs Interop",
// section 1). The kernel is a persistent, warp-specialised tcgen05 GEMM:
//
//   warp 0      TMA producer: fills a ring of shared-memory stages, each one
//               k-tile (256 FP4 elements = 128 bytes per row) of the two
//               operands (128B-swizzled) plus their scale atoms;
//   warp 1      MMA issuer: one thread copies the scale atoms into TMEM
//               (tcgen05.cp) and issues four K=64 block-scaled MMAs per k-tile
//               into a TMEM accumulator, then releases the stage;
//   warps 2..5  epilogue: TMEM -> registers (tcgen05.ld), * alpha, cast,
//               then either a swizzled shared tile + TMA store, or coalesced
//               direct stores of the transposed tile (swap-AB), or fp32
//               split-K partials.
//
// The warp roles follow the split shown for the SM100a two-CTA kernel in
// "TMA Pipelines, Tensor Cores, and ctm-rs Interop", section 2 (producer warp,
// single-thread MMA warp, epilogue warps draining TMEM); the K-tile of four MMA
// instructions and the 128-byte swizzle follow "Hopper GEMM in CUTLASS C++ and
// the CuTe DSL, part 1" (the K extent of the tile is four MMA instructions;
// the widest swizzle atom that divides the tile's K bytes is taken).
//
// "Slot A" is the operand on the MMA's 128-row M side, "slot B" the one on its
// N side. Direct mode: slot A = A, slot B = B. Swap-AB mode: slot A = B, slot
// B = A, and the epilogue writes D^T tiles into row-major D -- the swapped
// operands of the W4A8 kernel in "Hopper GEMM in CUTLASS C++ and the CuTe DSL,
// part 1" ("The operands are swapped").

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fp4_gemm.h"
#include "ptx.cuh"

namespace fp4 {

// Per-device status word: 0, or the first error a kernel recorded.
__device__ int g_status;

constexpr int kBM = 128;          // MMA M (cta_group::1)
constexpr int kBK = 256;          // FP4 elements per k-tile
constexpr int kBKBytes = 128;     // bytes per row per k-tile
constexpr int kMmaK = 64;         // FP4 elements per block-scaled MMA
constexpr int kAtomBytes = 512;   // one 128-row x 4-column scale atom
constexpr int kSfChunk = 2048;    // shared bytes per 128-row scale block per stage (4 atoms)
constexpr int kThreads = 192;     // producer warp, MMA warp, 4 epilogue warps
constexpr int kEpiThreads = 128;
constexpr int kSmemLimit = 232448;

enum EpiMode : int32_t { kEpiTmaStore = 0, kEpiTransposed = 1, kEpiSplitK = 2 };

struct Args {
    const uint8_t *sfa;      // atom-layout scales of slot A
    const uint8_t *sfb;      // atom-layout scales of slot B
    void *out;               // D (modes 0, 1) or split-K workspace (mode 2)
    int64_t ldo;             // row stride in elements of `out` for modes 1 and 2
    int64_t split_stride;    // elements between split partials (mode 2)
    uint64_t wait_ns;        // bound on every mbarrier wait
    int32_t rows_a, rows_b, K;
    int32_t kc4;             // scale atoms per 128-row block along K
    int32_t k_tiles;         // ceil(K / 256)
    int32_t kps;             // k-tiles per split
    int32_t tiles_a, tiles_b, splits, units, group_b;
    int32_t mx;              // 0 NVFP4 (vec 16, UE4M3), 1 MXFP4 (vec 32, UE8M0)
    int32_t bf16;            // output type for modes 0 and 1
    int32_t mode;            // EpiMode
    float alpha;
};

template <int BN>
struct Cfg {
    static constexpr int NRB = (BN + 127) / 128;              // 128-row scale blocks on the N side
    static constexpr int A_BYTES = kBM * kBKBytes;             // 16 KB
    static constexpr int B_BYTES = BN * kBKBytes;
    static constexpr int SFA_BYTES = kSfChunk;
    static constexpr int SFB_BYTES = NRB * kSfChunk;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr bool TMA_EPI = BN >= 128;                 // direct mode needs the store staging
    static constexpr int STAGING_BYTES = TMA_EPI ? 2 * kBM * 128 : 0;
    static constexpr int BAR_BYTES = 256;
    static constexpr int BUDGET = kSmemLimit - 1024 - BAR_BYTES;
    static constexpr int STAGES_FIT = (BUDGET - STAGING_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int ACC_BUFS = BN <= 128 ? 2 : 1;
    // TMEM per stage: SFA 4 atoms x 4 columns, SFB 4 atoms x 4 columns per row block.
    static constexpr int SF_COLS = 16 + NRB * 16;
    static constexpr int TMEM_USED = ACC_BUFS * BN + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256 : 512;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr int OFF_STG = OFF_SFB + STAGES * SFB_BYTES;
    static constexpr int OFF_BAR = OFF_STG + STAGING_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;   // + alignment slack
    static_assert(STAGES >= 2, "too few pipeline stages");
    static_assert(TMEM_USED <= 512, "TMEM budget exceeded");
    static_assert(SMEM_BYTES <= kSmemLimit, "shared memory budget exceeded");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N must be a multiple of 16 in [16, 256]");
};

// Records the first error of this device (later ones are dropped).
__device__ __forceinline__ void record_error(int code)
{
    atomicCAS(&g_status, 0, code);
}

// mbarrier wait with a time bound. On expiry it records FP4_ERR_TIMEOUT in the
// device status word, raises this CTA's abort flag and returns false; it also
// gives up early once another role of the CTA raised the flag.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          volatile uint32_t *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*abort_flag != 0) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                record_error(FP4_ERR_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Unit u -> (slot-A tile, slot-B tile, split). Splits are outermost; inside a
// split, tiles go in groups of `group_b` slot-B tiles with slot-A tiles
// running across each group, so the CTAs in flight share operand rows in L2.
__device__ __forceinline__ void unit_coords(const Args &a, int u, int &ta, int &tb, int &split)
{
    const int tiles = a.tiles_a * a.tiles_b;
    split = u / tiles;
    const int t = u - split * tiles;
    const int per_group = a.group_b * a.tiles_a;
    const int g = t / per_group;
    const int r = t - g * per_group;
    const int b0 = g * a.group_b;
    const int gw = min(a.group_b, a.tiles_b - b0);
    tb = b0 + r % gw;
    ta = r / gw;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    fp4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const Args args)
{
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const base_ptr = smem_raw + (base - raw);

    const uint32_t bar_full = base + C::OFF_BAR;
    const uint32_t bar_empty = bar_full + 8 * C::STAGES;
    const uint32_t bar_acc_full = bar_empty + 8 * C::STAGES;
    const uint32_t bar_acc_empty = bar_acc_full + 16;
    const uint32_t bar_drain = bar_acc_empty + 16;
    uint32_t *const tmem_holder = reinterpret_cast<uint32_t *>(base_ptr + C::OFF_BAR + 16 * C::STAGES + 40);
    volatile uint32_t *const abort_flag =
        reinterpret_cast<volatile uint32_t *>(base_ptr + C::OFF_BAR + 16 * C::STAGES + 44);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full + 8 * b, 1);
            mbar_init(bar_acc_empty + 8 * b, kEpiThreads);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        if (args.mode == kEpiTmaStore) prefetch_tensormap(&tmap_d);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    const int apk = args.mx ? 2 : 4;   // scale atoms per k-tile (per 128-row block)

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0;                   // bit s: stage s has a fill in flight
            uint32_t fill_parity = 0;              // bit s: parity of that fill
            bool ok = true;
            const int rbb_count = (args.rows_b + 127) / 128;
            for (int u = blockIdx.x; ok && u < args.units; u += gridDim.x) {
                int ta, tb, split;
                unit_coords(args, u, ta, tb, split);
                const int kt0 = split * args.kps;
                const int kt1 = min(kt0 + args.kps, args.k_tiles);
                const int row_a0 = ta * kBM, row_b0 = tb * BN;
                const int rbb0 = row_b0 / 128;
                const int nrb = min(C::NRB, rbb_count - rbb0);
                for (int kt = kt0; kt < kt1; ++kt) {
                    if (!wait_bounded(bar_empty + 8 * stage, phase ^ 1u, args.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int atoms = min(apk, args.kc4 - kt * apk);
                    const uint32_t sf_bytes = static_cast<uint32_t>(atoms) * kAtomBytes;
                    const uint32_t full = bar_full + 8 * stage;
                    mbar_arrive_expect_tx(full, C::A_BYTES + C::B_BYTES + sf_bytes * (1 + nrb));
                    tma_load_2d(base + C::OFF_A + stage * C::A_BYTES, &tmap_a, full, kt * kBKBytes, row_a0);
                    tma_load_2d(base + C::OFF_B + stage * C::B_BYTES, &tmap_b, full, kt * kBKBytes, row_b0);
                    bulk_load(base + C::OFF_SFA + stage * C::SFA_BYTES,
                              args.sfa + (static_cast<int64_t>(ta) * args.kc4 + kt * apk) * kAtomBytes,
                              sf_bytes, full);
                    for (int rb = 0; rb < nrb; ++rb)
                        bulk_load(base + C::OFF_SFB + stage * C::SFB_BYTES + rb * kSfChunk,
                                  args.sfb + (static_cast<int64_t>(rbb0 + rb) * args.kc4 + kt * apk) * kAtomBytes,
                                  sf_bytes, full);
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Let every copy this thread started land before the CTA can exit.
            for (int s = 0; s < C::STAGES; ++s)
                if (filled & (1u << s)) wait_bounded(bar_full + 8 * s, (fill_parity >> s) & 1u, args.wait_ns, abort_flag);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const bool mx = args.mx != 0;
            for (int u = blockIdx.x; ok && u < args.units; u += gridDim.x) {
                int ta, tb, split;
                unit_coords(args, u, ta, tb, split);
                const int kt0 = split * args.kps;
                const int kt1 = min(kt0 + args.kps, args.k_tiles);
                if (!wait_bounded(bar_acc_empty + 8 * acc, acc_phase ^ 1u, args.wait_ns, abort_flag)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
                for (int kt = kt0; kt < kt1; ++kt) {
                    if (!wait_bounded(bar_full + 8 * stage, phase, args.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // Scale atoms of this k-tile -> this stage's TMEM scale columns.
                    const uint32_t sf_col = tmem + static_cast<uint32_t>(C::ACC_BUFS * BN + stage * C::SF_COLS);
                    const uint32_t sfa_smem = base + C::OFF_SFA + stage * C::SFA_BYTES;
                    const uint32_t sfb_smem = base + C::OFF_SFB + stage * C::SFB_BYTES;
                    const int atoms = min(apk, args.kc4 - kt * apk);
                    for (int t = 0; t < atoms; ++t) {
                        tc_cp_32x128b_warpx4(sf_col + 4 * t, smem_desc(sfa_smem + t * kAtomBytes, 0, 128, 0));
                        for (int rb = 0; rb < C::NRB; ++rb)
                            tc_cp_32x128b_warpx4(sf_col + 16 + t * 4 * C::NRB + 4 * rb,
                                                 smem_desc(sfb_smem + rb * kSfChunk + t * kAtomBytes, 0, 128, 0));
                    }
                    const int nmma = min(kBK / kMmaK, (args.K - kt * kBK + kMmaK - 1) / kMmaK);
                    const uint32_t a_smem = base + C::OFF_A + stage * C::A_BYTES;
                    const uint32_t b_smem = base + C::OFF_B + stage * C::B_BYTES;
                    for (int j = 0; j < nmma; ++j) {
                        // K-major, 128-byte swizzle: rows 128 bytes apart, 8-row groups 1024 apart;
                        // MMA j reads bytes [32 j, 32 j + 32) of every row.
                        const uint64_t ad = smem_desc(a_smem + 32 * j, 16, 1024, 2);
                        const uint64_t bd = smem_desc(b_smem + 32 * j, 16, 1024, 2);
                        const int t = mx ? (j >> 1) : j;
                        const uint32_t sf_id = mx ? static_cast<uint32_t>((j & 1) * 2) : 0u;
                        const uint32_t idesc = idesc_fp4(kBM, BN, mx, sf_id, sf_id);
                        const uint32_t sfa_t = sf_col + 4 * t;
                        const uint32_t sfb_t = sf_col + 16 + t * 4 * C::NRB;
                        const uint32_t accumulate = (kt > kt0 || j > 0) ? 1u : 0u;
                        if (mx)
                            tc_mma_fp4_vec32(d_tmem, ad, bd, idesc, sfa_t, sfb_t, accumulate);
                        else
                            tc_mma_fp4_vec16(d_tmem, ad, bd, idesc, sfa_t, sfb_t, accumulate);
                    }
                    tc_commit(bar_empty + 8 * stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(bar_acc_full + 8 * acc);
                if (C::ACC_BUFS == 2) {
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                } else {
                    acc_phase ^= 1u;
                }
            }
            // Every MMA and scale copy this thread issued completes before teardown.
            tc_commit(bar_drain);
            wait_bounded(bar_drain, 0, args.wait_ns, abort_flag);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const int row_in_tile = 32 * q + lane;
        const bool leader = threadIdx.x == 64;
        int acc = 0;
        uint32_t acc_phase = 0;
        int sb = 0;
        for (int u = blockIdx.x; u < args.units; u += gridDim.x) {
            int ta, tb, split;
            unit_coords(args, u, ta, tb, split);
            // The four epilogue warps take the same exit decision (they meet at
            // named barriers below), so the wait's outcome is AND-reduced first.
            const bool got = wait_bounded(bar_acc_full + 8 * acc, acc_phase, args.wait_ns, abort_flag);
            if (!named_bar_and(1, kEpiThreads, got)) break;
            tc_fence_after();
            const uint32_t t_base = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(acc * BN);
            const int row_a0 = ta * kBM, row_b0 = tb * BN;
            if (C::TMA_EPI && args.mode == kEpiTmaStore) {
                // 128 rows x 128 bytes per subtile: 32 fp32 or 64 bf16 columns.
                const int cw = args.bf16 ? 64 : 32;
                const int nsub = BN / cw;
                const int r = row_in_tile;
                for (int c = 0; c < nsub; ++c) {
                    uint32_t packed[32];
                    if (args.bf16) {
                        uint32_t v0[32], v1[32];
                        tmem_ld_32x32b_x32(t_base + c * 64, v0);
                        tmem_ld_32x32b_x32(t_base + c * 64 + 32, v1);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v0[2 * i]) * args.alpha,
                                                                     __uint_as_float(v0[2 * i + 1]) * args.alpha);
                            packed[i] = *reinterpret_cast<uint32_t *>(&h);
                            __nv_bfloat162 g = __floats2bfloat162_rn(__uint_as_float(v1[2 * i]) * args.alpha,
                                                                     __uint_as_float(v1[2 * i + 1]) * args.alpha);
                            packed[16 + i] = *reinterpret_cast<uint32_t *>(&g);
                        }
                    } else {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(t_base + c * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) packed[i] = __float_as_uint(__uint_as_float(v[i]) * args.alpha);
                    }
                    if (c == nsub - 1) {
                        // the accumulator is fully read: hand it back to the MMA warp
                        tc_fence_before();
                        mbar_arrive(bar_acc_empty + 8 * acc);
                    }
                    if (leader) bulk_wait_group_read<1>();
                    named_bar_sync(1, kEpiThreads);
                    uint8_t *stg = base_ptr + C::OFF_STG + sb * (kBM * 128);
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint4 w = make_uint4(packed[4 * ch], packed[4 * ch + 1], packed[4 * ch + 2], packed[4 * ch + 3]);
                        *reinterpret_cast<uint4 *>(stg + r * 128 + ((ch ^ (r & 7)) << 4)) = w;
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1, kEpiThreads);
                    if (leader) {
                        tma_store_2d(&tmap_d, base + C::OFF_STG + sb * (kBM * 128), row_b0 + c * cw, row_a0);
                        bulk_commit_group();
                    }
                    sb ^= 1;
                }
            } else {
                // Transposed direct stores (swap-AB) or fp32 split-K partials: for a
                // fixed TMEM column the 32 lanes of a warp write 32 consecutive elements.
                const int ra = row_a0 + row_in_tile;
                const bool row_ok = ra < args.rows_a;
                constexpr int CH = BN < 32 ? BN : 32;
                for (int c = 0; c < BN / CH; ++c) {
                    uint32_t v[32];
                    if constexpr (CH == 32) {
                        tmem_ld_32x32b_x32(t_base + c * 32, v);
                    } else {
                        uint32_t w[16];
                        tmem_ld_32x32b_x16(t_base, w);
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = w[i];
                    }
                    tmem_ld_wait();
                    if (c == BN / CH - 1) {
                        tc_fence_before();
                        mbar_arrive(bar_acc_empty + 8 * acc);
                    }
                    if (!row_ok) continue;
                    if (args.mode == kEpiSplitK) {
                        float *ws = static_cast<float *>(args.out) + split * args.split_stride;
#pragma unroll
                        for (int i = 0; i < CH; ++i) {
                            const int rb = row_b0 + c * CH + i;
                            if (rb < args.rows_b) ws[static_cast<int64_t>(rb) * args.ldo + ra] = __uint_as_float(v[i]);
                        }
                    } else if (args.bf16) {
                        __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(args.out);
#pragma unroll
                        for (int i = 0; i < CH; ++i) {
                            const int rb = row_b0 + c * CH + i;
                            if (rb < args.rows_b)
                                d[static_cast<int64_t>(rb) * args.ldo + ra] = __float2bfloat16_rn(__uint_as_float(v[i]) * args.alpha);
                        }
                    } else {
                        float *d = static_cast<float *>(args.out);
#pragma unroll
                        for (int i = 0; i < CH; ++i) {
                            const int rb = row_b0 + c * CH + i;
                            if (rb < args.rows_b) d[static_cast<int64_t>(rb) * args.ldo + ra] = __uint_as_float(v[i]) * args.alpha;
                        }
                    }
                }
            }
            if (C::ACC_BUFS == 2) {
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            } else {
                acc_phase ^= 1u;
            }
        }
        if (leader) bulk_wait_group<0>();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// Split-K: D[rb][ra] = alpha * sum_s ws[s][rb][ra] (fixed order, deterministic).
__global__ void splitk_reduce_kernel(const float *__restrict__ ws, void *__restrict__ out, int64_t rows_b,
                                     int64_t rows_a, int64_t ldd, int splits, int64_t split_stride, float alpha,
                                     int bf16)
{
    const int64_t total = rows_b * rows_a;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t rb = i / rows_a, ra = i - rb * rows_a;
        float s = 0.f;
        for (int k = 0; k < splits; ++k) s += ws[k * split_stride + rb * rows_a + ra];
        s *= alpha;
        if (bf16)
            static_cast<__nv_bfloat16 *>(out)[rb * ldd + ra] = __float2bfloat16_rn(s);
        else
            static_cast<float *>(out)[rb * ldd + ra] = s;
    }
}

// Scale reorder: row-major sf[rows][ksf] -> 128x4 atoms. One thread writes one
// 4-byte word of the output: word w of atom (rb, cb) holds row
// rb*128 + 32*(w%4) + (w/4)%32, columns 4cb..4cb+3 (zero past the matrix).
__global__ void scale_reorder_kernel(const uint8_t *__restrict__ sf, uint32_t *__restrict__ out, int64_t rows,
                                     int64_t ksf, int64_t kc4, int64_t words)
{
    for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < words;
         w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t atom = w >> 7;
        const int within = static_cast<int>(w & 127);
        const int i = within >> 2, j = within & 3;
        const int64_t rb = atom / kc4, cb = atom - rb * kc4;
        const int64_t r = rb * 128 + 32 * j + i;
        const int64_t c0 = cb * 4;
        uint32_t word = 0;
        if (r < rows) {
            const uint8_t *row = sf + r * ksf;
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (c0 + t < ksf) word |= static_cast<uint32_t>(row[c0 + t]) << (8 * t);
        }
        out[w] = word;
    }
}

// ============================================================================ host

namespace {

std::mutex g_mu;
int64_t g_wait_ms = -1;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct DeviceInfo {
    bool probed = false;
    bool ok = false;
    int sms = 0;
    bool attr_set[9] = {};
};
DeviceInfo g_dev[64];

uint64_t wait_limit_ns()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_wait_ms < 0) {
        g_wait_ms = 2000;
        if (const char *e = std::getenv("FP4_GEMM_WAIT_LIMIT_MS")) {
            long long v = std::atoll(e);
            if (v > 0) g_wait_ms = v;
        }
    }
    return static_cast<uint64_t>(g_wait_ms) * 1000000ull;
}

fp4_status device_info(int &dev, DeviceInfo *&info)
{
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP4_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.probed) {
        d.probed = true;
        cudaDeviceProp p;
        if (cudaGetDeviceProperties(&p, dev) == cudaSuccess && p.major == 10 && p.minor == 3) {
            d.ok = true;
            d.sms = p.multiProcessorCount;
        }
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                    cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    info = &d;
    if (!d.ok || !g_encode) return FP4_ERR_NO_DEVICE;
    return FP4_OK;
}

bool encode_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int bn_index(int bn)
{
    switch (bn) {
    case 16: return 0;
    case 32: return 1;
    case 64: return 2;
    case 128: return 3;
    case 256: return 4;
    default: return -1;
    }
}

template <int BN>
cudaError_t launch_gemm(DeviceInfo &info, int grid, const CUtensorMap &ta, const CUtensorMap &tb,
                        const CUtensorMap &td, const Args &args, cudaStream_t stream)
{
    using C = Cfg<BN>;
    const int idx = bn_index(BN);
    if (!info.attr_set[idx]) {
        cudaError_t e = cudaFuncSetAttribute(fp4_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        info.attr_set[idx] = true;
    }
    fp4_gemm_kernel<BN><<<grid, kThreads, C::SMEM_BYTES, stream>>>(ta, tb, td, args);
    return cudaGetLastError();
}

cudaError_t launch_by_bn(int bn, DeviceInfo &info, int grid, const CUtensorMap &ta, const CUtensorMap &tb,
                         const CUtensorMap &td, const Args &args, cudaStream_t stream)
{
    switch (bn) {
    case 16: return launch_gemm<16>(info, grid, ta, tb, td, args, stream);
    case 32: return launch_gemm<32>(info, grid, ta, tb, td, args, stream);
    case 64: return launch_gemm<64>(info, grid, ta, tb, td, args, stream);
    case 128: return launch_gemm<128>(info, grid, ta, tb, td, args, stream);
    default: return launch_gemm<256>(info, grid, ta, tb, td, args, stream);
    }
}

struct Plan {
    bool swap;
    int bn;
    int splits;
    int grid;
};

int pow2_bn(int64_t rows)
{
    if (rows <= 16) return 16;
    if (rows <= 32) return 32;
    if (rows <= 64) return 64;
    if (rows <= 128) return 128;
    return 256;
}

// Chooses direct vs swap-AB, the tile N and the K split. `tma_ok` says whether
// D can take TMA stores (row pitch and base 16-byte aligned).
fp4_status make_plan(int64_t M, int64_t N, int64_t K, bool tma_ok, int sms, const fp4_gemm_config *cfg, Plan &p)
{
    const int mode = cfg ? cfg->mode : 0;
    if (mode < 0 || mode > 2) return FP4_ERR_INVALID_ARG;
    if (mode == 1)
        p.swap = false;
    else if (mode == 2)
        p.swap = true;
    else
        p.swap = (M <= 256) || !tma_ok;
    if (!p.swap && !tma_ok) return FP4_ERR_MISALIGNED;
    const int64_t rows_b = p.swap ? M : N;
    const int64_t rows_a = p.swap ? N : M;
    int bn = (cfg && cfg->bn) ? cfg->bn : (p.swap ? pow2_bn(rows_b) : 256);
    if (bn_index(bn) < 0) return FP4_ERR_INVALID_ARG;
    if (!p.swap && bn < 128) return FP4_ERR_UNSUPPORTED;           // direct mode stages through TMA store tiles
    if (rows_b > bn && bn < 128) return FP4_ERR_UNSUPPORTED;       // N-side tiles must start on scale blocks
    p.bn = bn;
    const int64_t tiles = cdiv(rows_a, kBM) * cdiv(rows_b, bn);
    const int64_t k_tiles = cdiv(K, kBK);
    int splits = (cfg && cfg->splits) ? cfg->splits : 0;
    if (splits < 0) return FP4_ERR_INVALID_ARG;
    if (splits > 1 && !p.swap) return FP4_ERR_UNSUPPORTED;
    if (splits == 0) {
        splits = 1;
        if (p.swap && tiles < sms) {
            // minimise (waves x k-tiles per split), preferring fewer splits on ties
            double best = 1e30;
            for (int s = 1; s <= std::min<int64_t>(k_tiles, 16); ++s) {
                const double waves = static_cast<double>(cdiv(tiles * s, sms));
                const double cost = waves * static_cast<double>(cdiv(k_tiles, s)) * (1.0 + 0.02 * (s - 1));
                if (cost < best - 1e-9) {
                    best = cost;
                    splits = s;
                }
            }
        }
    }
    splits = static_cast<int>(std::min<int64_t>(splits, k_tiles));
    p.splits = std::max(1, splits);
    const int64_t units = tiles * p.splits;
    int cap = (cfg && cfg->max_ctas > 0) ? cfg->max_ctas : sms;
    p.grid = static_cast<int>(std::min<int64_t>(units, cap));
    return FP4_OK;
}

fp4_status reorder_launch(const void *sf_plain, void *sf_atom, int64_t rows, int64_t ksf, cudaStream_t stream)
{
    const int64_t kc4 = cdiv(ksf, 4);
    const int64_t words = cdiv(rows, 128) * kc4 * 128;
    if (words == 0) return FP4_OK;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>(cdiv(words, threads), 148 * 16);
    scale_reorder_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint8_t *>(sf_plain), static_cast<uint32_t *>(sf_atom), rows, ksf, kc4, words);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

fp4_status gemm_impl(fp4_format fmt, int prepacked, const void *A, const void *sfA, const void *B,
                     const void *sfB, float alpha, void *D, int64_t M, int64_t N, int64_t K, fp4_out_dtype out,
                     const fp4_gemm_config *cfg, cudaStream_t stream)
{
    if (fmt != FP4_FMT_NVFP4 && fmt != FP4_FMT_MXFP4) return FP4_ERR_INVALID_ARG;
    if (out != FP4_OUT_F32 && out != FP4_OUT_BF16) return FP4_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return FP4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP4_OK;
    if (!D) return FP4_ERR_INVALID_ARG;
    const int64_t esize = out == FP4_OUT_BF16 ? 2 : 4;
    if (K == 0) {
        if (!aligned16(D)) return FP4_ERR_MISALIGNED;
        return cudaMemsetAsync(D, 0, static_cast<size_t>(M * N * esize), stream) == cudaSuccess ? FP4_OK
                                                                                              : FP4_ERR_CUDA;
    }
    if (!A || !B || !sfA || !sfB) return FP4_ERR_INVALID_ARG;
    if (K % 32 != 0) return FP4_ERR_UNSUPPORTED;
    if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30) || M * N > (1ll << 46))
        return FP4_ERR_UNSUPPORTED;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D)) return FP4_ERR_MISALIGNED;
    if (prepacked && (!aligned16(sfA) || !aligned16(sfB))) return FP4_ERR_MISALIGNED;

    int dev;
    DeviceInfo *info;
    fp4_status st = device_info(dev, info);
    if (st != FP4_OK) return st;

    const int vec = fmt == FP4_FMT_NVFP4 ? 16 : 32;
    const int64_t ksf = K / vec;
    const int64_t kc4 = cdiv(ksf, 4);
    const bool tma_ok = (N * esize) % 16 == 0;
    Plan plan;
    st = make_plan(M, N, K, tma_ok, info->sms, cfg, plan);
    if (st != FP4_OK) return st;

    const int64_t rows_a = plan.swap ? N : M, rows_b = plan.swap ? M : N;
    const void *op_a = plan.swap ? B : A, *op_b = plan.swap ? A : B;
    const void *sf_a = plan.swap ? sfB : sfA, *sf_b = plan.swap ? sfA : sfB;

    // scratch: reordered scales and split-K partials (stream-ordered)
    const size_t atoms_a = static_cast<size_t>(cdiv(rows_a, 128) * kc4 * kAtomBytes);
    const size_t atoms_b = static_cast<size_t>(cdiv(rows_b, 128) * kc4 * kAtomBytes);
    const size_t ws_bytes = plan.splits > 1 ? static_cast<size_t>(plan.splits) * rows_a * rows_b * 4 : 0;
    const size_t scratch_bytes = (prepacked ? 0 : atoms_a + atoms_b) + ws_bytes;
    uint8_t *scratch = nullptr;
    if (scratch_bytes) {
        if (cudaMallocAsync(reinterpret_cast<void **>(&scratch), scratch_bytes, stream) != cudaSuccess)
            return FP4_ERR_CUDA;
    }
    fp4_status result = FP4_OK;
    do {
        const uint8_t *sfa_atoms = static_cast<const uint8_t *>(sf_a);
        const uint8_t *sfb_atoms = static_cast<const uint8_t *>(sf_b);
        uint8_t *ws = scratch + (prepacked ? 0 : atoms_a + atoms_b);
        if (!prepacked) {
            if ((result = reorder_launch(sf_a, scratch, rows_a, ksf, stream)) != FP4_OK) break;
            if ((result = reorder_launch(sf_b, scratch + atoms_a, rows_b, ksf, stream)) != FP4_OK) break;
            sfa_atoms = scratch;
            sfb_atoms = scratch + atoms_a;
        }
        CUtensorMap tmap_a, tmap_b, tmap_d;
        std::memset(&tmap_d, 0, sizeof tmap_d);
        if (!encode_2d(&tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, op_a, static_cast<uint64_t>(K / 2),
                       static_cast<uint64_t>(rows_a), static_cast<uint64_t>(K / 2), kBKBytes, kBM) ||
            !encode_2d(&tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, op_b, static_cast<uint64_t>(K / 2),
                       static_cast<uint64_t>(rows_b), static_cast<uint64_t>(K / 2), kBKBytes,
                       static_cast<uint32_t>(plan.bn))) {
            result = FP4_ERR_CUDA;
            break;
        }
        Args a;
        std::memset(&a, 0, sizeof a);
        a.sfa = sfa_atoms;
        a.sfb = sfb_atoms;
        a.wait_ns = wait_limit_ns();
        a.rows_a = static_cast<int32_t>(rows_a);
        a.rows_b = static_cast<int32_t>(rows_b);
        a.K = static_cast<int32_t>(K);
        a.kc4 = static_cast<int32_t>(kc4);
        a.k_tiles = static_cast<int32_t>(cdiv(K, kBK));
        a.splits = plan.splits;
        a.kps = static_cast<int32_t>(cdiv(a.k_tiles, plan.splits));
        a.splits = static_cast<int32_t>(cdiv(a.k_tiles, a.kps));   // no empty split
        a.tiles_a = static_cast<int32_t>(cdiv(rows_a, kBM));
        a.tiles_b = static_cast<int32_t>(cdiv(rows_b, plan.bn));
        a.units = a.tiles_a * a.tiles_b * a.splits;
        a.group_b = std::max(1, std::min(a.tiles_b, 8));
        a.mx = fmt == FP4_FMT_MXFP4;
        a.bf16 = out == FP4_OUT_BF16;
        a.alpha = alpha;
        if (!plan.swap) {
            a.mode = kEpiTmaStore;
            a.out = D;
            const CUtensorMapDataType dt = a.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
            if (!encode_2d(&tmap_d, dt, D, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                           static_cast<uint64_t>(N * esize), static_cast<uint32_t>(128 / esize), kBM)) {
                result = FP4_ERR_CUDA;
                break;
            }
        } else if (a.splits > 1) {
            a.mode = kEpiSplitK;
            a.out = ws;
            a.ldo = rows_a;
            a.split_stride = rows_a * rows_b;
        } else {
            a.mode = kEpiTransposed;
            a.out = D;
            a.ldo = N;
        }
        const int grid = std::min(plan.grid, a.units);
        if (launch_by_bn(plan.bn, *info, grid, tmap_a, tmap_b, tmap_d, a, stream) != cudaSuccess) {
            result = FP4_ERR_CUDA;
            break;
        }
        if (a.mode == kEpiSplitK) {
            const int64_t total = rows_a * rows_b;
            const int64_t blocks = std::min<int64_t>(cdiv(total, 256), static_cast<int64_t>(info->sms) * 8);
            splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
                reinterpret_cast<const float *>(ws), D, rows_b, rows_a, N, a.splits, a.split_stride, alpha, a.bf16);
            if (cudaGetLastError() != cudaSuccess) {
                result = FP4_ERR_CUDA;
                break;
            }
        }
    } while (false);
    if (scratch && cudaFreeAsync(scratch, stream) != cudaSuccess && result == FP4_OK) result = FP4_ERR_CUDA;
    return result;
}

}  // namespace
}  // namespace fp4

// ============================================================================ C ABI

using namespace fp4;

extern "C" {

fp4_status fp4_gemm(fp4_format fmt, int scales_prepacked, const void *A, const void *sfA, const void *B,
                    const void *sfB, float alpha, void *D, int64_t M, int64_t N, int64_t K, fp4_out_dtype out,
                    const fp4_gemm_config *cfg, cudaStream_t stream)
{
    return gemm_impl(fmt, scales_prepacked, A, sfA, B, sfB, alpha, D, M, N, K, out, cfg, stream);
}

fp4_status fp4_gemm_nvfp4(const void *A, const void *sfA, const void *B, const void *sfB, float alpha, void *D,
                          int64_t M, int64_t N, int64_t K, fp4_out_dtype out, cudaStream_t stream)
{
    return gemm_impl(FP4_FMT_NVFP4, 0, A, sfA, B, sfB, alpha, D, M, N, K, out, nullptr, stream);
}

fp4_status fp4_gemm_mxfp4(const void *A, const void *sfA, const void *B, const void *sfB, float alpha, void *D,
                          int64_t M, int64_t N, int64_t K, fp4_out_dtype out, cudaStream_t stream)
{
    return gemm_impl(FP4_FMT_MXFP4, 0, A, sfA, B, sfB, alpha, D, M, N, K, out, nullptr, stream);
}

fp4_status fp4_gemm_nvfp4_prepacked(const void *A, const void *sfA, const void *B, const void *sfB, float alpha,
                                    void *D, int64_t M, int64_t N, int64_t K, fp4_out_dtype out, cudaStream_t stream)
{
    return gemm_impl(FP4_FMT_NVFP4, 1, A, sfA, B, sfB, alpha, D, M, N, K, out, nullptr, stream);
}

fp4_status fp4_gemm_mxfp4_prepacked(const void *A, const void *sfA, const void *B, const void *sfB, float alpha,
                                    void *D, int64_t M, int64_t N, int64_t K, fp4_out_dtype out, cudaStream_t stream)
{
    return gemm_impl(FP4_FMT_MXFP4, 1, A, sfA, B, sfB, alpha, D, M, N, K, out, nullptr, stream);
}

fp4_status fp4_gemm_host(fp4_format fmt, const void *A, const void *sfA, const void *B, const void *sfB,
                         float alpha, void *D, int64_t M, int64_t N, int64_t K, fp4_out_dtype out,
                         cudaStream_t stream)
{
    if (fmt != FP4_FMT_NVFP4 && fmt != FP4_FMT_MXFP4) return FP4_ERR_INVALID_ARG;
    if (out != FP4_OUT_F32 && out != FP4_OUT_BF16) return FP4_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return FP4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP4_OK;
    if (!D || (K > 0 && (!A || !B || !sfA || !sfB))) return FP4_ERR_INVALID_ARG;
    if (K % 32 != 0) return FP4_ERR_UNSUPPORTED;
    const int vec = fmt == FP4_FMT_NVFP4 ? 16 : 32;
    const size_t esize = out == FP4_OUT_BF16 ? 2 : 4;
    auto up256 = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    const size_t bA = static_cast<size_t>(M) * (K / 2), bB = static_cast<size_t>(N) * (K / 2);
    const size_t bsA = static_cast<size_t>(M) * (K / vec), bsB = static_cast<size_t>(N) * (K / vec);
    const size_t bD = static_cast<size_t>(M) * N * esize;
    const size_t total = up256(bA) + up256(bB) + up256(bsA) + up256(bsB) + up256(bD);
    uint8_t *buf = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&buf), total, stream) != cudaSuccess) return FP4_ERR_CUDA;
    uint8_t *dA = buf, *dB = dA + up256(bA), *dsA = dB + up256(bB), *dsB = dsA + up256(bsA), *dD = dsB + up256(bsB);
    fp4_status st = FP4_OK;
    if ((bA && cudaMemcpyAsync(dA, A, bA, cudaMemcpyHostToDevice, stream) != cudaSuccess) ||
        (bB && cudaMemcpyAsync(dB, B, bB, cudaMemcpyHostToDevice, stream) != cudaSuccess) ||
        (bsA && cudaMemcpyAsync(dsA, sfA, bsA, cudaMemcpyHostToDevice, stream) != cudaSuccess) ||
        (bsB && cudaMemcpyAsync(dsB, sfB, bsB, cudaMemcpyHostToDevice, stream) != cudaSuccess))
        st = FP4_ERR_CUDA;
    if (st == FP4_OK) st = gemm_impl(fmt, 0, dA, dsA, dB, dsB, alpha, dD, M, N, K, out, nullptr, stream);
    if (st == FP4_OK && cudaMemcpyAsync(D, dD, bD, cudaMemcpyDeviceToHost, stream) != cudaSuccess) st = FP4_ERR_CUDA;
    if (cudaFreeAsync(buf, stream) != cudaSuccess && st == FP4_OK) st = FP4_ERR_CUDA;
    return st;
}

size_t fp4_scale_atom_bytes(int64_t rows, int64_t k, int vec)
{
    if (rows < 0 || k < 0 || (vec != 16 && vec != 32) || k % vec != 0) return 0;
    return static_cast<size_t>(cdiv(rows, 128) * cdiv(k / vec, 4) * kAtomBytes);
}

fp4_status fp4_scale_reorder(const void *sf_plain, void *sf_atom, int64_t rows, int64_t k, int vec,
                             cudaStream_t stream)
{
    if (rows < 0 || k < 0 || (vec != 16 && vec != 32)) return FP4_ERR_INVALID_ARG;
    if (k % vec != 0) return FP4_ERR_UNSUPPORTED;
    if (rows == 0 || k == 0) return FP4_OK;
    if (!sf_plain || !sf_atom) return FP4_ERR_INVALID_ARG;
    if (!aligned16(sf_atom)) return FP4_ERR_MISALIGNED;
    int dev;
    DeviceInfo *info;
    fp4_status st = device_info(dev, info);
    if (st != FP4_OK) return st;
    return reorder_launch(sf_plain, sf_atom, rows, k / vec, stream);
}

fp4_status fp4_get_device_status(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FP4_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) return FP4_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status, &zero, sizeof zero) != cudaSuccess) return FP4_ERR_CUDA;
    }
    return static_cast<fp4_status>(v);
}

const char *fp4_status_string(fp4_status s)
{
    switch (s) {
    case FP4_OK: return "ok";
    case FP4_ERR_INVALID_ARG: return "invalid argument";
    case FP4_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case FP4_ERR_MISALIGNED: return "pointer or row pitch not 16-byte aligned";
    case FP4_ERR_CUDA: return "CUDA call failed";
    case FP4_ERR_TIMEOUT: return "bounded device wait ran out";
    case FP4_ERR_NO_DEVICE: return "no sm_103 device";
    default: return "unknown status";
    }
}

void fp4_set_wait_limit_ms(int64_t ms)
{
    std::lock_guard<std::mutex> lk(g_mu);
    g_wait_ms = ms < 1 ? 1 : ms;
}

}  // extern "C"
