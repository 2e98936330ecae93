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
// section 1). The kernel is a persistent, warp-specialised tcgen05 GEMM of 640
// threads (20 warps) per CTA, with a warpgroup register split (setmaxnreg: the
// epilogue's two warpgroups at 168 registers, the others at 48):
//
//   warp 0       TMA producer (one thread): fills a ring of shared-memory
//                stages; a stage is one k-tile (256 FP4 elements = 128 bytes
//                per row) of both operands (128B-swizzled) and their scale
//                atoms;
//   warp 1       MMA issuer (one thread of the leader CTA): per stage waits on
//                one `ready` barrier (batched, non-blocking look-ahead over four
//                stages), issues four K = 64 block-scaled MMAs into a TMEM
//                accumulator and frees the stage;
//   warps 4..11  epilogue: each warp drains its 32 TMEM lanes x BN/2 columns
//                into registers, hands the accumulator back at once, then
//                applies alpha, the bias and the activation (fp4_gemm_fused),
//                casts and stores -- in a CTA pair as TMA boxes through a 4 KB
//                staging buffer per warp (rows, or swap-AB's transposed tiles),
//                else with direct stores; or fp32 split-K partials -- while the
//                next tile's MMAs run;
//   warps 12..19 scale warps: two per TMEM lane quarter, each storing half of
//                every k-tile's scale atoms from shared memory into the stage's
//                TMEM scale columns (tcgen05.st), then arriving on `ready`.
//
// Every launch may start as a programmatic dependent of the scale reorder
// before it; all threads wait for that grid before touching memory. The
// grouped GEMM (fp4_gemm_grouped) instantiates the same body with its groups'
// geometry in the parameter block.
//
// CG = 2 runs a CTA pair (cluster of 2) on one 256-row MMA (tcgen05
// cta_group::2): each CTA loads 128 rows of the M side and half of the N side,
// the leader issues the MMAs, and each CTA's TMEM holds its 128 rows of D.
//
// The warp roles follow the SM100a two-CTA kernel in "TMA Pipelines, Tensor
// Cores, and ctm-rs Interop", section 2 (producer warp, single-thread MMA
// warp, epilogue warps draining TMEM, paired CTAs); the K-tile of four MMA
// instructions and the 128-byte swizzle follow "Hopper GEMM in CUTLASS C++ and
// the CuTe DSL, part 1" (tile K = four MMA instructions; the widest swizzle atom
// dividing the tile's K bytes), as does the stage count (shared capacity minus
// the epilogue carve-out, over the bytes of one stage).
//
// "Slot A" is the operand on the MMA's M side, "slot B" the one on its N side.
// Direct mode: slot A = A, slot B = B. Swap-AB mode: slot A = B, slot B = A,
// and the epilogue writes D^T tiles into row-major D -- the swapped operands of
// "Hopper GEMM in CUTLASS C++ and the CuTe DSL, part 1" ("The operands are
// swapped").

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <random>
#include <vector>

#include "epilogue.cuh"
#include "fp4_gemm.h"
#include "fp4_gemv.cuh"
#include "ptx.cuh"

namespace fp4 {

// Per-device status word: 0, or the first error a kernel recorded.
__device__ int g_status;

// Scratch of fp4_gemm_static_scratch (reordered scales, split-K partials) for
// callers that cannot allocate. In host code this name is only a stand-in: its
// device address comes from cudaGetSymbolAddress (static_scratch_address).
constexpr size_t kStaticScratchBytes = FP4_STATIC_SCRATCH_BYTES;
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kBM = 128;          // TMEM lanes / M rows per CTA
constexpr int kBK = 256;          // FP4 elements per k-tile
constexpr int kBKBytes = 128;     // bytes per row per k-tile
constexpr int kAtomBytes = 512;   // one 128-row x 4-column scale atom
// Warp roles, by warpgroup (4 warps): 0 = the TMA producer (warp 0), the MMA
// issuer (warp 1) and two idle warps; 1-2 = eight epilogue warps; 3-4 = eight
// scale warps. The epilogue warpgroups raise their registers to kEpiRegs (all
// BN/2 accumulator columns of a warp fit in registers, so the accumulator is
// handed back right after one drain) and the other three lower theirs to
// kLowRegs, within the pool of kLaunchRegs per thread the block is launched
// with (the host checks that count before the first launch).
constexpr int kEpiWarps = 8;
constexpr int kSfWarps = 8;                      // scale warps: two per TMEM lane quarter
constexpr int kFirstEpiWarp = 4;
constexpr int kFirstSfWarp = kFirstEpiWarp + kEpiWarps;
constexpr int kThreads = 32 * (kFirstSfWarp + kSfWarps);   // 640
constexpr int kLaunchRegs = 96;
constexpr int kEpiRegs = 168;
constexpr int kLowRegs = 48;
static_assert(kThreads % 128 == 0, "roles are whole warpgroups");
static_assert(3 * 128 * kLowRegs + 2 * 128 * kEpiRegs <= kLaunchRegs * kThreads, "register split fits the pool");
constexpr int kSmemLimit = 232448;

enum EpiMode : int32_t { kEpiRows = 0, kEpiTransposed = 1, kEpiSplitK = 2 };

// Grouped GEMM (fp4_gemm_grouped): where one group's tiles sit in the operands.
// Unit u of group g is tile (ta, tb) with u - first = tb * tiles_a + ta. Slot
// A's local row r is TMA row oa + r, scale block sa + r / 128 and D index
// da + r; rows r >= la are outside the group. Slot B likewise.
struct GroupGeo {
    int32_t first, tiles_a;
    int32_t oa, sa, da, la;
    int32_t ob, sb, db, lb;
    int32_t bias_off;        // first bias entry of the group
    int32_t pad;
};
static_assert(sizeof(GroupGeo) == 48, "three 16-byte loads");

// The groups travel in the grouped kernel's parameter block (constant memory,
// read with a uniform index): no table upload, so no host-side stream
// synchronisation, per call.
constexpr int kMaxGroups = 256;
struct GroupParams {
    int32_t count;
    int32_t pad[3];
    GroupGeo g[kMaxGroups];
};

// A unit's tile and where it sits (the whole problem when not grouped).
struct TileGeo {
    int ta, tb;
    int oa, sa, da, la;
    int ob, sb, db, lb;
    int bias_off;
};

struct Args {
    void *out;               // D (modes 0, 1) or split-K workspace (mode 2)
    int64_t ldo;             // row stride in elements of `out`
    int64_t split_stride;    // elements between split partials (mode 2)
    uint64_t wait_ns;        // bound on every mbarrier wait
    int32_t rows_a, rows_b;
    int32_t k_tiles;         // ceil(K / 256)
    int32_t kps;             // k-tiles per split
    int32_t tiles_a, tiles_b, splits, units, group_b;
    int32_t bf16;            // output type for modes 0 and 1
    int32_t mode;            // EpiMode
    int32_t act;             // fp4_activation (modes 0 and 1; split-K partials stay raw)
    float alpha;
    const float *bias;       // NULL, or one float per GEMM output column (modes 0 and 1)
    // Split tail (direct mode): units 0 .. split_units-1 are the two K halves of
    // the first split_units / 2 tiles (the tiles beyond the last full wave, run
    // first so that their extra epilogue work overlaps later tiles). The first
    // half leaves its fp32 partial in tail_ws and publishes `epoch` in its flag;
    // the second half adds it.
    int32_t split_units;
    int32_t kh;                          // k-tiles of a first half
    float *tail_ws;                      // [tail tile][CTA of the pair][BN][128]
    unsigned long long *tail_flags;      // [tail tile][CTA of the pair]
    unsigned long long epoch;            // this launch's flag value
    int32_t stop_after;                  // > 0: producers stop after this many stages (bounded-wait test)
    int32_t st32;                        // rows mode: D and its row pitch 32-byte aligned (256-bit stores)
    int32_t tma_d;                       // rows mode, CTA pairs: D stores go out as TMA boxes (tmap_d)
};

template <int CG, int BN, bool MX>
struct Cfg {
    static constexpr int APK = MX ? 2 : 4;             // scale atoms per k-tile per 128-row block
    static constexpr int NRB = (BN + 127) / 128;       // 128-row scale blocks on the N side (whole tile)
    static constexpr int BN_CTA = BN / CG;             // N-side rows loaded by one CTA
    // one k-tile slot of shared memory
    static constexpr int A_BYTES = kBM * kBKBytes;      // 16 KB
    static constexpr int B_BYTES = BN_CTA * kBKBytes;
    static constexpr int SFA_BYTES = APK * kAtomBytes;
    static constexpr int SFB_BYTES = NRB * APK * kAtomBytes;
    static constexpr int KTILE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int STAGE_BYTES = KTILE_BYTES;   // a stage is one k-tile
    static constexpr int BAR_BYTES = 512;
    // Pairs stage D through shared memory for TMA stores: one 32-row x 128-byte
    // box per epilogue warp (1024-aligned for the 128-byte swizzle).
    static constexpr bool TMA_D = CG == 2;
    static constexpr int STG_WARP = 32 * 128;
    static constexpr int STG_BYTES = TMA_D ? kEpiWarps * STG_WARP : 0;
    static constexpr int BUDGET = kSmemLimit - 1024 - BAR_BYTES - (TMA_D ? STG_BYTES + 1024 : 0);
    static constexpr int STAGES_FIT = BUDGET / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int SLOTS = STAGES;
    static constexpr int ACC_BUFS = BN <= 128 ? 2 : 1;
    static constexpr int SF_COLS = 4 * APK * (1 + NRB);        // TMEM columns of one k-tile's scales
    static constexpr int SFB_COLS = 4 * APK * NRB;              // of which slot B's (after slot A's 4 * APK)
    static constexpr int HA = APK / 2;                          // slot-A atoms staged by one scale warp
    static constexpr int HG = APK * NRB / 2;                    // slot-B atoms staged by one scale warp
    static constexpr int SF_TMEM = ACC_BUFS * BN;               // first scale column
    static constexpr int TMEM_USED = ACC_BUFS * BN + SLOTS * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256 : 512;
    static constexpr int OFF_A = 0;                              // slot k at OFF_X + k * X_BYTES
    static constexpr int OFF_B = OFF_A + SLOTS * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + SLOTS * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + SLOTS * SFA_BYTES;
    static constexpr int OFF_STG = (OFF_SFB + SLOTS * SFB_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_STG + STG_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;   // + alignment slack
    static constexpr int COLS_WARP = BN / 2;                        // accumulator columns per epilogue warp
    // The epilogue drains a warp's columns in one pass (its kEpiRegs registers
    // hold them all) and hands the accumulator back right after.
    static constexpr int PASSES = 1;
    static constexpr int PASS_COLS = COLS_WARP / PASSES;
    static constexpr uint32_t OPND_TX = CG * (A_BYTES + B_BYTES);   // operand bytes landing per stage (both CTAs)
    static constexpr uint32_t SF_TX = SFA_BYTES + SFB_BYTES;        // scale bytes landing per stage (this CTA)
    static_assert(CG == 1 || CG == 2, "CTA group of 1 or 2");
    static_assert(CG == 1 || BN >= 128, "paired CTAs use N tiles of 128 or 256");
    static_assert(STAGES >= 4, "at least four pipeline stages");
    static_assert(32 * STAGES + 56 <= BAR_BYTES, "barriers and flags fit");
    static_assert(TMEM_USED <= 512, "TMEM budget exceeded");
    static_assert(SMEM_BYTES <= kSmemLimit, "shared memory budget exceeded");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N must be a multiple of 16 in [16, 256]");
    static_assert(HG == 1 || HG == 2 || HG == 4, "a scale warp stores 4, 8 or 16 slot-B columns at once");
};

// Records the first error of this device (later ones are dropped).
__device__ __forceinline__ void record_error(int code)
{
    atomicCAS(&g_status, 0, code);
}

// Slow path of wait(): polls with a time bound. On expiry it records
// FP4_ERR_TIMEOUT in the device status word, raises this CTA's abort flag and
// returns false; it also gives up once another role of the CTA raised the flag.
// The teardown waits (for a CTA's own copies and MMAs in flight) pass no flag:
// they end only when the work lands or the time bound runs out.
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                       volatile uint32_t *abort_flag)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (abort_flag && *abort_flag != 0) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                record_error(FP4_ERR_TIMEOUT);
                if (abort_flag) *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                     volatile uint32_t *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, limit_ns, abort_flag);
}

// Acquire-wait (cluster scope) for barriers that the peer CTA of a pair arrives on.
__device__ __forceinline__ bool wait_cluster_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                               volatile uint32_t *abort_flag)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
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

__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                             volatile uint32_t *abort_flag)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    return wait_cluster_slow(bar, parity, limit_ns, abort_flag);
}

// Bounded wait until *flag == epoch (acquire, GPU scope): the first half of a
// split tail tile has left its partial.
__device__ __forceinline__ bool wait_flag(const unsigned long long *flag, unsigned long long epoch, uint64_t limit_ns,
                                       volatile uint32_t *abort_flag)
{
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ld_acquire_gpu_u64(flag) == epoch) return true;
        if ((it & 63u) == 0) {
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

// Where unit u's tile sits; ta / tb as unit_work gives them when not grouped.
template <bool GROUPED>
__device__ __forceinline__ void tile_geo(const Args &a, const GroupParams *gp, int u, int ta, int tb, TileGeo &t)
{
    if constexpr (GROUPED) {
        // the last group whose first unit is <= u (empty groups share a first)
        int lo = 0, hi = gp->count - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (gp->g[mid].first <= u) lo = mid; else hi = mid - 1;
        }
        const GroupGeo &q = gp->g[lo];
        const int lu = u - q.first;
        t.tb = lu / q.tiles_a;
        t.ta = lu - t.tb * q.tiles_a;
        t.oa = q.oa;
        t.sa = q.sa;
        t.da = q.da;
        t.la = q.la;
        t.ob = q.ob;
        t.sb = q.sb;
        t.db = q.db;
        t.lb = q.lb;
        t.bias_off = q.bias_off;
        return;
    }
    else {
        t.ta = ta;
        t.tb = tb;
        t.oa = t.sa = t.da = 0;
        t.la = a.rows_a;
        t.ob = t.sb = t.db = 0;
        t.lb = a.rows_b;
        t.bias_off = 0;
    }
}

// Unit u -> its tile and k-tile range. half = -1 for a whole tile (or a
// split-K unit); 0 / 1 for the first / second K half of a split tile, whose
// index among the split tiles is tidx.
template <bool GROUPED>
__device__ __forceinline__ void unit_work(const Args &a, int u, int &ta, int &tb, int &split, int &kt0, int &kt1,
                                          int &half, int &tidx)
{
    if constexpr (GROUPED) {          // whole tiles (tile_geo gives ta, tb)
        ta = tb = split = tidx = 0;
        kt0 = 0;
        kt1 = a.k_tiles;
        half = -1;
        return;
    }
    if (u >= a.split_units) {
        unit_coords(a, u - a.split_units / 2, ta, tb, split);
        kt0 = split * a.kps;
        kt1 = min(kt0 + a.kps, a.k_tiles);
        half = -1;
        tidx = 0;
        return;
    }
    tidx = u >> 1;
    half = u & 1;
    unit_coords(a, tidx, ta, tb, split);
    kt0 = half ? a.kh : 0;
    kt1 = half ? a.k_tiles : a.kh;
}

// Loads N consecutive 32-bit TMEM columns of this warp's 32 lanes.
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t *v)
{
    if constexpr (N == 8) {
        uint32_t (&r)[8] = *reinterpret_cast<uint32_t(*)[8]>(v);
        tmem_ld_32x32b_x8(taddr, r);
    } else if constexpr (N == 16) {
        uint32_t (&r)[16] = *reinterpret_cast<uint32_t(*)[16]>(v);
        tmem_ld_32x32b_x16(taddr, r);
    } else {
        static_assert(N % 32 == 0, "column count");
#pragma unroll
        for (int c = 0; c < N / 32; ++c) {
            uint32_t (&r)[32] = *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c);
            tmem_ld_32x32b_x32(taddr + 32 * c, r);
        }
    }
}

// One thread's 32-byte piece of its D row (w[0..8) = the bytes of columns col ..
// col + 2 * half_cols - 1): a single 256-bit store when the piece is whole and
// 32-byte aligned (`whole32`), else two 16-byte halves, each kept to the matrix.
// A warp's 32 lanes hold 32 rows, so one store instruction writes 32 whole
// sectors, straight from registers.
__device__ __forceinline__ void store_row32(const uint32_t (&w)[8], void *out, int64_t ldo, int esize, int row,
                                            int col, int half_cols, int rows, int cols, bool whole32,
                                            uint64_t policy)
{
    if (row >= rows || col >= cols) return;
    char *p = static_cast<char *>(out) + (static_cast<int64_t>(row) * ldo + col) * esize;
    if (whole32 && col + 2 * half_cols <= cols) {
        st_global_v8_hint(p, w, policy);
        return;
    }
    st_global_v4_hint(p, make_uint4(w[0], w[1], w[2], w[3]), policy);
    if (col + half_cols < cols)
        st_global_v4_hint(p + 16, make_uint4(w[4], w[5], w[6], w[7]), policy);
}

// Advances a (stage, phase) ring position.
template <int STAGES>
__device__ __forceinline__ void ring_next(int &stage, uint32_t &phase)
{
    if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
    }
}

// How many consecutive k-tiles, from the one at (stage, phase) on, have their
// ready barrier's phase completed (0 to 4), by one batched non-blocking test.
// Sound because the caller has consumed every earlier phase of these barriers:
// each barrier tested is at most one phase ahead of what the caller has seen,
// since the look-ahead (4) does not exceed the ring (STAGES).
template <int STAGES>
__device__ __forceinline__ int ready_run(uint32_t bar_ready, int stage, uint32_t phase)
{
    static_assert(STAGES >= 4, "the look-ahead stays within one turn of the ring");
    uint32_t b[4], p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        b[i] = bar_ready + 8 * stage;
        p[i] = phase;
        ring_next<STAGES>(stage, phase);
    }
    return __ffs(~mbar_test4_cluster(b, p)) - 1;
}

// One epilogue pass: v holds this warp's 32 TMEM lanes x PC accumulator columns,
// tile columns c0 .. c0 + PC - 1 (slot-B rows tg.tb * BN + c0 ...). Split tail:
// a first half parks its fp32 partial (column-major, so a fixed column is 32
// consecutive floats) and, after its last pass, raises its flag; the second
// half's matching warp waits for the flag once (first pass) and adds it. Then
// z = alpha * acc + bias, the activation, the cast and the stores.
template <int CG, int BN, int PC, bool TMA_D>
__device__ __forceinline__ void epilogue_pass(uint32_t (&v)[PC], const Args &args, const TileGeo &tg, int c0, int q,
                                              int lane, int ewarp, uint32_t rank, int split, int half, int tidx,
                                              bool first_pass, bool last_pass, bool &tail_ok, uint64_t d_policy,
                                              volatile uint32_t *abort_flag, const CUtensorMap *tmap_d,
                                              uint32_t stg)
{
    if (half >= 0) {
        const int slot = tidx * CG + static_cast<int>(rank);
        float *part = args.tail_ws + (static_cast<int64_t>(slot) * BN + c0) * kBM + 32 * q + lane;
        unsigned long long *flag = args.tail_flags + slot * kEpiWarps + ewarp;
        if (half == 0) {
#pragma unroll
            for (int i = 0; i < PC; ++i) __stcg(part + i * kBM, __uint_as_float(v[i]));
            if (last_pass) {
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_gpu_u64(flag, args.epoch);
            }
            return;
        }
        if (first_pass) {
            bool ok = true;
            if (lane == 0) ok = wait_flag(flag, args.epoch, args.wait_ns, abort_flag);
            tail_ok = __shfl_sync(0xFFFFFFFFu, ok, 0) && ld_acquire_gpu_u64(flag) == args.epoch;
        }
        if (tail_ok) {
#pragma unroll
            for (int i = 0; i < PC; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __ldcg(part + i * kBM));
        }
    }
    // local rows of the tile's problem (the group's, when grouped)
    const int row_base = (tg.ta * CG + static_cast<int>(rank)) * kBM + 32 * q;  // this warp's first row
    const int ra = row_base + lane;                                               // slot-A row of this lane
    const int col0 = tg.tb * BN + c0;                                             // first slot-B row
    const bool glu = args.act == FP4_ACT_SWIGLU;
    if (args.mode != kEpiSplitK) {
        // z = alpha * acc + bias, then the activation. Rows mode: v[i] is GEMM
        // column col0 + i; transposed: every v[i] of this lane is GEMM column ra.
        if (args.bias) {
            const float *bias = args.bias + tg.bias_off;
            if (args.mode == kEpiRows) {
#pragma unroll
                for (int i = 0; i < PC; ++i) {
                    const float b = col0 + i < tg.lb ? __ldg(bias + col0 + i) : 0.0f;
                    v[i] = __float_as_uint(fmaf(__uint_as_float(v[i]), args.alpha, b));
                }
            } else {
                const float b = ra < tg.la ? __ldg(bias + ra) : 0.0f;
#pragma unroll
                for (int i = 0; i < PC; ++i) v[i] = __float_as_uint(fmaf(__uint_as_float(v[i]), args.alpha, b));
            }
        } else {
#pragma unroll
            for (int i = 0; i < PC; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * args.alpha);
        }
        if (glu) {
            if (args.mode == kEpiRows) {
                // gate = even column, up = odd column: pack the PC/2 results into v[0 .. PC/2)
#pragma unroll
                for (int j = 0; j < PC / 2; ++j)
                    v[j] = __float_as_uint(silu(__uint_as_float(v[2 * j])) * __uint_as_float(v[2 * j + 1]));
            } else {
                // gate on the even lane, up on the odd lane next to it
#pragma unroll
                for (int i = 0; i < PC; ++i) {
                    const float z = __uint_as_float(v[i]);
                    const float up = __shfl_xor_sync(0xFFFFFFFFu, z, 1);
                    v[i] = __float_as_uint(silu(z) * up);
                }
            }
        } else if (args.act != FP4_ACT_NONE) {
#pragma unroll
            for (int i = 0; i < PC; ++i) v[i] = __float_as_uint(activate(__uint_as_float(v[i]), args.act));
        }
    }
    if (args.mode == kEpiRows) {
        // this lane's D row in 32-byte column pieces; SwiGLU stores half as many
        // columns, from D column col0 / 2
        const int oc0 = glu ? col0 >> 1 : col0;
        const int ocols = glu ? tg.lb >> 1 : tg.lb;
        const int nval = glu ? PC / 2 : PC;
        if (TMA_D && args.tma_d && (nval * (args.bf16 ? 2 : 4)) % 128 == 0) {
            // Boxes of the warp's 32 rows x 128 bytes through its staging buffer,
            // written with the 128-byte swizzle (16-byte chunk j of row r at
            // r * 128 + (j ^ r % 8) * 16) and stored by one TMA instruction each.
            // The TMA clips rows and columns past D; a box wholly past it is skipped.
            // (A warp whose columns do not fill whole boxes, bf16 SwiGLU with
            // N tiles of 128, keeps the direct stores: a box would cover the
            // neighbouring warp's columns.)
            const int y = tg.da + row_base;
            const bool rows_in = y < tg.da + tg.la;
            const uint32_t row_addr = stg + static_cast<uint32_t>(lane) * 128u;
            auto put_box = [&](int x, auto chunk) {
                if (lane == 0) bulk_wait_read_all();     // the previous box has left the buffer
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 w = chunk(j);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                     row_addr + (static_cast<uint32_t>(j ^ (lane & 7)) << 4)),
                                 "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                                 : "memory");
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0 && rows_in && x < ocols) {
                    tma_store_2d(tmap_d, stg, x, y, d_policy);
                    bulk_commit_group();
                }
            };
            if (args.bf16) {
#pragma unroll
                for (int b = 0; b < PC / 64; ++b) {
                    if (64 * b < nval)
                        put_box(oc0 + 64 * b, [&](int j) {
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(v[64 * b + 8 * j + 2 * i]),
                                                                         __uint_as_float(v[64 * b + 8 * j + 2 * i + 1]));
                                w[i] = *reinterpret_cast<uint32_t *>(&p);
                            }
                            return make_uint4(w[0], w[1], w[2], w[3]);
                        });
                }
            } else {
#pragma unroll
                for (int b = 0; b < PC / 32; ++b) {
                    if (32 * b < nval)
                        put_box(oc0 + 32 * b, [&](int j) {
                            return make_uint4(v[32 * b + 4 * j], v[32 * b + 4 * j + 1], v[32 * b + 4 * j + 2],
                                              v[32 * b + 4 * j + 3]);
                        });
                }
            }
        } else if (args.bf16) {
#pragma unroll
            for (int ch = 0; ch < PC / 16; ++ch) {
                if (16 * ch < nval) {
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(v[16 * ch + 2 * i]),
                                                                 __uint_as_float(v[16 * ch + 2 * i + 1]));
                        w[i] = *reinterpret_cast<uint32_t *>(&p);
                    }
                    store_row32(w, args.out, args.ldo, 2, tg.da + ra, oc0 + 16 * ch, 8, tg.da + tg.la, ocols,
                                args.st32, d_policy);
                }
            }
        } else {
#pragma unroll
            for (int ch = 0; ch < PC / 8; ++ch) {
                if (8 * ch < nval) {
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[i] = v[8 * ch + i];
                    store_row32(w, args.out, args.ldo, 4, tg.da + ra, oc0 + 8 * ch, 4, tg.da + tg.la, ocols,
                                args.st32, d_policy);
                }
            }
        }
    } else if (TMA_D && args.tma_d && args.mode == kEpiTransposed && !glu) {
        // D^T through TMA boxes: the warp's 32 GEMM columns are 32 consecutive D
        // columns; a box is those columns x R D rows (R = 4 KB / 32 elements), laid
        // out row by row in the staging buffer (lane l writes element l of each
        // row, so a row's 32 writes are one contiguous piece). The TMA clips rows
        // and columns past D; a box wholly past it is skipped.
        const int x = tg.da + row_base;
        const int y0 = tg.db + col0;
        const bool cols_in = x < tg.da + tg.la;
        auto box_done = [&](int y) {
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0 && cols_in && y < tg.db + tg.lb) {
                tma_store_2d(tmap_d, stg, x, y, d_policy);
                bulk_commit_group();
            }
        };
        if (args.bf16) {
#pragma unroll
            for (int b = 0; b < PC / 64; ++b) {
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const uint16_t e = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[64 * b + i])));
                    asm volatile("st.shared.b16 [%0], %1;" ::"r"(stg + static_cast<uint32_t>((i * 32 + lane) * 2)),
                                 "h"(e)
                                 : "memory");
                }
                box_done(y0 + 64 * b);
            }
        } else {
#pragma unroll
            for (int b = 0; b < PC / 32; ++b) {
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(stg + static_cast<uint32_t>((i * 32 + lane) * 4)),
                                 "r"(v[32 * b + i])
                                 : "memory");
                box_done(y0 + 32 * b);
            }
        }
    } else if (ra < tg.la) {
        if (args.mode == kEpiSplitK) {
            // fp32 partials, transposed: for a fixed column the 32 lanes of a warp
            // write 32 consecutive elements
            float *ws = static_cast<float *>(args.out) + split * args.split_stride + ra;
#pragma unroll
            for (int i = 0; i < PC; ++i)
                if (col0 + i < args.rows_b)
                    st_global_b32_hint(ws + static_cast<int64_t>(col0 + i) * args.ldo, v[i], d_policy);
        } else if (!glu || (lane & 1) == 0) {
            // D^T: this lane's GEMM column ra (SwiGLU: D column ra / 2, from the gate
            // lane); D row db + (slot-B row)
            const int oc = tg.da + (glu ? ra >> 1 : ra);
            const int r0 = tg.db + col0;
            if (args.bf16) {
                __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(args.out) + oc;
#pragma unroll
                for (int i = 0; i < PC; ++i)
                    if (col0 + i < tg.lb)
                        st_global_b16_hint(d + static_cast<int64_t>(r0 + i) * args.ldo,
                                           __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[i]))), d_policy);
            } else {
                float *d = static_cast<float *>(args.out) + oc;
#pragma unroll
                for (int i = 0; i < PC; ++i)
                    if (col0 + i < tg.lb) st_global_b32_hint(d + static_cast<int64_t>(r0 + i) * args.ldo, v[i], d_policy);
            }
        }
    }
}

// End of a warp role: all of the block (and of the pair) meets once every
// role's work, with its copies, MMAs and TMEM accesses, is done. Each role
// branch has its own copy (the branches run with different register counts, so
// no code may follow them in common).
template <int CG>
__device__ __forceinline__ void role_end()
{
    __syncwarp();
    tc_fence_before();
    if constexpr (CG == 2) cluster_sync_any(); else cta_sync_any();
    tc_fence_after();
}

template <int CG, int BN, bool MX, bool GROUPED>
__device__ __forceinline__ void gemm_body(const CUtensorMap *tmap_d, const CUtensorMap &tmap_a, const CUtensorMap &tmap_b,
                                          const CUtensorMap &tmap_sfa, const CUtensorMap &tmap_sfb, const Args &args,
                                          const GroupParams *gp)
{
    using C = Cfg<CG, BN, MX>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const base_ptr = smem_raw + (base - raw);

    // Barriers, per stage s: full (the leader's: both CTAs' operand tiles landed),
    // full_sf (this CTA's scale atoms landed), empty (the stage's MMAs completed;
    // the leader's commit reaches both CTAs), ready (the leader's: both CTAs'
    // scale warps have stored the stage's scales in TMEM and the leader's have
    // seen `full`, so the MMA issuer waits on this one barrier alone).
    const uint32_t bar_full = base + C::OFF_BAR;
    const uint32_t bar_full_sf = bar_full + 8 * C::STAGES;
    const uint32_t bar_empty = bar_full_sf + 8 * C::STAGES;
    const uint32_t bar_ready = bar_empty + 8 * C::STAGES;
    const uint32_t bar_acc_full = bar_ready + 8 * C::STAGES;
    const uint32_t bar_acc_empty = bar_acc_full + 16;
    const uint32_t bar_drain = bar_acc_empty + 16;
    uint32_t *const tmem_holder = reinterpret_cast<uint32_t *>(base_ptr + C::OFF_BAR + 32 * C::STAGES + 40);
    volatile uint32_t *const abort_flag =
        reinterpret_cast<volatile uint32_t *>(base_ptr + C::OFF_BAR + 32 * C::STAGES + 44);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;   // 0 = leader of the pair
    const int pair = CG == 2 ? static_cast<int>(blockIdx.x / 2) : static_cast<int>(blockIdx.x);
    const int npairs = CG == 2 ? static_cast<int>(gridDim.x / 2) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_full_sf + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
            mbar_init(bar_ready + 8 * s, kSfWarps * CG);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full + 8 * b, 1);
            mbar_init(bar_acc_empty + 8 * b, kEpiWarps * CG);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        prefetch_tensormap(&tmap_sfa);
        prefetch_tensormap(&tmap_sfb);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // Launched as a dependent of the scale reorder, the set-up above overlaps
    // its tail; nothing in memory is touched before it has completed.
    griddep_wait();

    // Roles by warpgroup; each warpgroup's register split comes first in its own
    // branch, so the code after it is compiled for that many registers.
    if (warp < kFirstEpiWarp) {
        regs_lower<kLowRegs>();
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // every CTA's operand tiles signal the leader's full barrier (the leader
            // posts the byte count of both CTAs); its scale atoms signal its own
            // full_sf barrier
            const uint32_t full0 = CG == 2 ? mapa_shared(bar_full, 0) : bar_full;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t filled = 0, fill_parity = 0;
            uint32_t pfilled = 0;                 // stages this producer has filled
            bool ok = true;
            for (int u = pair; ok && u < args.units; u += npairs) {
                int ta, tb, split, kt0, kt1, half, tidx;
                unit_work<GROUPED>(args, u, ta, tb, split, kt0, kt1, half, tidx);
                TileGeo tg;
                tile_geo<GROUPED>(args, gp, u, ta, tb, tg);
                const int rba = tg.ta * CG + static_cast<int>(rank);     // this CTA's 128-row block of slot A
                const int row_a = tg.oa + rba * kBM;
                const int row_b = tg.ob + tg.tb * BN + static_cast<int>(rank) * C::BN_CTA;
                const int sba = tg.sa + rba;                             // its scale block
                const int rbb = tg.sb + (tg.tb * BN) / 128;              // first scale block of the N side
                for (int kt = kt0; kt < kt1; ++kt) {
                    if (args.stop_after > 0 && pfilled >= static_cast<uint32_t>(args.stop_after)) {
                        ok = false;     // (bounded-wait test: this stage is never loaded)
                        break;
                    }
                    if (!wait(bar_empty + 8 * stage, phase ^ 1u, args.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ++pfilled;
                    const uint32_t full = full0 + 8 * stage;                 // shared::cluster address
                    const uint32_t full_sf = bar_full_sf + 8 * stage;
                    if (rank == 0) mbar_arrive_expect_tx(bar_full + 8 * stage, C::OPND_TX);
                    mbar_arrive_expect_tx(full_sf, C::SF_TX);
                    // the scale atoms first: they land first, and the scale warps
                    // stage them into TMEM while the operand tiles are still landing
                    // (measured 1-2% faster than operands first on every large shape)
                    tma_load_2d<1>(base + C::OFF_SFA + stage * C::SFA_BYTES, &tmap_sfa, full_sf,
                                   kt * C::APK * (kAtomBytes / 8), sba);
                    tma_load_2d<1>(base + C::OFF_SFB + stage * C::SFB_BYTES, &tmap_sfb, full_sf,
                                   kt * C::APK * (kAtomBytes / 8), rbb);
                    tma_load_2d<CG>(base + C::OFF_A + stage * C::A_BYTES, &tmap_a, full, kt * kBKBytes, row_a);
                    tma_load_2d<CG>(base + C::OFF_B + stage * C::B_BYTES, &tmap_b, full, kt * kBKBytes, row_b);
                    filled |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    ring_next<C::STAGES>(stage, phase);
                }
            }
            // Every copy this CTA issued lands before it can exit: its scale atoms on
            // its own barriers, both CTAs' operand tiles on the leader's.
            for (int s = 0; s < C::STAGES; ++s)
                if (filled & (1u << s)) {
                    wait(bar_full_sf + 8 * s, (fill_parity >> s) & 1u, args.wait_ns, nullptr);
                    if (rank == 0) wait(bar_full + 8 * s, (fill_parity >> s) & 1u, args.wait_ns, nullptr);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // This thread issues only MMAs and commits. The tensor pipe queues about
        // one MMA beyond the one running, so whatever this thread does between
        // two k-tiles' MMAs must stay short: it waits on one barrier per stage
        // (ready), and tests up to four stages ahead in one batched, non-blocking
        // probe, so that a run of landed stages costs one shared-memory round trip.
        if (lane == 0 && rank == 0) {
            // Instruction descriptors: MXFP4 alternates the scale byte ids 0 / 2
            // between the two K=64 halves of one 4-block atom.
            constexpr uint32_t ID0 = idesc_fp4(kBM * CG, BN, MX, 0, 0);
            constexpr uint32_t ID2 = idesc_fp4(kBM * CG, BN, MX, 2, 2);
            // K-major, 128-byte swizzle: rows 128 bytes apart, 8-row groups 1024
            // apart; MMA j of a k-tile starts 32 bytes (two 16-byte units) in.
            const uint64_t desc_a0 = smem_desc(base + C::OFF_A, 16, 1024, 2);
            const uint64_t desc_b0 = smem_desc(base + C::OFF_B, 16, 1024, 2);
            int stage = 0;
            uint32_t phase = 0;
            int known = 0;                  // k-tiles from (stage, phase) on seen ready
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = pair; ok && u < args.units; u += npairs) {
                int ta, tb, split, kt0, kt1, half, tidx;
                unit_work<GROUPED>(args, u, ta, tb, split, kt0, kt1, half, tidx);
                // the epilogue has drained this accumulator (once per tile)
                if (!wait_cluster(bar_acc_empty + 8 * acc, acc_phase ^ 1u, args.wait_ns, abort_flag)) break;
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
                for (int kt = kt0; kt < kt1; ++kt) {
                    // the stage's operands (both CTAs) and scales (both CTAs' TMEM) are in place
                    if (known == 0) {
                        known = ready_run<C::STAGES>(bar_ready, stage, phase);
                        if (known == 0) {
                            if (!wait_cluster(bar_ready + 8 * stage, phase, args.wait_ns, abort_flag)) {
                                ok = false;
                                break;
                            }
                            known = 1;
                        }
                        tc_fence_after();
                    }
                    --known;
                    const uint32_t sf = tmem + static_cast<uint32_t>(C::SF_TMEM + stage * C::SF_COLS);
                    const uint64_t da = desc_a0 + static_cast<uint64_t>((stage * C::A_BYTES) >> 4);
                    const uint64_t db = desc_b0 + static_cast<uint64_t>((stage * C::B_BYTES) >> 4);
#pragma unroll
                    for (int i = 0; i < kBK / 64; ++i) {
                        const int t = MX ? (i >> 1) : i;
                        const uint32_t idesc = (MX && (i & 1)) ? ID2 : ID0;
                        tc_mma_fp4<CG, MX>(d_tmem, da + 2 * i, db + 2 * i, idesc, sf + 4 * t,
                                           sf + 4 * C::APK + 4 * C::NRB * t, (kt > kt0 || i > 0) ? 1u : 0u);
                    }
                    // frees the stage: its shared memory and its TMEM scale columns
                    tc_commit<CG>(bar_empty + 8 * stage);
                    ring_next<C::STAGES>(stage, phase);
                }
                if (!ok) break;
                tc_commit<CG>(bar_acc_full + 8 * acc);
                if (C::ACC_BUFS == 2) {
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                } else {
                    acc_phase ^= 1u;
                }
            }
            // Every MMA this thread issued completes before teardown.
            tc_commit<CG>(bar_drain, 1);
            wait(bar_drain, 0, args.wait_ns, nullptr);
        }
    }
        role_end<CG>();
        if (warp == 1) tmem_dealloc<CG>(tmem, C::TMEM_COLS);
    } else if (warp >= kFirstSfWarp) {
        regs_lower<kLowRegs>();
        // ------------------------------------------------------------ scale warps
        // Two scale warps per TMEM lane quarter q, each staging half of every
        // k-tile's scale atoms (half h: slot-A atoms h*HA .., slot-B atoms h*HG ..)
        // into this quarter's lanes of the stage's TMEM scale columns with
        // tcgen05.st, then arriving on the leader's ready barrier; in the leader,
        // the (quarter 0, half 0) warp first waits for the stage's operand tiles
        // (full), so that ready alone tells the MMA issuer the stage is complete.
        // Every warp takes every k-tile, so it waits on every phase of the
        // barriers it helps complete, in order (a parity wait is only sound when
        // the waiter has seen the barrier's previous phase and the next one cannot
        // complete without it), and the staging latency of a k-tile is that of
        // half its atoms. Word c of line i of a scale atom holds the four scales
        // of row 32c + i for one K-chunk. Slot-A atom t goes to columns
        // 4t .. 4t+3, of which the MMA reads, in quarter q, only column 4t + q:
        // so the warp loads just word q of its lane's line (4 bytes per atom) and
        // stores that one column. Slot-B atom (t, rb), group g = t*NRB + rb, goes
        // to columns 4 (APK + g) + c, all four of which the MMA reads in every
        // quarter: the warp loads whole 16-byte lines. (Copying the atoms with
        // tcgen05.cp instead, beside the MMAs, measured 1.5-2.5x slower per k-tile
        // on this part; one warp per quarter staging a whole k-tile, with all four
        // slot-A columns, left NVFP4 bound by the ring's latency at ~850 cycles
        // per k-tile.)
        const int q = warp & 3;
        const int h = (warp - kFirstSfWarp) >> 2;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t ready0 = CG == 2 ? mapa_shared(bar_ready, 0) : bar_ready;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = pair; ok && u < args.units; u += npairs) {
            int ta, tb, split, kt0, kt1, half, tidx;
            unit_work<GROUPED>(args, u, ta, tb, split, kt0, kt1, half, tidx);
            for (int kt = kt0; kt < kt1; ++kt) {
                // this CTA's scale atoms of the stage have landed (which also means
                // the MMAs that read the slot's previous scales have completed)
                bool landed = true;
                if (lane == 0) landed = wait(bar_full_sf + 8 * stage, phase, args.wait_ns, abort_flag);
                if (!__shfl_sync(0xFFFFFFFFu, landed, 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col = lane_base + tmem + static_cast<uint32_t>(C::SF_TMEM + stage * C::SF_COLS);
                const uint8_t *sfa = base_ptr + C::OFF_SFA + stage * C::SFA_BYTES + lane * 16 + q * 4;
                const uint8_t *sfb = base_ptr + C::OFF_SFB + stage * C::SFB_BYTES + lane * 16;
#pragma unroll
                for (int i = 0; i < C::HA; ++i) {
                    const int t = h * C::HA + i;
                    tmem_st_32x32b_x1(col + static_cast<uint32_t>(4 * t + q),
                                      *reinterpret_cast<const uint32_t *>(sfa + t * kAtomBytes));
                }
                uint32_t r[4 * C::HG];
#pragma unroll
                for (int i = 0; i < C::HG; ++i) {
                    const int g = h * C::HG + i;
                    const uint4 w =
                        *reinterpret_cast<const uint4 *>(sfb + ((g % C::NRB) * C::APK + g / C::NRB) * kAtomBytes);
                    r[4 * i] = w.x, r[4 * i + 1] = w.y, r[4 * i + 2] = w.z, r[4 * i + 3] = w.w;
                }
                const uint32_t colb = col + static_cast<uint32_t>(4 * C::APK + 4 * h * C::HG);
                if constexpr (C::HG == 4)
                    tmem_st_32x32b_x16(colb, r);
                else if constexpr (C::HG == 2)
                    tmem_st_32x32b_x8(colb, r);
                else
                    tmem_st_32x32b_x4(colb, r);
                tmem_st_wait();
                tc_fence_before();
                bool opnd = true;
                if (lane == 0 && rank == 0 && q == 0 && h == 0)
                    opnd = wait(bar_full + 8 * stage, phase, args.wait_ns, abort_flag);
                if (!__shfl_sync(0xFFFFFFFFu, opnd, 0)) {    // (also: every lane's stores are done)
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    if constexpr (CG == 2)
                        mbar_arrive_cluster(ready0 + 8 * stage);
                    else
                        mbar_arrive(bar_ready + 8 * stage);
                }
                ring_next<C::STAGES>(stage, phase);
            }
        }
        role_end<CG>();
    } else {
        regs_raise<kEpiRegs>();
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                          // TMEM lane quarter of this warp
        const int ew = warp - kFirstEpiWarp;             // epilogue warp index
        const uint32_t stg = base + C::OFF_STG + static_cast<uint32_t>(ew * C::STG_WARP);   // its D staging box
        const int h = ew >> 2;                           // which half of the tile's columns
        const uint32_t acc_empty0 = CG == 2 ? mapa_shared(bar_acc_empty, 0) : bar_acc_empty;
        // D is written once and not read again here: evict it from L2 first, so the
        // operand tiles that other CTAs still load stay resident.
        const uint64_t d_policy = policy_evict_first();
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = pair; u < args.units; u += npairs) {
            int ta, tb, split, kt0, kt1, half, tidx;
            unit_work<GROUPED>(args, u, ta, tb, split, kt0, kt1, half, tidx);
            TileGeo tg;
            tile_geo<GROUPED>(args, gp, u, ta, tb, tg);
            if (!wait(bar_acc_full + 8 * acc, acc_phase, args.wait_ns, abort_flag)) break;
            tc_fence_after();
            // This warp's 32 lanes x BN/2 columns, in passes; the accumulator is
            // handed back as soon as the last pass is in registers.
            bool tail_ok = false;
#pragma unroll 1
            for (int p = 0; p < C::PASSES; ++p) {
                const int c0 = h * C::COLS_WARP + p * C::PASS_COLS;
                uint32_t v[C::PASS_COLS];
                tmem_load_cols<C::PASS_COLS>(tmem + (static_cast<uint32_t>(32 * q) << 16) +
                                                 static_cast<uint32_t>(acc * BN + c0),
                                             v);
                tmem_ld_wait_regs(v);
                if (p == C::PASSES - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (CG == 2)
                            mbar_arrive_cluster(acc_empty0 + 8 * acc);
                        else
                            mbar_arrive(bar_acc_empty + 8 * acc);
                    }
                }
                epilogue_pass<CG, BN, C::PASS_COLS, C::TMA_D && !GROUPED>(
                    v, args, tg, c0, q, lane, ew, rank, split, half, tidx, p == 0, p == C::PASSES - 1, tail_ok,
                    d_policy, abort_flag, tmap_d, stg);
            }
            if (C::ACC_BUFS == 2) {
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            } else {
                acc_phase ^= 1u;
            }
        }
        // the TMA stores this warp issued have completed before the CTA exits
        if (C::TMA_D && !GROUPED && lane == 0) bulk_wait_all();
        role_end<CG>();
    }
}

template <int CG, int BN, bool MX>
__global__ void __launch_bounds__(kThreads, 1)
    fp4_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                    const Args args, const __grid_constant__ CUtensorMap tmap_d)
{
    gemm_body<CG, BN, MX, false>(&tmap_d, tmap_a, tmap_b, tmap_sfa, tmap_sfb, args, nullptr);
}

template <int CG, int BN, bool MX>
__global__ void __launch_bounds__(kThreads, 1)
    fp4_gemm_grouped_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                            const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                            const Args args, const __grid_constant__ GroupParams groups)
{
    gemm_body<CG, BN, MX, true>(nullptr, tmap_a, tmap_b, tmap_sfa, tmap_sfb, args, &groups);
}

// Split-K: z[rb][ra] = alpha * sum_s ws[s][rb][ra] (+ bias[ra]) in a fixed
// order (deterministic), then the fused epilogue into D[rb][.]. With splits = 0
// (K = 0) z is the bias alone.
__device__ __forceinline__ float splitk_z(const float *__restrict__ ws, int64_t at, int splits, int64_t split_stride,
                                          float alpha, const float *__restrict__ bias, int64_t ra)
{
    float s = 0.f;
    for (int k = 0; k < splits; ++k) s += ws[k * split_stride + at];
    return bias ? fmaf(s, alpha, bias[ra]) : s * alpha;
}

__global__ void splitk_reduce_kernel(const float *__restrict__ ws, void *__restrict__ out, int64_t rows_b,
                                     int64_t rows_a, int64_t ldd, int splits, int64_t split_stride, float alpha,
                                     int bf16, const float *__restrict__ bias, int act)
{
    const bool glu = act == FP4_ACT_SWIGLU;
    const int64_t cols = glu ? rows_a / 2 : rows_a;   // D columns
    const int64_t total = rows_b * cols;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t rb = i / cols, c = i - rb * cols;
        float r;
        if (glu) {
            const float g = splitk_z(ws, rb * rows_a + 2 * c, splits, split_stride, alpha, bias, 2 * c);
            const float u = splitk_z(ws, rb * rows_a + 2 * c + 1, splits, split_stride, alpha, bias, 2 * c + 1);
            r = silu(g) * u;
        } else {
            r = activate(splitk_z(ws, rb * rows_a + c, splits, split_stride, alpha, bias, c), act);
        }
        if (bf16)
            static_cast<__nv_bfloat16 *>(out)[rb * ldd + c] = __float2bfloat16_rn(r);
        else
            static_cast<float *>(out)[rb * ldd + c] = r;
    }
}

// Which source rows an atom row-block holds. Plain (groups == 0): block rb
// holds rows rb*128 .. of a `rows`-row matrix. Grouped (each group's rows start
// a fresh 128-row block): every group `uniform` rows (uniform > 0), or group g
// = rows row0[g] .. row0[g+1]-1 starting at block first_blk[g].
struct RowBlocks {
    int32_t groups;
    int32_t uniform;
    int32_t first_blk[kMaxGroups + 1];
    int32_t row0[kMaxGroups + 1];
};

__device__ __forceinline__ void block_rows(const RowBlocks &rbm, int64_t rows, int64_t rb, int64_t &src0,
                                           int64_t &valid)
{
    src0 = rb * 128;
    valid = rows - rb * 128;
    if (rbm.groups > 0 && rbm.uniform > 0) {
        const int64_t per = (rbm.uniform + 127) / 128;
        const int64_t g = rb / per, b = rb - g * per;
        src0 = g * rbm.uniform + 128 * b;
        valid = rbm.uniform - 128 * b;
    } else if (rbm.groups > 0) {
        int lo = 0, hi = rbm.groups - 1;          // the last group starting at or before rb
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (rbm.first_blk[mid] <= rb) lo = mid; else hi = mid - 1;
        }
        const int64_t b = rb - rbm.first_blk[lo];
        src0 = rbm.row0[lo] + 128 * b;
        valid = rbm.row0[lo + 1] - rbm.row0[lo] - 128 * b;
    }
    valid = valid < 0 ? 0 : (valid > 128 ? 128 : valid);
}

// Scale reorder: row-major sf[rows][ksf] -> 128x4 atoms. A CTA takes a tile of
// one 128-row block x 32 scale columns (8 atoms): each thread reads one
// 16-byte piece (two per row, so a warp's load covers whole 32-byte sectors of
// 16 rows) into shared memory (rows padded to 9 words, so the transposing
// reads below are conflict-free), then writes one 16-byte atom line -- line i
// of an atom holds rows i, i+32, i+64, i+96 of the block, 4 columns each -- so
// a warp writes one 512-byte atom. Zero past the matrix. One launch can carry
// two matrices (the two operands of a GEMM call): job 0's tiles, then job 1's.
constexpr int kReorderThreads = 256;
constexpr int kReorderAtoms = 8;                  // atoms (of 4 scale columns) per tile
constexpr int kReorderRowWords = kReorderAtoms + 1;

struct ReorderJob {
    const uint8_t *sf;
    uint4 *out;
    int64_t rows, row_blocks, tiles;
};

__global__ void __launch_bounds__(kReorderThreads)
    scale_reorder_kernel(ReorderJob j0, ReorderJob j1, int64_t ksf, int64_t kc4,
                         const __grid_constant__ RowBlocks map0, const __grid_constant__ RowBlocks map1)
{
    __shared__ uint32_t tile[128 * kReorderRowWords];
    griddep_launch_dependents();          // the GEMM that follows may start its set-up
    const int64_t col_tiles = (kc4 + kReorderAtoms - 1) / kReorderAtoms;
    const int64_t ncols = kReorderAtoms * 4;
    for (int64_t t = blockIdx.x; t < j0.tiles + j1.tiles; t += gridDim.x) {
        const bool second = t >= j0.tiles;
        const ReorderJob &j = second ? j1 : j0;
        const int64_t tt = second ? t - j0.tiles : t;
        const int64_t rb = tt / col_tiles, ct = tt - rb * col_tiles;
        int64_t src0, valid;
        block_rows(second ? map1 : map0, j.rows, rb, src0, valid);
        const int64_t c0 = ct * ncols;                // first scale column of the tile
        const bool vec16 = (ksf & 15) == 0 && (reinterpret_cast<uintptr_t>(j.sf) & 15) == 0;
        __syncthreads();                              // the previous tile's reads are done
        {
            const int r = threadIdx.x >> 1, pc = threadIdx.x & 1;   // row, 16-byte piece
            const int64_t col = c0 + 16 * pc;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (r < valid && col < ksf) {
                const uint8_t *src = j.sf + (src0 + r) * ksf + col;
                if (vec16) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
                    w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
                } else {
                    for (int b = 0; b < 16 && col + b < ksf; ++b)
                        w[b >> 2] |= static_cast<uint32_t>(__ldg(src + b)) << (8 * (b & 3));
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) tile[r * kReorderRowWords + 4 * pc + q] = w[q];
        }
        __syncthreads();
        {
            const int a = threadIdx.x >> 5, i = threadIdx.x & 31;  // line i of atom a
            if (ct * kReorderAtoms + a < kc4) {
                const uint4 v = make_uint4(tile[i * kReorderRowWords + a], tile[(i + 32) * kReorderRowWords + a],
                                           tile[(i + 64) * kReorderRowWords + a], tile[(i + 96) * kReorderRowWords + a]);
                j.out[(rb * kc4 + ct * kReorderAtoms + a) * 32 + i] = v;
            }
        }
    }
}

// ============================================================================ host

namespace {

std::mutex g_mu;
int64_t g_wait_ms = -1;
std::atomic<unsigned long long> g_epoch{0};   // launches so far (see next_epoch)

// The split-tail flags' value for the next launch. The flags live in scratch
// that earlier calls (or other code) filled with arbitrary bytes, so a flag
// counts as raised only when it holds this launch's value: a per-process random
// 64-bit nonce mixed with the launch counter through a bijective finaliser
// (SplitMix64's), so two launches of one process never share a value and stale
// bytes match one with probability 2^-64.
unsigned long long next_epoch()
{
    static const unsigned long long nonce = [] {
        std::random_device rd;
        unsigned long long n = (static_cast<unsigned long long>(rd()) << 32) ^ rd();
        n ^= static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count());
        return n;
    }();
    unsigned long long z = nonce + 0x9E3779B97F4A7C15ull * ++g_epoch;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z ? z : 1ull;
}
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// True when work issued to `stream` is being recorded into a CUDA graph (or
// when that cannot be told, so the caller takes the safe branch).
bool stream_capturing(cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        (void)cudaGetLastError();   // not sticky: keep it out of the launch checks
        return true;
    }
    return cs != cudaStreamCaptureStatusNone;
}

constexpr int kNumKernels = 22;   // kernel variants that can be launched (see kernel_index)
struct DeviceInfo {
    bool probed = false;
    bool ok = false;
    int sms = 0;
    bool attr_set[kNumKernels] = {};
    int max_clusters[kNumKernels] = {};
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

bool encode(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *ptr, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw)
{
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, dt, rank, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand map: rows x K/2 bytes, box of `box_rows` rows x one 128-byte k-tile,
// 128-byte swizzle.
bool encode_operand(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), static_cast<cuuint32_t>(box_rows)};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Scale-atom map: the atom buffer as int64 rows of ceil(K/vec/4) * 64 elements
// per 128-row block; a box is one k-tile's atoms of `box_blocks` blocks. Past the
// matrix the box is zero-filled.
bool encode_scales(CUtensorMap *m, const void *atoms, int64_t row_blocks, int64_t kc4, int apk, int box_blocks)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kc4 * 64), static_cast<cuuint64_t>(row_blocks)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kc4 * kAtomBytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(apk * 64), static_cast<cuuint32_t>(box_blocks)};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_INT64, 2, atoms, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Output map for TMA stores: D as rows x cols elements (fp32 or bf16) with the
// given row count; a box is 32 rows x 128 bytes, 128-byte swizzle.
bool encode_output(CUtensorMap *m, void *D, int64_t rows, int64_t cols, bool bf16)
{
    const int64_t esize = bf16 ? 2 : 4;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esize)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), 32u};
    return encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, D, dims, strides,
                  box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The same for swap-AB's transposed tiles: a box is 32 columns x (4 KB / 32
// elements) rows, no swizzle.
bool encode_output_t(CUtensorMap *m, void *D, int64_t rows, int64_t cols, bool bf16)
{
    const int64_t esize = bf16 ? 2 : 4;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esize)};
    const cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(4096 / (32 * esize))};
    return encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, D, dims, strides,
                  box, CU_TENSOR_MAP_SWIZZLE_NONE);
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

struct Maps {
    CUtensorMap a, b, sfa, sfb, d;      // d: only for TMA stores of D (rows mode, pairs)
};

// With `slots_out` set, only reports how many CTA groups a launch can keep
// resident (after the cap) and launches nothing.
template <int CG, int BN, bool MX, bool GROUPED>
cudaError_t launch_gemm(DeviceInfo &info, int kidx, int units, int cap, const Maps &m, const Args &args,
                        cudaStream_t stream, int *slots_out, const GroupParams *gp = nullptr)
{
    using C = Cfg<CG, BN, MX>;
    auto kern = [] {
        if constexpr (GROUPED) return fp4_gemm_grouped_kernel<CG, BN, MX>;
        else return fp4_gemm_kernel<CG, BN, MX>;
    }();
    cudaLaunchAttribute cluster_attr[2];
    cluster_attr[0].id = cudaLaunchAttributeClusterDimension;
    cluster_attr[0].val.clusterDim.x = CG;
    cluster_attr[0].val.clusterDim.y = 1;
    cluster_attr[0].val.clusterDim.z = 1;
    cluster_attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    cluster_attr[1].val.programmaticStreamSerializationAllowed = 1;
    std::unique_lock<std::mutex> lk(g_mu);      // (calls from several host threads)
    if (!info.attr_set[kidx]) {
        // The warpgroups' register split (setmaxnreg) draws on the registers the
        // block is launched with: a kernel built with fewer than kLaunchRegs per
        // thread is never launched (its raise would wait forever).
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        int slots = info.sms;
        if (CG == 2) {
            cudaLaunchConfig_t qc = {};
            qc.gridDim = dim3(2 * info.sms, 1, 1);
            qc.blockDim = dim3(kThreads, 1, 1);
            qc.dynamicSmemBytes = C::SMEM_BYTES;
            qc.attrs = cluster_attr;
            qc.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &qc) != cudaSuccess || n <= 0) {
                cudaGetLastError();
                n = info.sms / 2;
            }
            slots = n;
        }
        info.max_clusters[kidx] = slots;
        info.attr_set[kidx] = true;
    }
    const int slots = info.max_clusters[kidx];
    lk.unlock();
    if (slots_out) {
        *slots_out = cap > 0 ? std::max(1, std::min(slots, cap / CG)) : slots;
        return cudaSuccess;
    }
    int groups = std::min(units, slots);
    if (cap > 0) groups = std::min(groups, std::max(1, cap / CG));
    groups = std::max(groups, 1);
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(groups * CG, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = C::SMEM_BYTES;
    lc.stream = stream;
    // a pair needs its cluster shape; every launch may start as a programmatic
    // dependent of the preceding kernel (see griddep_wait)
    lc.attrs = CG == 2 ? cluster_attr : cluster_attr + 1;
    lc.numAttrs = CG == 2 ? 2 : 1;
    if constexpr (GROUPED)
        return cudaLaunchKernelEx(&lc, kern, m.a, m.b, m.sfa, m.sfb, args, *gp);
    else
        return cudaLaunchKernelEx(&lc, kern, m.a, m.b, m.sfa, m.sfb, args, m.d);
}

// Variants: one CTA: N 16..256, pair: N 128 / 256; each for both formats.
// Grouped: one CTA with N 64..256, or a pair with N 256.
int kernel_index(int cg, int bn, bool mx, bool grouped = false)
{
    if (grouped) {
        if (cg == 2) return bn == 256 ? 20 + (mx ? 1 : 0) : -1;                // 20..21
        return bn >= 64 ? 14 + (bn_index(bn) - 2) * 2 + (mx ? 1 : 0) : -1;   // 14..19
    }
    if (cg == 1) return bn_index(bn) * 2 + (mx ? 1 : 0);                   // 0..9
    return 10 + (bn == 256 ? 2 : 0) + (mx ? 1 : 0);                         // 10..13
}

cudaError_t launch_grouped(int cg, int bn, bool mx, DeviceInfo &info, int units, const Maps &m, const Args &args,
                           const GroupParams &gp, cudaStream_t stream)
{
    const int k = kernel_index(cg, bn, mx, true);
#define FP4_LAUNCH_G(CG_, BN_, MX_) \
    return launch_gemm<CG_, BN_, MX_, true>(info, k, units, 0, m, args, stream, nullptr, &gp)
    if (k < 0) return cudaErrorInvalidValue;
    if (cg == 2) {
        if (mx) FP4_LAUNCH_G(2, 256, true);
        FP4_LAUNCH_G(2, 256, false);
    }
    switch (bn) {
    case 64:
        if (mx) FP4_LAUNCH_G(1, 64, true);
        FP4_LAUNCH_G(1, 64, false);
    case 128:
        if (mx) FP4_LAUNCH_G(1, 128, true);
        FP4_LAUNCH_G(1, 128, false);
    default:
        if (mx) FP4_LAUNCH_G(1, 256, true);
        FP4_LAUNCH_G(1, 256, false);
    }
#undef FP4_LAUNCH_G
}

cudaError_t launch_by_cfg(int cg, int bn, bool mx, DeviceInfo &info, int units, int cap, const Maps &m,
                          const Args &args, cudaStream_t stream, int *slots_out = nullptr)
{
    const int k = kernel_index(cg, bn, mx);
#define FP4_LAUNCH(CG_, BN_, MX_) \
    return launch_gemm<CG_, BN_, MX_, false>(info, k, units, cap, m, args, stream, slots_out)
    if (cg == 2) {
        if (bn == 256) {
            if (mx) FP4_LAUNCH(2, 256, true);
            FP4_LAUNCH(2, 256, false);
        }
        if (mx) FP4_LAUNCH(2, 128, true);
        FP4_LAUNCH(2, 128, false);
    }
    switch (bn) {
    case 16:
        if (mx) FP4_LAUNCH(1, 16, true);
        FP4_LAUNCH(1, 16, false);
    case 32:
        if (mx) FP4_LAUNCH(1, 32, true);
        FP4_LAUNCH(1, 32, false);
    case 64:
        if (mx) FP4_LAUNCH(1, 64, true);
        FP4_LAUNCH(1, 64, false);
    case 128:
        if (mx) FP4_LAUNCH(1, 128, true);
        FP4_LAUNCH(1, 128, false);
    default:
        if (mx) FP4_LAUNCH(1, 256, true);
        FP4_LAUNCH(1, 256, false);
    }
#undef FP4_LAUNCH
}

struct Plan {
    bool swap;
    int bn;
    int cg;
    int splits;
    int cap;
};

int pow2_bn(int64_t rows)
{
    if (rows <= 16) return 16;
    if (rows <= 32) return 32;
    if (rows <= 64) return 64;
    if (rows <= 128) return 128;
    return 256;
}

// The narrow-M CUDA-core kernel: forced by mode 3 (M <= kGemvMaxM), or chosen
// automatically where it measured faster than the tcgen05 path (one launch
// instead of the scale reorder plus the GEMM): M == 1 with plain scales. On
// prepacked scales, and from M = 2, the tcgen05 path measured faster on
// 28672 x 4096. Either way only when its shared staging of A fits and B's
// scales are 2-byte aligned (it reads NVFP4 scale pairs as 16-bit words).
fp4_status choose_gemv(int64_t M, int64_t K, bool mx, int prepacked, const fp4_gemm_config *cfg, bool sfb_even,
                       bool &gemv)
{
    const int mode = cfg ? cfg->mode : 0;
    if (mode < 0 || mode > 3) return FP4_ERR_INVALID_ARG;
    const bool fits = gemv_smem_bytes(M, K, mx) != 0;
    if (mode == 3 && !fits) return FP4_ERR_UNSUPPORTED;
    if (mode == 3 && !sfb_even) return FP4_ERR_MISALIGNED;
    gemv = mode == 3 || (mode == 0 && fits && sfb_even && !prepacked && M == 1);
    return FP4_OK;
}

// Chooses direct vs swap-AB, the tile N, the CTA group, the K split and the
// k-tiles per stage. `rows_ok` says whether D's rows take 16-byte vector stores
// (pitch a multiple of 16 bytes), which direct mode needs.
fp4_status make_plan(int64_t M, int64_t N, int64_t K, bool rows_ok, bool mx, int sms, const fp4_gemm_config *cfg,
                     Plan &p)
{
    const int mode = cfg ? cfg->mode : 0;
    if (mode < 0 || mode > 2) return FP4_ERR_INVALID_ARG;   // (mode 3 never reaches here)
    if (cfg && (cfg->split_tail < 0 || cfg->split_tail > 1)) return FP4_ERR_INVALID_ARG;
    if (mode == 1)
        p.swap = false;
    else if (mode == 2)
        p.swap = true;
    else
        p.swap = (M <= 256) || !rows_ok;
    // Few tiles: where the plan so far leaves more than half of the CTA pairs
    // idle, direct mode with pairs and N tiles of 128 at least doubles the tiles
    // in flight (256 x 4096 x 14336: 30.3 against 34.8 us for swap-AB with N
    // tiles of 256; 512 x 4096 x 14336: 30.8 against 36.2 for direct with 256).
    bool direct128 = false;
    if (mode == 0 && !(cfg && (cfg->bn || cfg->cta_group)) && rows_ok && M > 128) {
        const int64_t pairs = std::max(1, sms / 2);
        const int64_t ra = p.swap ? N : M, rb = p.swap ? M : N;
        const int64_t bn0 = p.swap ? pow2_bn(rb) : 256;
        const int64_t cur = cdiv(ra, 2 * kBM) * cdiv(rb, bn0);       // pair tiles (bn0 >= 256 here)
        const int64_t t128 = cdiv(M, 2 * kBM) * cdiv(N, 128);
        direct128 = 2 * cur <= pairs && t128 <= pairs && t128 > cur;
    }
    if (direct128) p.swap = false;
    if (!p.swap && !rows_ok) return FP4_ERR_MISALIGNED;
    const int64_t rows_b = p.swap ? M : N;
    const int64_t rows_a = p.swap ? N : M;
    const int bn = (cfg && cfg->bn) ? cfg->bn : (direct128 ? 128 : (p.swap ? pow2_bn(rows_b) : 256));
    if (bn_index(bn) < 0) return FP4_ERR_INVALID_ARG;
    if (rows_b > bn && bn < 128) return FP4_ERR_UNSUPPORTED;       // N-side tiles must start on scale blocks
    p.bn = bn;
    // CTA pairs wherever the M side has more than one 128-row block: each CTA of a
    // pair loads half of the N side, so a k-tile takes 38 KB (NVFP4, N = 256) of
    // L2 -> shared memory traffic per SM instead of 54, and pairs store D with TMA
    // boxes. Measured faster for both formats on every large shape (8192^3 NVFP4
    // fp32: 217 against 262 us).
    const int cg = (cfg && cfg->cta_group) ? cfg->cta_group : ((bn >= 128 && rows_a > 128) ? 2 : 1);
    if (cg != 1 && cg != 2) return FP4_ERR_INVALID_ARG;
    if (cg == 2 && bn < 128) return FP4_ERR_UNSUPPORTED;
    p.cg = cg;
    const int64_t tiles = cdiv(rows_a, kBM * cg) * cdiv(rows_b, bn);
    const int64_t k_tiles = cdiv(K, kBK);
    const int slots = std::max(1, sms / cg);
    int splits = (cfg && cfg->splits) ? cfg->splits : 0;
    if (splits < 0) return FP4_ERR_INVALID_ARG;
    if (splits > 1 && !p.swap) return FP4_ERR_UNSUPPORTED;         // partials are written swap-AB style
    if (splits == 0) {
        splits = 1;
        if (p.swap && tiles < slots) {
            // Estimated cycles: waves of units x (k-tiles x per-k-tile time + per-unit
            // epilogue), plus, when split, the reduce launch, a set-up per split and
            // the fp32 partials (written transposed, then read by the reduce).
            // Fitted to a sweep of 11 skinny shapes (M 16-256, K 8192-28672):
            // a k-tile ~700 cycles for one CTA per MMA and ~900 for a pair, the
            // split's fixed cost ~21000 cycles, ~340 partial bytes per cycle. (An
            // earlier model, 10000 cycles and 1500 bytes per cycle, split shapes
            // where one split was faster: 256 x 2048 x 8192 42.6 against 23.9 us.)
            // Fewer splits win ties.
            const double kTileCycles = cg == 2 ? 900.0 : 700.0;
            constexpr double kUnitCycles = 1500.0, kReduceCycles = 21000.0, kSplitCycles = 1000.0;
            constexpr double kPartialBytesPerCycle = 340.0;
            double best = 1e30;
            for (int s = 1; s <= std::min<int64_t>(k_tiles, 16); ++s) {
                const double waves = static_cast<double>(cdiv(tiles * s, slots));
                double cost = waves * (static_cast<double>(cdiv(k_tiles, s)) * kTileCycles + kUnitCycles);
                if (s > 1)
                    cost += kReduceCycles + kSplitCycles * s +
                            s * static_cast<double>(rows_a) * rows_b * 4.0 / kPartialBytesPerCycle;
                if (cost < best - 1e-9) {
                    best = cost;
                    splits = s;
                }
            }
        }
    }
    p.splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(splits, k_tiles)));
    p.cap = (cfg && cfg->max_ctas > 0) ? cfg->max_ctas : 0;
    return FP4_OK;
}

// One reorder launch for up to two scale matrices with the same K (the second
// may be absent: sf1 == nullptr). `row_blocks` / `rbm`: the grouped forms (see
// RowBlocks); plain when rbm is null.
struct ReorderSpec {
    const void *sf = nullptr;
    void *out = nullptr;
    int64_t rows = 0;
    int64_t row_blocks = -1;
    const RowBlocks *rbm = nullptr;
};

fp4_status reorder2_launch(const ReorderSpec &a, const ReorderSpec &b, int64_t ksf, int sms, cudaStream_t stream)
{
    const int64_t kc4 = cdiv(ksf, 4);
    const int64_t col_tiles = cdiv(kc4, kReorderAtoms);
    auto job = [&](const ReorderSpec &sp) {
        ReorderJob j;
        j.sf = static_cast<const uint8_t *>(sp.sf);
        j.out = static_cast<uint4 *>(sp.out);
        j.rows = sp.rows;
        j.row_blocks = sp.sf ? (sp.rbm ? sp.row_blocks : cdiv(sp.rows, 128)) : 0;
        j.tiles = j.row_blocks * col_tiles;
        return j;
    };
    const ReorderJob j0 = job(a), j1 = job(b);
    const int64_t tiles = j0.tiles + j1.tiles;
    if (tiles == 0) return FP4_OK;
    const int64_t blocks = std::min<int64_t>(tiles, static_cast<int64_t>(sms) * 8);
    static const RowBlocks plain = {};
    scale_reorder_kernel<<<static_cast<unsigned>(blocks), kReorderThreads, 0, stream>>>(
        j0, j1, ksf, kc4, a.rbm ? *a.rbm : plain, b.rbm ? *b.rbm : plain);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

fp4_status reorder_launch(const void *sf_plain, void *sf_atom, int64_t rows, int64_t ksf, int sms,
                          cudaStream_t stream, int64_t row_blocks = -1, const RowBlocks *rbm = nullptr)
{
    ReorderSpec a;
    a.sf = sf_plain;
    a.out = sf_atom;
    a.rows = rows;
    a.row_blocks = row_blocks;
    a.rbm = rbm;
    return reorder2_launch(a, ReorderSpec(), ksf, sms, stream);
}

// `ext_scratch` (with `ext_bytes`), when given, replaces the stream-ordered
// allocation of the call's scratch; a plan that needs more is refused.
fp4_status gemm_impl(fp4_format fmt, int prepacked, const void *A, const void *sfA, const void *B,
                     const void *sfB, float alpha, void *D, int64_t M, int64_t N, int64_t K, fp4_out_dtype out,
                     const fp4_gemm_config *cfg, cudaStream_t stream, uint8_t *ext_scratch = nullptr,
                     size_t ext_bytes = 0, const fp4_epilogue *epi = nullptr)
{
    if (fmt != FP4_FMT_NVFP4 && fmt != FP4_FMT_MXFP4) return FP4_ERR_INVALID_ARG;
    if (out != FP4_OUT_F32 && out != FP4_OUT_BF16) return FP4_ERR_INVALID_ARG;
    const int act = epi ? epi->act : FP4_ACT_NONE;
    const float *bias = epi ? epi->bias : nullptr;
    if (act < FP4_ACT_NONE || act > FP4_ACT_SWIGLU) return FP4_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return FP4_ERR_INVALID_ARG;
    const bool glu = act == FP4_ACT_SWIGLU;
    if (glu && N % 2 != 0) return FP4_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FP4_OK;
    if (!D) return FP4_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(bias) & 3u) return FP4_ERR_MISALIGNED;
    const int64_t esize = out == FP4_OUT_BF16 ? 2 : 4;
    const int64_t d_cols = glu ? N / 2 : N;          // columns of D
    if (K == 0) {
        if (!aligned16(D)) return FP4_ERR_MISALIGNED;
        if (act == FP4_ACT_NONE && !bias)
            return cudaMemsetAsync(D, 0, static_cast<size_t>(M * d_cols * esize), stream) == cudaSuccess
                       ? FP4_OK
                       : FP4_ERR_CUDA;
        if (M > (1ll << 30) || N > (1ll << 30) || M * N > (1ll << 46)) return FP4_ERR_UNSUPPORTED;
        int dev;
        DeviceInfo *info;
        fp4_status st = device_info(dev, info);
        if (st != FP4_OK) return st;
        // D = epilogue(bias): the split-K reduce with no partials
        const int64_t blocks = std::min<int64_t>(cdiv(M * d_cols, 256), static_cast<int64_t>(info->sms) * 8);
        splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            nullptr, D, M, N, d_cols, 0, 0, alpha, out == FP4_OUT_BF16, bias, act);
        return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
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

    const bool mx = fmt == FP4_FMT_MXFP4;
    const int vec = mx ? 32 : 16;
    const int64_t ksf = K / vec;
    const int64_t kc4 = cdiv(ksf, 4);
    bool gemv = false;
    if ((st = choose_gemv(M, K, mx, prepacked, cfg, (reinterpret_cast<uintptr_t>(sfB) & 1u) == 0, gemv)) != FP4_OK) return st;
    if (gemv) {
        // M <= 4: the CUDA-core kernel streams B once, reading the scales in
        // either layout in place (no reorder, no scratch)
        GemvParams g;
        std::memset(&g, 0, sizeof g);
        g.A = static_cast<const uint8_t *>(A);
        g.sfA = static_cast<const uint8_t *>(sfA);
        g.B = static_cast<const uint8_t *>(B);
        g.sfB = static_cast<const uint8_t *>(sfB);
        g.D = D;
        g.ldd = d_cols;
        g.M = static_cast<int32_t>(M);
        g.N = static_cast<int32_t>(N);
        g.K = static_cast<int32_t>(K);
        g.mx = mx;
        g.atoms = prepacked ? 1 : 0;
        g.bf16 = out == FP4_OUT_BF16;
        g.act = act;
        g.alpha = alpha;
        g.bias = bias;
        return launch_gemv(g, info->sms, stream) == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
    }
    const bool rows_ok = (d_cols * esize) % 16 == 0;
    Plan plan;
    st = make_plan(M, N, K, rows_ok, mx, info->sms, cfg, plan);
    if (st != FP4_OK) return st;

    const int64_t rows_a = plan.swap ? N : M, rows_b = plan.swap ? M : N;
    const void *op_a = plan.swap ? B : A, *op_b = plan.swap ? A : B;
    const void *sf_a = plan.swap ? sfB : sfA, *sf_b = plan.swap ? sfA : sfB;

    // scratch: reordered scales and split-K partials (stream-ordered)
    const int64_t rb_a = cdiv(rows_a, 128), rb_b = cdiv(rows_b, 128);
    const size_t atoms_a = static_cast<size_t>(rb_a * kc4 * kAtomBytes);
    const size_t atoms_b = static_cast<size_t>(rb_b * kc4 * kAtomBytes);
    const size_t atom_bytes = prepacked ? 0 : atoms_a + atoms_b;
    // With caller-given scratch (the static array), fewer K splits where the
    // partials would not fit: only the atoms themselves are a hard limit.
    if (ext_scratch)
        while (plan.splits > 1 && atom_bytes + static_cast<size_t>(plan.splits) * rows_a * rows_b * 4 > ext_bytes)
            --plan.splits;
    const size_t ws_bytes = plan.splits > 1 ? static_cast<size_t>(plan.splits) * rows_a * rows_b * 4 : 0;
    size_t scratch_bytes = atom_bytes + ws_bytes;

    // Split tail (direct mode): when the last wave of tiles fills at most half of
    // the resident CTA groups, each of its tiles runs as two K halves on two
    // groups, so the wave ends after about half a tile.
    const int64_t tiles = cdiv(rows_a, kBM * plan.cg) * cdiv(rows_b, plan.bn);
    const int64_t k_tiles = cdiv(K, kBK);
    int64_t tail = 0;
    // The split tail runs only when asked for (it measured slower than whole
    // tiles on every shape where it applied: 4096^3 44.1 against 39.9 us,
    // 512 x 14336 x 4096 32.1 against 26.8, 8192^3 fp32 214.1 against 212.6).
    if (cfg && cfg->split_tail == 1 && !plan.swap && plan.splits == 1 && k_tiles >= 2) {
        int slots = 0;
        Maps none;
        Args none_args;
        std::memset(&none, 0, sizeof none);
        std::memset(&none_args, 0, sizeof none_args);
        if (launch_by_cfg(plan.cg, plan.bn, mx, *info, 0, plan.cap, none, none_args, stream, &slots) != cudaSuccess)
            return FP4_ERR_CUDA;
        const int64_t t = tiles % std::max(slots, 1);
        if (t > 0 && 2 * t <= slots) tail = t;
    }
    const size_t tail_ws_bytes = static_cast<size_t>(tail) * plan.cg * plan.bn * kBM * 4;
    const size_t tail_flag_bytes = static_cast<size_t>(tail) * plan.cg * kEpiWarps * 8;
    if (tail && ext_scratch && scratch_bytes + tail_ws_bytes + tail_flag_bytes > ext_bytes) tail = 0;
    const size_t tail_off = scratch_bytes;
    if (tail) scratch_bytes += tail_ws_bytes + tail_flag_bytes;
    uint8_t *scratch = nullptr;
    if (ext_scratch) {
        if (scratch_bytes > ext_bytes) return FP4_ERR_SCRATCH_LIMIT;
        scratch = ext_scratch;
    } else if (scratch_bytes) {
        if (cudaMallocAsync(reinterpret_cast<void **>(&scratch), scratch_bytes, stream) != cudaSuccess)
            return FP4_ERR_CUDA;
    }
    fp4_status result = FP4_OK;
    do {
        // A split-tail flag only ever matches its own launch's epoch, which a
        // plain call never repeats. A captured call's epoch is replayed with the
        // graph, so the flags a replay left behind would already match: zero them
        // first (ahead of the reorder, which the GEMM follows as a dependent launch).
        if (tail && stream_capturing(stream) &&
            cudaMemsetAsync(scratch + tail_off + tail_ws_bytes, 0, tail_flag_bytes, stream) != cudaSuccess) {
            result = FP4_ERR_CUDA;
            break;
        }
        const uint8_t *sfa_atoms = static_cast<const uint8_t *>(sf_a);
        const uint8_t *sfb_atoms = static_cast<const uint8_t *>(sf_b);
        uint8_t *ws = scratch + (prepacked ? 0 : atoms_a + atoms_b);
        if (!prepacked) {
            ReorderSpec ra, rbs;
            ra.sf = sf_a, ra.out = scratch, ra.rows = rows_a;
            rbs.sf = sf_b, rbs.out = scratch + atoms_a, rbs.rows = rows_b;
            if ((result = reorder2_launch(ra, rbs, ksf, info->sms, stream)) != FP4_OK) break;
            sfa_atoms = scratch;
            sfb_atoms = scratch + atoms_a;
        }
        const int apk = mx ? 2 : 4;
        const int nrb = static_cast<int>(cdiv(plan.bn, 128));
        Maps m;
        std::memset(&m, 0, sizeof m);
        if (!encode_operand(&m.a, op_a, rows_a, K, kBM) || !encode_operand(&m.b, op_b, rows_b, K, plan.bn / plan.cg) ||
            !encode_scales(&m.sfa, sfa_atoms, rb_a, kc4, apk, 1) ||
            !encode_scales(&m.sfb, sfb_atoms, rb_b, kc4, apk, nrb)) {
            result = FP4_ERR_CUDA;
            break;
        }
        Args a;
        std::memset(&a, 0, sizeof a);
        a.wait_ns = wait_limit_ns();
        a.rows_a = static_cast<int32_t>(rows_a);
        a.rows_b = static_cast<int32_t>(rows_b);
        a.k_tiles = static_cast<int32_t>(cdiv(K, kBK));
        a.kps = static_cast<int32_t>(cdiv(a.k_tiles, plan.splits));
        a.splits = static_cast<int32_t>(cdiv(a.k_tiles, a.kps));   // no empty split
        a.tiles_a = static_cast<int32_t>(cdiv(rows_a, kBM * plan.cg));
        a.tiles_b = static_cast<int32_t>(cdiv(rows_b, plan.bn));
        a.units = a.tiles_a * a.tiles_b * a.splits + static_cast<int32_t>(tail);
        a.split_units = static_cast<int32_t>(2 * tail);
        a.kh = static_cast<int32_t>(k_tiles / 2);
        if (tail) {
            a.tail_ws = reinterpret_cast<float *>(scratch + tail_off);
            a.tail_flags = reinterpret_cast<unsigned long long *>(scratch + tail_off + tail_ws_bytes);
        }
        a.epoch = next_epoch();
        a.stop_after = cfg ? std::max(0, cfg->stop_after) : 0;
        // Groups of 8 slot-B tiles keep the tiles in flight about square (a wave
        // of 76 pairs spans ~9 x 8 tiles); a slot-A operand of 16 MiB or more
        // would be read again from DRAM for every group, so it gets groups of 32
        // (8192^3 NVFP4 fp32 220.2 -> 217.2 us, 8192 x 14336 x 4096 188.8 -> 186.6;
        // with 8 MiB, 2048 x 28672 x 8192, 32 was slower: 173.3 -> 178.0).
        const bool big_a = static_cast<int64_t>(rows_a) * (K / 2) >= (int64_t(16) << 20);
        a.group_b = std::max(1, std::min(a.tiles_b, big_a ? 32 : 8));
        a.bf16 = out == FP4_OUT_BF16;
        a.alpha = alpha;
        a.act = act;
        a.bias = bias;
        if (!plan.swap) {
            a.mode = kEpiRows;
            a.out = D;
            a.ldo = d_cols;
            a.st32 = (reinterpret_cast<uintptr_t>(D) & 31u) == 0 && (d_cols * esize) % 32 == 0;
            // CTA pairs store D with TMA boxes where the tensor map allows it (16-byte
            // aligned base and row pitch); otherwise with the direct stores.
            if (plan.cg == 2 && aligned16(D) && (d_cols * esize) % 16 == 0 &&
                encode_output(&m.d, D, M, d_cols, out == FP4_OUT_BF16))
                a.tma_d = 1;
        } else if (a.splits > 1) {
            a.mode = kEpiSplitK;
            a.out = ws;
            a.ldo = rows_a;
            a.split_stride = rows_a * rows_b;
        } else {
            a.mode = kEpiTransposed;
            a.out = D;
            a.ldo = d_cols;
            // CTA pairs store D^T with TMA boxes where the tensor map allows it
            // (SwiGLU keeps the direct stores: its gate/up pairs meet across lanes)
            if (plan.cg == 2 && act != FP4_ACT_SWIGLU && aligned16(D) && (d_cols * esize) % 16 == 0 &&
                encode_output_t(&m.d, D, M, d_cols, out == FP4_OUT_BF16))
                a.tma_d = 1;
        }
        if (launch_by_cfg(plan.cg, plan.bn, mx, *info, a.units, plan.cap, m, a, stream) != cudaSuccess) {
            result = FP4_ERR_CUDA;
            break;
        }
        if (a.mode == kEpiSplitK) {
            const int64_t total = rows_a * rows_b;
            const int64_t blocks = std::min<int64_t>(cdiv(total, 256), static_cast<int64_t>(info->sms) * 8);
            splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
                reinterpret_cast<const float *>(ws), D, rows_b, rows_a, d_cols, a.splits, a.split_stride, alpha,
                a.bf16, bias, act);
            if (cudaGetLastError() != cudaSuccess) {
                result = FP4_ERR_CUDA;
                break;
            }
        }
    } while (false);
    if (scratch && !ext_scratch && cudaFreeAsync(scratch, stream) != cudaSuccess && result == FP4_OK)
        result = FP4_ERR_CUDA;
    return result;
}

// Grouped GEMM: one persistent launch over every group's tiles (GroupGeo).
fp4_status grouped_impl(fp4_format fmt, int prepacked, int64_t G, const int64_t *offsets, const void *A,
                        const void *sfA, const void *B, const void *sfB, float alpha, const fp4_epilogue *epi,
                        void *D, int64_t N, int64_t K, fp4_out_dtype out, const fp4_gemm_config *cfg,
                        cudaStream_t stream)
{
    if (fmt != FP4_FMT_NVFP4 && fmt != FP4_FMT_MXFP4) return FP4_ERR_INVALID_ARG;
    if (out != FP4_OUT_F32 && out != FP4_OUT_BF16) return FP4_ERR_INVALID_ARG;
    const int act = epi ? epi->act : FP4_ACT_NONE;
    const float *bias = epi ? epi->bias : nullptr;
    if (act < FP4_ACT_NONE || act > FP4_ACT_SWIGLU) return FP4_ERR_INVALID_ARG;
    if (G < 0 || N < 0 || K < 0) return FP4_ERR_INVALID_ARG;
    if (G == 0) return FP4_OK;
    if (!offsets || offsets[0] != 0) return FP4_ERR_INVALID_ARG;
    if (G > kMaxGroups) return FP4_ERR_UNSUPPORTED;
    int64_t max_rows = 0;
    for (int64_t g = 0; g < G; ++g) {
        if (offsets[g + 1] < offsets[g]) return FP4_ERR_INVALID_ARG;
        max_rows = std::max(max_rows, offsets[g + 1] - offsets[g]);
    }
    const int64_t M = offsets[G];
    const bool glu = act == FP4_ACT_SWIGLU;
    if (glu && N % 2 != 0) return FP4_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FP4_OK;
    if (!D) return FP4_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(bias) & 3u) return FP4_ERR_MISALIGNED;
    const int mode = cfg ? cfg->mode : 0;
    if (mode < 0 || mode > 2) return FP4_ERR_INVALID_ARG;
    if (cfg && (cfg->bn || cfg->splits > 1 || cfg->cta_group || cfg->max_ctas)) return FP4_ERR_UNSUPPORTED;
    const int64_t esize = out == FP4_OUT_BF16 ? 2 : 4;
    const int64_t d_cols = glu ? N / 2 : N;
    if (K == 0) {
        if (!aligned16(D)) return FP4_ERR_MISALIGNED;
        if (act == FP4_ACT_NONE && !bias)
            return cudaMemsetAsync(D, 0, static_cast<size_t>(M * d_cols * esize), stream) == cudaSuccess
                       ? FP4_OK
                       : FP4_ERR_CUDA;
        if (M > (1ll << 30) || G * N > (1ll << 30)) return FP4_ERR_UNSUPPORTED;
        int dev;
        DeviceInfo *info;
        const fp4_status st = device_info(dev, info);
        if (st != FP4_OK) return st;
        // D = epilogue(bias of the row's group), group by group (the split-K reduce with no partials)
        for (int64_t g = 0; g < G; ++g) {
            const int64_t m = offsets[g + 1] - offsets[g];
            if (m == 0) continue;
            const int64_t blocks = std::min<int64_t>(cdiv(m * d_cols, 256), static_cast<int64_t>(info->sms) * 8);
            splitk_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
                nullptr, static_cast<uint8_t *>(D) + offsets[g] * d_cols * esize, m, N, d_cols, 0, 0, alpha,
                out == FP4_OUT_BF16, bias ? bias + g * N : nullptr, act);
            if (cudaGetLastError() != cudaSuccess) return FP4_ERR_CUDA;
        }
        return FP4_OK;
    }
    if (!A || !B || !sfA || !sfB) return FP4_ERR_INVALID_ARG;
    if (K % 32 != 0) return FP4_ERR_UNSUPPORTED;
    if (M > (1ll << 30) || G * N > (1ll << 30) || K > (1ll << 30) || M * N > (1ll << 46)) return FP4_ERR_UNSUPPORTED;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D)) return FP4_ERR_MISALIGNED;
    if (prepacked & ~3) return FP4_ERR_INVALID_ARG;
    const bool b_pre = prepacked & FP4_GROUPED_B_ATOMS, a_pre = prepacked & FP4_GROUPED_A_ATOMS;
    if ((b_pre && !aligned16(sfB)) || (a_pre && !aligned16(sfA))) return FP4_ERR_MISALIGNED;

    int dev;
    DeviceInfo *info;
    fp4_status st = device_info(dev, info);
    if (st != FP4_OK) return st;
    const bool mx = fmt == FP4_FMT_MXFP4;
    const int vec = mx ? 32 : 16;
    const int64_t ksf = K / vec, kc4 = cdiv(ksf, 4);
    const bool rows_ok = (d_cols * esize) % 16 == 0;
    const bool swap = mode == 2 || (mode == 0 && (max_rows <= 256 || !rows_ok));
    if (!swap && !rows_ok) return FP4_ERR_MISALIGNED;
    // swap-AB: one CTA per 128 weight rows, a group's rows in N tiles of BN (one
    // tile when every group fits); direct: CTA pairs, N tiles of 256
    const int bn = swap ? std::max(64, pow2_bn(std::min<int64_t>(max_rows, 256))) : 256;
    const int cg = swap ? 1 : 2;
    const int nrb = static_cast<int>(cdiv(bn, 128));
    const int64_t nb = cdiv(N, 128);                 // scale blocks of one B_g

    // The groups' geometry (kernel parameters) and the row map of A's scale
    // reorder (each group's rows start a fresh 128-row block)
    GroupParams gp;
    RowBlocks a_map;
    std::memset(&gp, 0, sizeof gp);
    std::memset(&a_map, 0, sizeof a_map);
    gp.count = static_cast<int32_t>(G);
    a_map.groups = static_cast<int32_t>(G);
    int64_t units = 0, a_nblk = 0;
    for (int64_t g = 0; g < G; ++g) {
        const int64_t m = offsets[g + 1] - offsets[g];
        a_map.first_blk[g] = static_cast<int32_t>(a_nblk);
        a_map.row0[g] = static_cast<int32_t>(offsets[g]);
        GroupGeo &q = gp.g[g];
        q.first = static_cast<int32_t>(units);
        q.bias_off = static_cast<int32_t>(g * N);
        if (swap) {
            q.tiles_a = static_cast<int32_t>(cdiv(N, 128));
            q.oa = static_cast<int32_t>(g * N), q.sa = static_cast<int32_t>(g * nb), q.da = 0,
            q.la = static_cast<int32_t>(N);
            q.ob = static_cast<int32_t>(offsets[g]), q.sb = static_cast<int32_t>(a_nblk),
            q.db = static_cast<int32_t>(offsets[g]), q.lb = static_cast<int32_t>(m);
            units += q.tiles_a * cdiv(m, bn);
        } else {
            q.tiles_a = static_cast<int32_t>(cdiv(m, 128 * cg));
            q.oa = static_cast<int32_t>(offsets[g]), q.sa = static_cast<int32_t>(a_nblk),
            q.da = static_cast<int32_t>(offsets[g]), q.la = static_cast<int32_t>(m);
            q.ob = static_cast<int32_t>(g * N), q.sb = static_cast<int32_t>(g * nb), q.db = 0,
            q.lb = static_cast<int32_t>(N);
            units += q.tiles_a * cdiv(N, bn);
        }
        if (q.tiles_a == 0) q.tiles_a = 1;        // (an empty group owns no unit)
        a_nblk += cdiv(m, 128);
    }
    a_map.first_blk[G] = static_cast<int32_t>(a_nblk);
    a_map.row0[G] = static_cast<int32_t>(M);
    if (units > (1ll << 30)) return FP4_ERR_UNSUPPORTED;
    RowBlocks b_map;
    std::memset(&b_map, 0, sizeof b_map);
    b_map.groups = static_cast<int32_t>(G);
    b_map.uniform = static_cast<int32_t>(N);

    // scratch (stream-ordered): the reordered scales, 256-byte aligned
    auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    const size_t atoms_a = a_pre ? 0 : static_cast<size_t>(a_nblk * kc4 * kAtomBytes);
    const size_t atoms_b = b_pre ? 0 : static_cast<size_t>(G * nb * kc4 * kAtomBytes);
    const size_t off_b = up(atoms_a);
    uint8_t *scratch = nullptr;
    if (atoms_a + atoms_b > 0 &&
        cudaMallocAsync(reinterpret_cast<void **>(&scratch), off_b + atoms_b, stream) != cudaSuccess)
        return FP4_ERR_CUDA;
    fp4_status result = FP4_OK;
    do {
        const uint8_t *a_atoms = static_cast<const uint8_t *>(sfA);
        const uint8_t *b_atoms = static_cast<const uint8_t *>(sfB);
        {
            ReorderSpec ra, rbs;                      // both in one launch
            if (!a_pre) {
                ra.sf = sfA, ra.out = scratch, ra.rows = M, ra.row_blocks = a_nblk, ra.rbm = &a_map;
                a_atoms = scratch;
            }
            if (!b_pre) {
                rbs.sf = sfB, rbs.out = scratch + off_b, rbs.rows = G * N, rbs.row_blocks = G * nb, rbs.rbm = &b_map;
                b_atoms = scratch + off_b;
            }
            if ((result = reorder2_launch(ra, rbs, ksf, info->sms, stream)) != FP4_OK) break;
        }
        const int apk = mx ? 2 : 4;
        Maps m;
        std::memset(&m, 0, sizeof m);
        const bool ok = swap ? (encode_operand(&m.a, B, G * N, K, kBM) && encode_operand(&m.b, A, M, K, bn) &&
                                encode_scales(&m.sfa, b_atoms, G * nb, kc4, apk, 1) &&
                                encode_scales(&m.sfb, a_atoms, a_nblk, kc4, apk, nrb))
                             : (encode_operand(&m.a, A, M, K, kBM) && encode_operand(&m.b, B, G * N, K, bn / cg) &&
                                encode_scales(&m.sfa, a_atoms, a_nblk, kc4, apk, 1) &&
                                encode_scales(&m.sfb, b_atoms, G * nb, kc4, apk, nrb));
        if (!ok) {
            result = FP4_ERR_CUDA;
            break;
        }
        Args a;
        std::memset(&a, 0, sizeof a);
        a.wait_ns = wait_limit_ns();
        a.rows_a = static_cast<int32_t>(swap ? N : M);
        a.rows_b = static_cast<int32_t>(swap ? M : N);
        a.k_tiles = static_cast<int32_t>(cdiv(K, kBK));
        a.kps = a.k_tiles;
        a.splits = 1;
        a.tiles_a = a.tiles_b = 1;
        a.units = static_cast<int32_t>(units);
        a.group_b = 1;
        a.bf16 = out == FP4_OUT_BF16;
        a.mode = swap ? kEpiTransposed : kEpiRows;
        a.st32 = (reinterpret_cast<uintptr_t>(D) & 31u) == 0 && (d_cols * esize) % 32 == 0;
        a.act = act;
        a.alpha = alpha;
        a.bias = bias;
        a.out = D;
        a.ldo = d_cols;
        a.split_units = 0;
        a.epoch = next_epoch();
        if (units > 0 &&
            launch_grouped(cg, bn, mx, *info, static_cast<int>(units), m, a, gp, stream) != cudaSuccess)
            result = FP4_ERR_CUDA;
    } while (false);
    if (scratch && cudaFreeAsync(scratch, stream) != cudaSuccess && result == FP4_OK) result = FP4_ERR_CUDA;
    return result;
}

// Device address of g_static_scratch on device `dev`, looked up once per
// device (with that device current) and kept.
uint8_t *g_static_scratch_addr[64] = {};

fp4_status static_scratch_address(int dev, uint8_t **out)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_static_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return FP4_ERR_CUDA;
        g_static_scratch_addr[dev] = static_cast<uint8_t *>(p);
    }
    *out = g_static_scratch_addr[dev];
    return FP4_OK;
}

}  // namespace

// Shared with the quantiser's translation unit (fp4_quant.cu): the limit of
// its bounded waits, and its device status word (read and cleared), which
// fp4_get_device_status reports too.
uint64_t library_wait_limit_ns() { return wait_limit_ns(); }
int quant_take_device_status();
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

fp4_status fp4_gemm_plan(fp4_format fmt, int scales_prepacked, int64_t M, int64_t N, int64_t K, fp4_out_dtype out,
                         int32_t act, const fp4_gemm_config *cfg, fp4_plan_info *info)
{
    if (!info) return FP4_ERR_INVALID_ARG;
    std::memset(info, 0, sizeof *info);
    if (fmt != FP4_FMT_NVFP4 && fmt != FP4_FMT_MXFP4) return FP4_ERR_INVALID_ARG;
    if (out != FP4_OUT_F32 && out != FP4_OUT_BF16) return FP4_ERR_INVALID_ARG;
    if (act < FP4_ACT_NONE || act > FP4_ACT_SWIGLU) return FP4_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return FP4_ERR_INVALID_ARG;
    if (act == FP4_ACT_SWIGLU && N % 2 != 0) return FP4_ERR_UNSUPPORTED;
    if (K % 32 != 0) return FP4_ERR_UNSUPPORTED;
    if (M == 0 || N == 0 || K == 0) return FP4_OK;      // no GEMM kernel (K == 0: a fill)
    int dev;
    DeviceInfo *di;
    fp4_status st = device_info(dev, di);
    if (st != FP4_OK) return st;
    const bool mx = fmt == FP4_FMT_MXFP4;
    bool gemv = false;
    if ((st = choose_gemv(M, K, mx, scales_prepacked, cfg, true, gemv)) != FP4_OK) return st;
    if (gemv) {
        info->kernel = 1;
        info->launches = 1;
        return FP4_OK;
    }
    const int64_t esize = out == FP4_OUT_BF16 ? 2 : 4;
    const int64_t d_cols = act == FP4_ACT_SWIGLU ? N / 2 : N;
    Plan plan;
    if ((st = make_plan(M, N, K, (d_cols * esize) % 16 == 0, mx, di->sms, cfg, plan)) != FP4_OK) return st;
    info->swap = plan.swap;
    info->bn = plan.bn;
    info->cta_group = plan.cg;
    info->splits = static_cast<int32_t>(cdiv(cdiv(K, kBK), cdiv(cdiv(K, kBK), plan.splits)));
    info->launches = (scales_prepacked ? 0 : 1) + 1 + (info->splits > 1 ? 1 : 0);
    return FP4_OK;
}

fp4_status fp4_gemm_grouped(fp4_format fmt, int weights_prepacked, int64_t G, const int64_t *offsets,
                            const void *A, const void *sfA, const void *B, const void *sfB, float alpha,
                            const fp4_epilogue *epi, void *D, int64_t N, int64_t K, fp4_out_dtype out,
                            const fp4_gemm_config *cfg, cudaStream_t stream)
{
    return grouped_impl(fmt, weights_prepacked, G, offsets, A, sfA, B, sfB, alpha, epi, D, N, K, out, cfg, stream);
}

size_t fp4_scale_atom_bytes_grouped(int64_t G, const int64_t *offsets, int64_t k, int vec)
{
    if (G < 0 || k < 0 || (vec != 16 && vec != 32) || k % vec != 0 || (G > 0 && !offsets)) return 0;
    int64_t blocks = 0;
    for (int64_t g = 0; g < G; ++g) {
        if (offsets[g + 1] < offsets[g]) return 0;
        blocks += cdiv(offsets[g + 1] - offsets[g], 128);
    }
    return static_cast<size_t>(blocks * cdiv(k / vec, 4) * kAtomBytes);
}

fp4_status fp4_scale_reorder_grouped(const void *sf_plain, void *sf_atom, int64_t G, const int64_t *offsets,
                                     int64_t k, int vec, cudaStream_t stream)
{
    if (G < 0 || k < 0 || (vec != 16 && vec != 32)) return FP4_ERR_INVALID_ARG;
    if (k % vec != 0) return FP4_ERR_UNSUPPORTED;
    if (G == 0 || k == 0) return FP4_OK;
    if (!offsets || offsets[0] != 0) return FP4_ERR_INVALID_ARG;
    if (G > kMaxGroups) return FP4_ERR_UNSUPPORTED;
    RowBlocks map;
    std::memset(&map, 0, sizeof map);
    map.groups = static_cast<int32_t>(G);
    int64_t blocks = 0;
    for (int64_t g = 0; g < G; ++g) {
        if (offsets[g + 1] < offsets[g]) return FP4_ERR_INVALID_ARG;
        map.first_blk[g] = static_cast<int32_t>(blocks);
        map.row0[g] = static_cast<int32_t>(offsets[g]);
        blocks += cdiv(offsets[g + 1] - offsets[g], 128);
    }
    if (offsets[G] > (1ll << 30)) return FP4_ERR_UNSUPPORTED;
    map.first_blk[G] = static_cast<int32_t>(blocks);
    map.row0[G] = static_cast<int32_t>(offsets[G]);
    if (blocks == 0) return FP4_OK;
    if (!sf_plain || !sf_atom) return FP4_ERR_INVALID_ARG;
    if (!aligned16(sf_atom)) return FP4_ERR_MISALIGNED;
    int dev;
    DeviceInfo *info;
    const fp4_status st = device_info(dev, info);
    if (st != FP4_OK) return st;
    return reorder_launch(sf_plain, sf_atom, offsets[G], k / vec, info->sms, stream, blocks, &map);
}

fp4_status fp4_gemm_fused(fp4_format fmt, int scales_prepacked, const void *A, const void *sfA, const void *B,
                          const void *sfB, float alpha, const fp4_epilogue *epi, void *D, int64_t M, int64_t N,
                          int64_t K, fp4_out_dtype out, const fp4_gemm_config *cfg, cudaStream_t stream)
{
    return gemm_impl(fmt, scales_prepacked, A, sfA, B, sfB, alpha, D, M, N, K, out, cfg, stream, nullptr, 0, epi);
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

fp4_status fp4_gemm_static_scratch(fp4_format fmt, const void *A, const void *sfA, const void *B,
                                   const void *sfB, float alpha, void *D, int64_t M, int64_t N, int64_t K,
                                   fp4_out_dtype out, cudaStream_t stream)
{
    int dev;
    DeviceInfo *info;
    fp4_status st = device_info(dev, info);
    if (st != FP4_OK) return st;
    uint8_t *scratch = nullptr;
    if ((st = static_scratch_address(dev, &scratch)) != FP4_OK) return st;
    return gemm_impl(fmt, 0, A, sfA, B, sfB, alpha, D, M, N, K, out, nullptr, stream, scratch,
                     kStaticScratchBytes);
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
    return reorder_launch(sf_plain, sf_atom, rows, k / vec, info->sms, stream);
}

fp4_status fp4_scale_reorder2(const void *sf_a, void *atoms_a, int64_t rows_a, const void *sf_b, void *atoms_b,
                              int64_t rows_b, int64_t k, int vec, cudaStream_t stream)
{
    if (rows_a < 0 || rows_b < 0 || k < 0 || (vec != 16 && vec != 32)) return FP4_ERR_INVALID_ARG;
    if (k % vec != 0) return FP4_ERR_UNSUPPORTED;
    if (k == 0 || (rows_a == 0 && rows_b == 0)) return FP4_OK;
    if ((rows_a && (!sf_a || !atoms_a)) || (rows_b && (!sf_b || !atoms_b))) return FP4_ERR_INVALID_ARG;
    if ((rows_a && !aligned16(atoms_a)) || (rows_b && !aligned16(atoms_b))) return FP4_ERR_MISALIGNED;
    int dev;
    DeviceInfo *info;
    const fp4_status st = device_info(dev, info);
    if (st != FP4_OK) return st;
    ReorderSpec a, b;
    if (rows_a) a.sf = sf_a, a.out = atoms_a, a.rows = rows_a;
    if (rows_b) b.sf = sf_b, b.out = atoms_b, b.rows = rows_b;
    return reorder2_launch(a, b, k / vec, info->sms, stream);
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
    const int q = fp4::quant_take_device_status();   // the quantiser's word, cleared too
    return static_cast<fp4_status>(v != 0 ? v : q);
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
    case FP4_ERR_SCRATCH_LIMIT: return "problem needs more than the 16 MiB static scratch array";
    default: return "unknown status";
    }
}

void fp4_set_wait_limit_ms(int64_t ms)
{
    std::lock_guard<std::mutex> lk(g_mu);
    g_wait_ms = ms < 1 ? 1 : ms;
}

}  // extern "C"
