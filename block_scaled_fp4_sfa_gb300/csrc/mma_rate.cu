// Micro-benchmark: the issue rate of dense block-scaled FP4 MMAs on this GPU.
//
// One thread per CTA (the leader of the pair for cta_group::2) issues the
// K = 64 `tcgen05.mma ... kind::mxf4nvf4.block_scale` of 4096 k-tiles (four MMAs
// of K = 64 each, one per 256-element k-tile) back to back, from operand tiles
// already in shared memory and scale factors already in TMEM, on every SM at
// once. Clock64 and the global timer around the loop give cycles per k-tile and
// the SM clock. Modes:
//   0  MMAs only (the tensor pipe's own rate)
//   1  before each k-tile's MMAs, the same thread copies that k-tile's scale
//      atoms from shared memory to TMEM (`tcgen05.cp .32x128b.warpx4`, one per
//      atom): the cost of staging scales through the tensor pipe
//   2  MMAs + one `tcgen05.commit` per k-tile (how a pipeline stage is released)
// Operand bytes are arbitrary E2M1 pairs; every scale is 1.0 (UE4M3 0x38 for
// NVFP4, UE8M0 0x7F for MXFP4). Results are not read back: only the timing is.
//
// Built and run by `python -m block_scaled_fp4_sfa_gb300.mma_rate`; prints one
// line per case.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "ptx.cuh"

using namespace fp4;

namespace {

constexpr int kKtiles = 4096;
constexpr int kThreads = 128;
constexpr int kSmem = 200 * 1024;   // one CTA per SM

__device__ bool wait_bounded(uint32_t bar, uint32_t parity)
{
    for (long it = 0; it < 200000000L; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

template <int CG, int N, bool MX, int MODE>
__global__ void __launch_bounds__(kThreads, 1) mma_rate_kernel(unsigned long long *cycles, unsigned long long *ns,
                                                               int *err)
{
    constexpr int APK = MX ? 2 : 4;                 // scale atoms per k-tile per 128 rows
    constexpr int NRB = (N + 127) / 128;
    constexpr int A_BYTES = 128 * 128;
    constexpr int B_BYTES = (N / CG) * 128;
    constexpr int SFA_BYTES = APK * 512, SFB_BYTES = NRB * APK * 512;
    constexpr int OFF_A = 0, OFF_B = A_BYTES, OFF_SFA = OFF_B + B_BYTES, OFF_SFB = OFF_SFA + SFA_BYTES,
                  OFF_BAR = OFF_SFB + SFB_BYTES;
    static_assert(OFF_BAR + 64 + 1024 <= kSmem, "shared memory");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *bp = smem_raw + (base - raw);
    const uint32_t bar_done = base + OFF_BAR, bar_step = bar_done + 8;
    uint32_t *holder = reinterpret_cast<uint32_t *>(bp + OFF_BAR + 32);
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;

    for (int i = threadIdx.x; i < OFF_SFA; i += blockDim.x) bp[i] = static_cast<uint8_t>((i * 2654435761u) >> 13);
    for (int i = OFF_SFA + threadIdx.x; i < OFF_BAR; i += blockDim.x) bp[i] = MX ? 0x7F : 0x38;
    if (threadIdx.x == 0) {
        mbar_init(bar_done, 1);
        mbar_init(bar_step, 1);
        fence_mbarrier_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor-core reads
    if (threadIdx.x / 32 == 1) {
        tmem_alloc<CG>(smem_u32(holder), 512);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    const uint32_t sf = tmem + 256;                 // scale columns after the accumulator
    const uint64_t dsa = smem_desc(base + OFF_SFA, 0, 128, 0);
    const uint64_t dsb = smem_desc(base + OFF_SFB, 0, 128, 0);
    auto copies = [&]() {
#pragma unroll
        for (int t = 0; t < APK; ++t) {
            tc_cp_32x128b_warpx4<CG>(sf + 4 * t, dsa + (t * 512 >> 4));
#pragma unroll
            for (int rb = 0; rb < NRB; ++rb)
                tc_cp_32x128b_warpx4<CG>(sf + 4 * APK + 4 * (t * NRB + rb), dsb + ((rb * APK + t) * 512 >> 4));
        }
    };
    if (threadIdx.x == 0 && rank == 0) {
        constexpr uint32_t ID0 = idesc_fp4(128 * CG, N, MX, 0, 0);
        constexpr uint32_t ID2 = idesc_fp4(128 * CG, N, MX, 2, 2);
        const uint64_t da = smem_desc(base + OFF_A, 16, 1024, 2);
        const uint64_t db = smem_desc(base + OFF_B, 16, 1024, 2);
        bool ok = true;
        if (MODE != 1) {                            // scales staged once
            copies();
            tc_commit<CG>(bar_step, 3);
            ok = wait_bounded(bar_step, 0);
            tc_fence_after();
        }
        const unsigned long long t0 = clock64();
        const uint64_t g0 = global_timer_ns();
        for (int kt = 0; ok && kt < kKtiles; ++kt) {
            if (MODE == 1) copies();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = MX ? (i >> 1) : i;
                tc_mma_fp4<CG, MX>(tmem, da + 2 * i, db + 2 * i, (MX && (i & 1)) ? ID2 : ID0, sf + 4 * t,
                                   sf + 4 * APK + 4 * NRB * t, (kt > 0 || i > 0) ? 1u : 0u);
            }
            if (MODE == 2) tc_commit<CG>(bar_step, 3);
        }
        tc_commit<CG>(bar_done, 3);
        if (!wait_bounded(bar_done, 0)) ok = false;
        const unsigned long long t1 = clock64();
        const uint64_t g1 = global_timer_ns();
        cycles[blockIdx.x] = t1 - t0;
        ns[blockIdx.x] = g1 - g0;
        if (!ok) atomicExch(err, 1);
    }
    tc_fence_before();
    if constexpr (CG == 2) cluster_sync(); else __syncthreads();
    tc_fence_after();
    if (threadIdx.x / 32 == 1) tmem_dealloc<CG>(tmem, 512);
}

template <int CG, int N, bool MX, int MODE>
int run(const char *name, int sms)
{
    auto k = mma_rate_kernel<CG, N, MX, MODE>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) return 1;
    const int ctas = CG == 2 ? sms & ~1 : sms;
    unsigned long long *cyc, *ns;
    int *err;
    cudaMalloc(&cyc, ctas * sizeof(unsigned long long));
    cudaMalloc(&ns, ctas * sizeof(unsigned long long));
    cudaMalloc(&err, sizeof(int));
    cudaMemset(cyc, 0, ctas * sizeof(unsigned long long));
    cudaMemset(ns, 0, ctas * sizeof(unsigned long long));
    cudaMemset(err, 0, sizeof(int));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    for (int rep = 0; rep < 2; ++rep)               // the first launch warms up
        if (cudaLaunchKernelEx(&cfg, k, cyc, ns, err) != cudaSuccess) return 1;
    if (cudaDeviceSynchronize() != cudaSuccess) return 1;
    unsigned long long hc[256] = {}, hn[256] = {};
    int herr = 0;
    cudaMemcpy(hc, cyc, ctas * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaMemcpy(hn, ns, ctas * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost);
    double c = 0, t = 0;
    int n = 0;
    for (int i = 0; i < ctas; i += CG) {
        c += static_cast<double>(hc[i]);
        t += static_cast<double>(hn[i]);
        ++n;
    }
    c /= n;
    t /= n;
    const double per_kt = c / kKtiles;
    const double mhz = c / t * 1e3;
    const double flop_cyc_sm = 2.0 * 128 * N * 256 / per_kt;          // per SM: 128 rows of the tile each
    printf("%-28s ctas=%3d err=%d  cycles/k-tile=%7.1f  cycles/MMA=%6.1f  SM MHz=%5.0f  FLOP/cycle/SM=%6.0f  "
           "whole-GPU TFLOP/s=%7.1f\n",
           name, ctas, herr, per_kt, per_kt / 4, mhz, flop_cyc_sm, flop_cyc_sm * ctas * mhz * 1e6 / 1e12);
    cudaFree(cyc);
    cudaFree(ns);
    cudaFree(err);
    return herr;
}

}  // namespace

int main()
{
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    if (sms > 256) sms = 256;
    int bad = 0;
    bad |= run<1, 256, false, 0>("cg1 128x256 NVFP4 MMA only", sms);
    bad |= run<1, 256, true, 0>("cg1 128x256 MXFP4 MMA only", sms);
    bad |= run<2, 256, false, 0>("cg2 256x256 NVFP4 MMA only", sms);
    bad |= run<2, 256, true, 0>("cg2 256x256 MXFP4 MMA only", sms);
    bad |= run<1, 128, false, 0>("cg1 128x128 NVFP4 MMA only", sms);
    bad |= run<1, 256, false, 2>("cg1 NVFP4 + commit/k-tile", sms);
    bad |= run<2, 256, false, 2>("cg2 NVFP4 + commit/k-tile", sms);
    bad |= run<1, 256, false, 1>("cg1 NVFP4 + 12 copies/k-tile", sms);
    bad |= run<2, 256, false, 1>("cg2 NVFP4 + 12 copies/k-tile", sms);
    bad |= run<1, 256, true, 1>("cg1 MXFP4 + 6 copies/k-tile", sms);
    bad |= run<2, 256, true, 1>("cg2 MXFP4 + 6 copies/k-tile", sms);
    return bad ? 1 : 0;
}
