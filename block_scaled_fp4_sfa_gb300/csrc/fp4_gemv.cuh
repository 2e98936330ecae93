// fp4_gemv.cuh -- internal interface between the GEMM front end (fp4_gemm.cu)
// and the narrow-M kernel (fp4_gemv.cu). Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace fp4 {

// Largest M the narrow kernel takes; above it the tcgen05 GEMM runs.
constexpr int kGemvMaxM = 4;

struct GemvParams {
    const uint8_t *A;      // [M][K/2] codes
    const uint8_t *sfA;    // plain [M][K/vec] or 128x4 atoms
    const uint8_t *B;      // [N][K/2] codes
    const uint8_t *sfB;    // plain [N][K/vec] or 128x4 atoms
    void *D;               // [M][ldd]
    int64_t ldd;           // D row pitch in elements (N, or N/2 for SwiGLU)
    int32_t M, N, K;
    int32_t mx;            // 0: NVFP4 (E4M3 per 16), 1: MXFP4 (E8M0 per 32)
    int32_t atoms;         // scales in the atom layout (both operands)
    int32_t bf16;          // output type
    int32_t act;           // fp4_activation
    float alpha;
    const float *bias;     // NULL or N floats
};

// Shared memory one CTA needs for K (0 if K is beyond what the kernel stages).
size_t gemv_smem_bytes(int64_t M, int64_t K, bool mx);

// Launches the narrow-M kernel on `stream` (M in 1..kGemvMaxM).
cudaError_t launch_gemv(const GemvParams &p, int sms, cudaStream_t stream);

}  // namespace fp4
