// epilogue.cuh -- the fused epilogue's element functions (fp4_gemm_fused),
// shared by the tcgen05 GEMM and the narrow-M kernel.
#pragma once

#include "fp4_gemm.h"

namespace fp4 {

// silu(x) = x / (1 + e^-x) in fp32 (expf and an IEEE division); -0 for x below
// about -88, where e^-x overflows.
__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

// ReLU or squared ReLU of one element (SwiGLU pairs two elements and is done
// by the callers); FP4_ACT_NONE passes z through.
__device__ __forceinline__ float activate(float z, int act)
{
    if (act == FP4_ACT_RELU) return fmaxf(z, 0.0f);
    if (act == FP4_ACT_RELU2) {
        const float r = fmaxf(z, 0.0f);
        return r * r;
    }
    return z;
}

}  // namespace fp4
