// The epilogue fused into every output store: C = act(acc + bias) + residual, in float32, then
// one rounding to C's type. The pull request "vulkan: 在骁龙 8 Gen 3（Adreno 750，安卓）上跑通并调优
// 无协作矩阵档" keeps a GEMM's accumulators in float32 until bias, residual and activation have
// been applied (its note on the DIRECT build's fp16 shared tiles); the order (activation, then
// residual) and the activations offered (ReLU, SiLU, tanh-form GELU) are this library's reading.
// Split-K partial sums never see it: the reduction that adds the splits applies it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace qg {

__device__ __forceinline__ float act_apply(int act, float v) {
    switch (act) {
        case ACT_RELU: return fmaxf(v, 0.f);
        case ACT_SILU: return v / (1.f + expf(-v));   // v * sigmoid(v)
        case ACT_GELU_TANH: {
            // tanh form of GELU: 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))
            const float u = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
            return 0.5f * v * (1.f + tanhf(u));
        }
        default: return v;
    }
}

template <int CDT>
__device__ __forceinline__ float load_c(const void* p, size_t i) {
    if constexpr (CDT == DT_F32) return __ldg(static_cast<const float*>(p) + i);
    else if constexpr (CDT == DT_F16) return __half2float(__ldg(static_cast<const __half*>(p) + i));
    else return __bfloat162float(__ldg(static_cast<const __nv_bfloat16*>(p) + i));
}

// v: the float32 result of output (m, n), mn = m * N + n (in range).
template <int CDT>
__device__ __forceinline__ float epilogue_apply(const Epilogue& e, float v, size_t mn, int n) {
    if (e.bias) v += __ldg(e.bias + n);
    v = act_apply(e.act, v);
    if (e.residual) v += load_c<CDT>(e.residual, mn);
    return v;
}

}  // namespace qg
