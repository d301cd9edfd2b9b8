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

// The activations use the fast exponential (a few ulp) and the fast divide: the epilogue runs
// once per output on the few epilogue warps, and the results are rounded to C's type next.
__device__ __forceinline__ float act_apply(int act, float v) {
    switch (act) {
        case ACT_RELU: return fmaxf(v, 0.f);
        case ACT_SILU: return __fdividef(v, 1.f + __expf(-v));   // v * sigmoid(v)
        case ACT_GELU_TANH: {
            // tanh form of GELU, 0.5 v (1 + tanh(u)) with u = sqrt(2/pi) (v + 0.044715 v^3); as
            // 1 + tanh(u) = 2 - 2 / (1 + e^(2u)), this is v - v / (1 + e^(2u)), whose error is
            // absolute in v (no cancellation is amplified) and which is exact at both tails
            const float u = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
            return v - __fdividef(v, 1.f + __expf(2.f * u));
        }
        default: return v;
    }
}

// The same with the activation fixed at compile time (loops that hoist the choice).
template <int ACT>
__device__ __forceinline__ float act_fixed(float v) {
    if constexpr (ACT == ACT_RELU) return fmaxf(v, 0.f);
    else if constexpr (ACT == ACT_SILU) return __fdividef(v, 1.f + __expf(-v));
    else if constexpr (ACT == ACT_GELU_TANH) {
        const float u = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
        return v - __fdividef(v, 1.f + __expf(2.f * u));
    } else return v;
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
// Output type chosen at run time (kernels that store one value per output at their very end).
__device__ __forceinline__ void store_out_rt(void* C, size_t idx, float v, int cdt) {
    if (cdt == DT_F32) static_cast<float*>(C)[idx] = v;
    else if (cdt == DT_F16) static_cast<__half*>(C)[idx] = __float2half_rn(v);
    else static_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(v);
}
__device__ __forceinline__ float epilogue_apply_rt(const Epilogue& e, float v, size_t mn, int n, int cdt) {
    if (e.bias) v += __ldg(e.bias + n);
    v = act_apply(e.act, v);
    if (e.residual)
        v += cdt == DT_F32 ? load_c<DT_F32>(e.residual, mn)
                           : (cdt == DT_F16 ? load_c<DT_F16>(e.residual, mn) : load_c<DT_BF16>(e.residual, mn));
    return v;
}

}  // namespace qg
