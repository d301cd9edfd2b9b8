// W4A8 activation step: dynamic per-row symmetric INT8 quantization of A.
//
// Benchmark page "MNN GemmSpeed 基准测试实战", «测试用例与注册机制»: the W4A8 path quantizes the
// activations dynamically to INT8. Per row, in float32: as = max|a| / 127, qa = clamp(rint(a / as),
// -127, 127) with ties to even (qa = 0 when as == 0), rowsum = sum qa. The codes equal those of
// the correctly rounded IEEE quotient bit for bit. The quotient itself is not needed, only the
// integer it rounds to, so each element first uses y = a * RN(1 / as): for |a / as| <= 127 it is
// within 2.3e-5 of RN(a / as), hence rounds to the same integer unless it lies within 3e-5 of a
// half-integer; only those rare elements take the exact division. A row whose scale is below the
// smallest normal float32 (max|a| < 127 * 2^-126) takes the exact division for every element:
// RN(1 / as) can overflow there (to +inf below 2^-128), and the error bound above assumes a
// normal reciprocal.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace qg {
namespace {

constexpr int kThreads = 256;

// 8 consecutive activations as float32
template <int ADT>
__device__ __forceinline__ void load8(const void* A, size_t i, float (&v)[8]) {
    if constexpr (ADT == DT_F32) {
        const float4 x = *reinterpret_cast<const float4*>(static_cast<const float*>(A) + i);
        const float4 y = *reinterpret_cast<const float4*>(static_cast<const float*>(A) + i + 4);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w; v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
    } else {
        const uint4 x = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(A) + i);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (ADT == DT_BF16) {
                v[2 * j] = __uint_as_float(w[j] << 16);
                v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            } else {
                v[2 * j] = __half2float(__ushort_as_half((unsigned short)(w[j] & 0xFFFFu)));
                v[2 * j + 1] = __half2float(__ushort_as_half((unsigned short)(w[j] >> 16)));
            }
        }
    }
}

// The codes of 8 values: RN-even of v * RN(1/s) unless one of them lies within 3e-5 of a
// half-integer (or the row's scale is subnormal: `exact`), then of the correctly rounded quotient
// for all 8; clamped to +-127 (as rounded floats, exact); the f16 copies, the int8 bytes and the
// running sum of the codes.
__device__ __forceinline__ void quantize8(const float (&v)[8], float s, float rcp, bool exact, int& sum, uint4& h16,
                                          uint2& q8) {
    float r[8];
    float dev = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float y = v[j] * rcp;
        r[j] = rintf(y);
        dev = fmaxf(dev, fabsf(y - r[j]));   // distance to the nearest integer, <= 0.5
    }
    if (exact || dev > 0.49997f) {   // near a half-integer: decide by the exact quotient
#pragma unroll
        for (int j = 0; j < 8; ++j) r[j] = rintf(__fdiv_rn(v[j], s));
    }
    uint32_t hw[4];
    float cs = 0.f;   // the chunk's code sum, exact (|cs| <= 1016)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        r[j] = fminf(fmaxf(r[j], -127.f), 127.f);
        cs += r[j];
    }
    sum += __float2int_rn(cs);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __half2 h = __floats2half2_rn(r[2 * j], r[2 * j + 1]);   // integers <= 127: exact
        hw[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    h16 = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    uint32_t b[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j >> 2] |= ((uint32_t)__float2int_rn(r[j]) & 0xFFu) << (8 * (j & 3));
    q8 = make_uint2(b[0], b[1]);
}

// One block per row. The row is read once: each thread keeps up to kCache chunks of 8 values in
// registers between the max pass and the quantize pass (K <= 8192); longer rows re-read the rest.
template <int ADT>
__global__ void __launch_bounds__(kThreads) act_quant_kernel(int K, const void* __restrict__ A,
                                                             int8_t* __restrict__ qa, __half* __restrict__ qa16,
                                                             float* __restrict__ as, int32_t* __restrict__ rowsum) {
    constexpr int kCache = 4;
    __shared__ float s_max[kThreads / 32];
    __shared__ int s_sum[kThreads / 32];
    const int m = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t row = (size_t)m * K;

    float v[kCache][8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kCache; ++i) {
        const int k = (threadIdx.x + i * kThreads) * 8;
        if (k < K) {
            load8<ADT>(A, row + k, v[i]);
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
        }
    }
    for (int k = (threadIdx.x + kCache * kThreads) * 8; k < K; k += kThreads * 8) {
        float w[8];
        load8<ADT>(A, row + k, w);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(w[j]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) s_max[warp] = amax;
    __syncthreads();
    amax = s_max[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, s_max[w]);
    const float s = __fdiv_rn(amax, 127.0f);
    // s == 0: every code is 0. A subnormal s (its reciprocal may overflow) divides exactly.
    const bool exact = s != 0.f && s < 1.17549435e-38f;
    const float rcp = (s != 0.f && !exact) ? __frcp_rn(s) : 0.f;

    int sum = 0;
    auto emit = [&](int k, const float (&w)[8]) {
        uint4 h16;
        uint2 q8;
        quantize8(w, s, rcp, exact, sum, h16, q8);
        if (qa16) *reinterpret_cast<uint4*>(qa16 + row + k) = h16;
        if (qa) *reinterpret_cast<uint2*>(qa + row + k) = q8;
    };
#pragma unroll
    for (int i = 0; i < kCache; ++i) {
        const int k = (threadIdx.x + i * kThreads) * 8;
        if (k < K) emit(k, v[i]);
    }
    for (int k = (threadIdx.x + kCache * kThreads) * 8; k < K; k += kThreads * 8) {
        float w[8];
        load8<ADT>(A, row + k, w);
        emit(k, w);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) s_sum[warp] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int total = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) total += s_sum[w];
        as[m] = s;
        rowsum[m] = total;
    }
}

// Row sums of A in float32 (the Int8-Block0 tensor-core path's offset term o * sum_k a): one
// warp per row, 8 consecutive values per lane and step (16-byte loads), a shuffle reduction.
template <int ADT>
__global__ void __launch_bounds__(kThreads) row_sum_kernel(int M, int K, const void* __restrict__ A,
                                                           float* __restrict__ out) {
    const int m = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (m >= M) return;
    float acc = 0.f;
    for (int k = lane * 8; k < K; k += 32 * 8) {
        float v[8];
        load8<ADT>(A, (size_t)m * K + k, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc += v[j];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) out[m] = acc;
}

}  // namespace

cudaError_t launch_row_sums(int M, int K, const void* A, int a_dtype, float* out, cudaStream_t s) {
    const int blocks = (M + kThreads / 32 - 1) / (kThreads / 32);
    if (a_dtype == DT_F32)
        row_sum_kernel<DT_F32><<<blocks, kThreads, 0, s>>>(M, K, A, out);
    else if (a_dtype == DT_F16)
        row_sum_kernel<DT_F16><<<blocks, kThreads, 0, s>>>(M, K, A, out);
    else
        row_sum_kernel<DT_BF16><<<blocks, kThreads, 0, s>>>(M, K, A, out);
    return cudaGetLastError();
}

cudaError_t launch_act_quant(int M, int K, const void* A, int a_dtype, int8_t* qa, void* qa16, float* as,
                             int32_t* rowsum, cudaStream_t s) {
    __half* h = static_cast<__half*>(qa16);
    if (a_dtype == DT_F32)
        act_quant_kernel<DT_F32><<<M, kThreads, 0, s>>>(K, A, qa, h, as, rowsum);
    else if (a_dtype == DT_F16)
        act_quant_kernel<DT_F16><<<M, kThreads, 0, s>>>(K, A, qa, h, as, rowsum);
    else
        act_quant_kernel<DT_BF16><<<M, kThreads, 0, s>>>(K, A, qa, h, as, rowsum);
    return cudaGetLastError();
}

}  // namespace qg
