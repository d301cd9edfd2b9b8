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

#include <type_traits>

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

// 1.5 * 2^23: for |y| < 2^22, y + kRound lies in [2^23, 2^24), where the float spacing is 1, so
// the addition itself rounds y to an integer, ties to even, and that integer sits in the low
// mantissa bits: (y + kRound) - kRound == rint(y) exactly, and for |rint(y)| <= 127 the low byte
// of the sum's bit pattern is the code as an int8. This replaces a float-to-integer conversion
// (a quarter-rate instruction) per element.
constexpr float kRound = 12582912.0f;

// The codes of 8 values: RN-even of y = RN(v * RN(1/s)) unless one of them lies within 3e-5 of a
// half-integer (or the row's scale is subnormal: `exact`), then of the correctly rounded quotient
// for all 8, clamped to +-127. With a normal scale no clamp is needed: s = RN(max|a| / 127) and
// three roundings keep |y| below 127 (1 + 2^-24)^3 < 127.5, and |v / s| below 127 (1 + 2^-24).
// Adds the chunk's code sum to `sum`; writes the f16 copies (H16) and the int8 bytes (Q8).
template <bool H16, bool Q8>
__device__ __forceinline__ void quantize8(const float (&v)[8], float s, float rcp, bool exact, int& sum, uint4& h16,
                                          uint2& q8) {
    float t[8];   // kRound + code
    float dev = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float y = __fmul_rn(v[j], rcp);   // no contraction: y is the rounded product
        t[j] = __fadd_rn(y, kRound);
        dev = fmaxf(dev, fabsf(__fsub_rn(y, __fsub_rn(t[j], kRound))));   // distance to rint(y), <= 0.5
    }
    if (exact || dev > 0.49997f) {   // near a half-integer: decide by the exact quotient
#pragma unroll
        for (int j = 0; j < 8; ++j) t[j] = __fadd_rn(fminf(fmaxf(rintf(__fdiv_rn(v[j], s)), -127.f), 127.f), kRound);
    }
    float r[8];
    float cs = 0.f;   // the chunk's code sum, exact (|cs| <= 1016)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        r[j] = __fsub_rn(t[j], kRound);
        cs += r[j];
    }
    sum += __float2int_rn(cs);
    if constexpr (H16) {
        uint32_t hw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 h = __floats2half2_rn(r[2 * j], r[2 * j + 1]);   // integers <= 127: exact
            hw[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        h16 = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
    if constexpr (Q8) {
        uint32_t b[2];
#pragma unroll
        for (int w = 0; w < 2; ++w) {   // byte 0 of each of the four t's bit patterns
            const uint32_t lo = __byte_perm(__float_as_uint(t[4 * w]), __float_as_uint(t[4 * w + 1]), 0x0040u);
            const uint32_t hi = __byte_perm(__float_as_uint(t[4 * w + 2]), __float_as_uint(t[4 * w + 3]), 0x0040u);
            b[w] = __byte_perm(lo, hi, 0x5410u);
        }
        q8 = make_uint2(b[0], b[1]);
    }
}

// One block per row. The row is read once: each thread keeps up to kCache chunks of 8 values as
// raw bits in registers between the max pass and the quantize pass (K <= 4096), all requested
// before the first is used; longer rows re-read the rest. Raw 16-bit words keep the register
// count at 40 for 16-bit activations (6 blocks per SM; measured at 2048 x 4096 bf16: 9.4 us, against
// 9.6 us with float values cached at 48 registers and 9.7 us when held to 32 registers).
template <int ADT>
struct Raw8 {   // 8 activations as stored
    static constexpr int kWords = ADT == DT_F32 ? 8 : 4;
    uint32_t w[kWords];
    __device__ __forceinline__ void load(const void* A, size_t i) {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(A) + i * (ADT == DT_F32 ? 4 : 2));
        const uint4 x = __ldcs(p);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        if constexpr (ADT == DT_F32) {
            const uint4 y = __ldcs(p + 1);
            w[4] = y.x; w[5] = y.y; w[6] = y.z; w[7] = y.w;
        }
    }
    __device__ __forceinline__ void values(float (&v)[8]) const {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if constexpr (ADT == DT_F32) v[j] = __uint_as_float(w[j]);
            else if constexpr (ADT == DT_BF16) v[j] = __uint_as_float((j & 1) ? (w[j >> 1] & 0xFFFF0000u) : (w[j >> 1] << 16));
            else v[j] = __half2float(__ushort_as_half((unsigned short)(w[j >> 1] >> (16 * (j & 1)))));
        }
    }
};

template <int ADT, bool H16, bool Q8>
__global__ void __launch_bounds__(kThreads, ADT == DT_F32 ? 4 : 6) act_quant_kernel(
    int K, const void* __restrict__ A, int8_t* __restrict__ qa, __half* __restrict__ qa16, float* __restrict__ as,
    int32_t* __restrict__ rowsum) {
    constexpr int kCache = 2;
    __shared__ float s_max[kThreads / 32];
    __shared__ int s_sum[kThreads / 32];
    const int m = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t row = (size_t)m * K;

    Raw8<ADT> c[kCache];
#pragma unroll
    for (int i = 0; i < kCache; ++i) {
        const int k = (threadIdx.x + i * kThreads) * 8;
        if (k < K) c[i].load(A, row + k);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kCache; ++i) {
        if ((threadIdx.x + i * kThreads) * 8 < K) {
            float v[8];
            c[i].values(v);
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
        }
    }
    for (int k = (threadIdx.x + kCache * kThreads) * 8; k < K; k += kThreads * 8) {
        Raw8<ADT> x;
        float v[8];
        x.load(A, row + k);
        x.values(v);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
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
    auto emit = [&](int k, const float (&v)[8]) {
        uint4 h16;
        uint2 q8;
        quantize8<H16, Q8>(v, s, rcp, exact, sum, h16, q8);
        if constexpr (H16) *reinterpret_cast<uint4*>(qa16 + row + k) = h16;
        if constexpr (Q8) *reinterpret_cast<uint2*>(qa + row + k) = q8;
    };
#pragma unroll
    for (int i = 0; i < kCache; ++i) {
        const int k = (threadIdx.x + i * kThreads) * 8;
        if (k < K) {
            float v[8];
            c[i].values(v);
            emit(k, v);
        }
    }
    for (int k = (threadIdx.x + kCache * kThreads) * 8; k < K; k += kThreads * 8) {
        Raw8<ADT> x;
        float v[8];
        x.load(A, row + k);
        x.values(v);
        emit(k, v);
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

// The next layer's activation step on a layer output C whose row maxima are already known per
// 128-channel tile (the tensor-core epilogue wrote them): one block per row takes the max of its
// tile maxima and quantizes the row in a single read, with the arithmetic of act_quant_kernel, so
// the codes are the ones act_quant_kernel would give for C.
template <int CDT>
__global__ void __launch_bounds__(kThreads) quant_rows_kernel(int N, const void* __restrict__ C,
                                                              const float* __restrict__ rowmax, int ntiles, int M,
                                                              __half* __restrict__ qa16, float* __restrict__ as,
                                                              int32_t* __restrict__ rowsum) {
    __shared__ int s_sum[kThreads / 32];
    const int m = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t row = (size_t)m * N;
    float amax = 0.f;
    for (int t = lane; t < ntiles; t += 32) amax = fmaxf(amax, __ldg(rowmax + (size_t)t * M + m));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = __fdiv_rn(amax, 127.0f);
    const bool exact = s != 0.f && s < 1.17549435e-38f;
    const float rcp = (s != 0.f && !exact) ? __frcp_rn(s) : 0.f;
    int sum = 0;
    // two chunks per thread and step, both requested before either is quantized
    for (int k0 = threadIdx.x * 8; k0 < N; k0 += 2 * kThreads * 8) {
        const int k1 = k0 + kThreads * 8;
        float v0[8], v1[8];
        load8<CDT>(C, row + k0, v0);
        if (k1 < N) load8<CDT>(C, row + k1, v1);
        uint4 h16;
        uint2 q8;
        quantize8<true, false>(v0, s, rcp, exact, sum, h16, q8);
        *reinterpret_cast<uint4*>(qa16 + row + k0) = h16;
        if (k1 < N) {
            quantize8<true, false>(v1, s, rcp, exact, sum, h16, q8);
            *reinterpret_cast<uint4*>(qa16 + row + k1) = h16;
        }
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

cudaError_t launch_quant_rows(int M, int N, const void* C, int c_dtype, const float* rowmax, int ntiles,
                              void* qa16, float* as, int32_t* rowsum, cudaStream_t s) {
    __half* h = static_cast<__half*>(qa16);
    if (c_dtype == DT_F32)
        quant_rows_kernel<DT_F32><<<M, kThreads, 0, s>>>(N, C, rowmax, ntiles, M, h, as, rowsum);
    else if (c_dtype == DT_F16)
        quant_rows_kernel<DT_F16><<<M, kThreads, 0, s>>>(N, C, rowmax, ntiles, M, h, as, rowsum);
    else
        quant_rows_kernel<DT_BF16><<<M, kThreads, 0, s>>>(N, C, rowmax, ntiles, M, h, as, rowsum);
    return cudaGetLastError();
}

cudaError_t launch_act_quant(int M, int K, const void* A, int a_dtype, int8_t* qa, void* qa16, float* as,
                             int32_t* rowsum, cudaStream_t s) {
    __half* h = static_cast<__half*>(qa16);
    auto go = [&](auto adt) {
        constexpr int ADT = decltype(adt)::value;
        if (qa && h)
            act_quant_kernel<ADT, true, true><<<M, kThreads, 0, s>>>(K, A, qa, h, as, rowsum);
        else if (h)
            act_quant_kernel<ADT, true, false><<<M, kThreads, 0, s>>>(K, A, qa, h, as, rowsum);
        else
            act_quant_kernel<ADT, false, true><<<M, kThreads, 0, s>>>(K, A, qa, h, as, rowsum);
    };
    if (a_dtype == DT_F32)
        go(std::integral_constant<int, DT_F32>{});
    else if (a_dtype == DT_F16)
        go(std::integral_constant<int, DT_F16>{});
    else
        go(std::integral_constant<int, DT_BF16>{});
    return cudaGetLastError();
}

}  // namespace qg
