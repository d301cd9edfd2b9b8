// Weight preparation: asymmetric block quantization + packing, and the float-mode copy.
//
// Quantization follows the benchmark page "MNN GemmSpeed 基准测试实战", section
// «为什么用 Conv1x1 来测 GEMM» (asymmetric, one [offset, scale] pair per output channel and
// K-block, oc x blockNum pairs), with the min/max scheme: every decision is taken in float32
// with explicitly rounded intrinsics (no contraction), so the codes are bit-identical to any
// IEEE float32 evaluation of  q = clamp(rint((w - lo) / ((hi - lo) / qmax)), 0, qmax).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace qg {
namespace {

constexpr int kCh = 32;      // output channels per block (one warp lane each)
constexpr int kRows = 8;     // warps per block, striding over K
constexpr int kChunk = 64;   // K-chunk staged in shared memory before packing

// grid: (ceil(N / 32), K / block); block: 256 threads = 32 channels x 8 K-strides.
template <int NBITS>
__global__ void __launch_bounds__(256) quant_pack_kernel(const float* __restrict__ W, int K, int N, int block,
                                                         uint8_t* __restrict__ Bp, float* __restrict__ T) {
    constexpr int kQmax = NBITS == 4 ? 15 : 255;
    __shared__ float s_lo[kRows][kCh], s_hi[kRows][kCh];
    __shared__ uint8_t s_code[kCh][kChunk + 4];

    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int n0 = blockIdx.x * kCh;
    const int n = n0 + tx;
    const int nc = n < N ? n : N - 1;   // clamp the column read; results of n >= N are dropped
    const int b = blockIdx.y;
    const int nb = K / block;
    const int k0 = b * block;

    // 1) group min / max (exact, order independent)
    float lo = W[(size_t)(k0 + ty) * N + nc], hi = lo;
    for (int k = k0 + ty + kRows; k < k0 + block; k += kRows) {
        const float w = W[(size_t)k * N + nc];
        lo = w < lo ? w : lo;
        hi = w > hi ? w : hi;
    }
    s_lo[ty][tx] = lo;
    s_hi[ty][tx] = hi;
    __syncthreads();
    lo = s_lo[0][tx];
    hi = s_hi[0][tx];
#pragma unroll
    for (int r = 1; r < kRows; ++r) {
        lo = s_lo[r][tx] < lo ? s_lo[r][tx] : lo;
        hi = s_hi[r][tx] > hi ? s_hi[r][tx] : hi;
    }
    // 2) scale and offset
    const float scale = __fdiv_rn(__fsub_rn(hi, lo), (float)kQmax);
    if (ty == 0 && n < (N + 15) / 16 * 16) {   // channels past N fill their 16-channel group with zeros
        T[tab_index(n, nb, b) * 2 + 0] = n < N ? lo : 0.f;
        T[tab_index(n, nb, b) * 2 + 1] = n < N ? scale : 0.f;
    }
    // 3) codes, a K-chunk at a time, then packed rows written along K
    constexpr int kBytesPerRow = kChunk * NBITS / 8;       // 32 or 64
    constexpr int kWordsPerRow = kBytesPerRow / 4;         // 8 or 16
    const size_t row_bytes = (size_t)K * NBITS / 8;
    for (int kc = k0; kc < k0 + block; kc += kChunk) {
#pragma unroll
        for (int kk = ty; kk < kChunk; kk += kRows) {
            int code = 0;
            if (scale != 0.0f) {
                const float w = W[(size_t)(kc + kk) * N + nc];
                const float u = __fdiv_rn(__fsub_rn(w, lo), scale);
                code = __float2int_rn(u);   // round half to even
                code = code < 0 ? 0 : (code > kQmax ? kQmax : code);
            }
            s_code[tx][kk] = (uint8_t)code;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kCh * kWordsPerRow; i += blockDim.x) {
            const int r = i / kWordsPerRow, wd = i % kWordsPerRow;
            if (n0 + r >= N) continue;
            uint32_t word = 0;
            if (NBITS == 4) {
#pragma unroll
                for (int j = 0; j < 8; ++j) word |= (uint32_t)s_code[r][wd * 8 + j] << (4 * j);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) word |= (uint32_t)s_code[r][wd * 4 + j] << (8 * j);
            }
            uint8_t* dst = Bp + (size_t)(n0 + r) * row_bytes + (size_t)(kc - 0) * NBITS / 8 + wd * 4;
            *reinterpret_cast<uint32_t*>(dst) = word;
        }
        __syncthreads();
    }
}

// Float mode: transpose W [K][N] -> [N][K] and round to the storage dtype (nearest even).
template <typename T>
__device__ __forceinline__ T cvt_store(float x);
template <>
__device__ __forceinline__ float cvt_store<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half cvt_store<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt_store<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T>
__global__ void __launch_bounds__(256) float_pack_kernel(const float* __restrict__ W, int K, int N,
                                                         T* __restrict__ out) {
    __shared__ float tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int n0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int k = k0 + ty + 8 * i, n = n0 + tx;
        if (k < K && n < N) tile[ty + 8 * i][tx] = W[(size_t)k * N + n];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int n = n0 + ty + 8 * i, k = k0 + tx;
        if (k < K && n < N) out[(size_t)n * K + k] = cvt_store<T>(tile[tx][ty + 8 * i]);
    }
}

}  // namespace

cudaError_t launch_quant_pack(const float* W, int K, int N, int block, int nbits, uint8_t* Bp, float* T,
                              cudaStream_t s) {
    dim3 grid((N + kCh - 1) / kCh, K / block);
    if (nbits == 4)
        quant_pack_kernel<4><<<grid, 256, 0, s>>>(W, K, N, block, Bp, T);
    else
        quant_pack_kernel<8><<<grid, 256, 0, s>>>(W, K, N, block, Bp, T);
    return cudaGetLastError();
}

cudaError_t launch_float_pack(const float* W, int K, int N, int w_dtype, void* Bp, cudaStream_t s) {
    dim3 grid((N + 31) / 32, (K + 31) / 32);
    if (w_dtype == DT_F16)
        float_pack_kernel<__half><<<grid, 256, 0, s>>>(W, K, N, static_cast<__half*>(Bp));
    else if (w_dtype == DT_BF16)
        float_pack_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(W, K, N, static_cast<__nv_bfloat16*>(Bp));
    else
        float_pack_kernel<float><<<grid, 256, 0, s>>>(W, K, N, static_cast<float*>(Bp));
    return cudaGetLastError();
}

}  // namespace qg
