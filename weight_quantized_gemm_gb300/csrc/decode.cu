// Decode path (small M) host logic: K-split choice, 16-row launches, the fixed-order split-K
// reduction (also used by the tensor-core path), and the exact float32 CUDA-core kernel (float32
// activations, any M). The tensor-core weight-streaming kernels are in decode_stream.cuh (TMA-fed)
// and decode_kernel.cuh (the other shapes).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_stream.cuh"

namespace qg {

cudaError_t launch_decode_int4(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_int8(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_float(const DecodeArgs& a, cudaStream_t s);

namespace {

using dec::store_out;
using dec::Share;

template <int CDT>
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int splits, size_t count, int N, Epilogue ep,
                                     void* C) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count; i += (size_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int y = 0; y < splits; ++y) s += partial[(size_t)y * count + i];
        store_out<CDT>(C, i, epilogue_apply<CDT>(ep, s, i, ep.bias ? (int)(i % (size_t)N) : 0));
    }
}

// ---------------------------------------------------------------- exact float32 kernel
template <int ADT>
__device__ __forceinline__ float load_a(const void* A, size_t i) {
    if constexpr (ADT == DT_F32) return static_cast<const float*>(A)[i];
    else if constexpr (ADT == DT_F16) return __half2float(static_cast<const __half*>(A)[i]);
    else return __bfloat162float(static_cast<const __nv_bfloat16*>(A)[i]);
}

// One warp per output channel and group of 4 rows of A; lanes stride over 16-byte pieces of the
// weight row, dequantize each weight once in float32 (w = q * s + o, one rounding) and
// accumulate a * w in float32; the 32 lane partials are summed with warp shuffles.
template <int FMT, int ADT, int WDT, int CDT>
__global__ void __launch_bounds__(256) decode_f32_kernel(DecodeArgs p) {
    constexpr int kRowsM = 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = blockIdx.x * 8 + warp;
    if (n >= p.N) return;
    const int K = p.K;
    const int nb = K / p.block;
    // elements per 16-byte piece
    constexpr int kPer = FMT == FMT_INT4 ? 32 : (FMT == FMT_INT8 ? 16 : (WDT == DT_F32 ? 4 : 8));
    const int pieces = K / kPer;
    const uint8_t* row = static_cast<const uint8_t*>(p.Bp) + (size_t)n * pieces * 16;
    for (int m0 = blockIdx.y * kRowsM; m0 < p.M; m0 += gridDim.y * kRowsM) {
    float acc[kRowsM] = {0.f, 0.f, 0.f, 0.f};
    for (int pc = lane; pc < pieces; pc += 32) {
        const uint4 raw = *reinterpret_cast<const uint4*>(row + (size_t)pc * 16);
        const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
        const int k0 = pc * kPer;
        float s = 1.f, o = 0.f;
        if constexpr (FMT != FMT_FLOAT) {
            const int blk = k0 / p.block;
            o = p.T[tab_index(n, nb, blk) * 2 + 0];
            s = p.T[tab_index(n, nb, blk) * 2 + 1];
        }
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            float w;
            if constexpr (FMT == FMT_INT4) {
                w = fmaf((float)((wd[e >> 3] >> (4 * (e & 7))) & 15u), s, o);
            } else if constexpr (FMT == FMT_INT8) {
                w = fmaf((float)((wd[e >> 2] >> (8 * (e & 3))) & 255u), s, o);
            } else if constexpr (WDT == DT_F32) {
                w = __uint_as_float(wd[e]);
            } else if constexpr (WDT == DT_F16) {
                w = __half2float(__ushort_as_half((unsigned short)(wd[e >> 1] >> (16 * (e & 1)))));
            } else {
                w = __uint_as_float(((wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16);
            }
#pragma unroll
            for (int r = 0; r < kRowsM; ++r)
                if (m0 + r < p.M) acc[r] = fmaf(load_a<ADT>(p.A, (size_t)(m0 + r) * K + k0 + e), w, acc[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsM; ++r) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kRowsM; ++r)
            if (m0 + r < p.M) {
                const size_t mn = (size_t)(m0 + r) * p.N + n;
                store_out<CDT>(p.C, mn, epilogue_apply<CDT>(p.ep, acc[r], mn, n));
            }
    }
    }
}

template <int FMT, int ADT, int WDT>
cudaError_t launch_f32_c(const DecodeArgs& a, cudaStream_t s) {
    dim3 grid((a.N + 7) / 8, (a.M + 3) / 4 < 65535 ? (a.M + 3) / 4 : 65535);
    switch (a.c_dtype) {
        case DT_F32: decode_f32_kernel<FMT, ADT, WDT, DT_F32><<<grid, 256, 0, s>>>(a); break;
        case DT_F16: decode_f32_kernel<FMT, ADT, WDT, DT_F16><<<grid, 256, 0, s>>>(a); break;
        default: decode_f32_kernel<FMT, ADT, WDT, DT_BF16><<<grid, 256, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

template <int ADT>
cudaError_t launch_f32_a(const DecodeArgs& a, cudaStream_t s) {
    if (a.fmt == FMT_INT4) return launch_f32_c<FMT_INT4, ADT, ADT>(a, s);
    if (a.fmt == FMT_INT8) return launch_f32_c<FMT_INT8, ADT, ADT>(a, s);
    return launch_f32_c<FMT_FLOAT, ADT, ADT>(a, s);   // float-mode weights share A's dtype
}

}  // namespace

int decode_splits(int M, int K, int N, int fmt, int block) {
    // K-range per thread block: 64 sub-blocks for the TMA-fed kernel (and the cp.async kernel at
    // M <= 8), 32 for the cp.async kernel at 9 <= M <= 16, so that the activations fit in
    // registers or shared memory; split further while the units alone cannot give every SM a
    // thread block, keeping at least one sub-block per warp.
    const int nsb = K / 64;
    const int sb_max = (dstream::stream_takes(M, K, fmt, block) || M <= 8) ? Share<1>::kSbMaxNt : Share<2>::kSbMaxNt;
    int splits = (nsb + sb_max - 1) / sb_max;
    const int groups = (N + 15) / 16;
    while (groups * splits < kTargetSms && nsb / (splits * 2) >= dec::kWarps) splits *= 2;
    return splits;
}

static cudaError_t launch_one(const DecodeArgs& a, cudaStream_t s) {
    if (a.fmt == FMT_INT4) return launch_decode_int4(a, s);
    if (a.fmt == FMT_INT8) return launch_decode_int8(a, s);
    return launch_decode_float(a, s);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    // The kernel takes at most 16 rows of A; larger M runs as consecutive 16-row launches.
    const size_t esz = dt_size(a.a_dtype), csz = dt_size(a.c_dtype);
    for (int m0 = 0; m0 < a.M; m0 += 16) {
        DecodeArgs c = a;
        c.M = a.M - m0 < 16 ? a.M - m0 : 16;
        c.A = static_cast<const uint8_t*>(a.A) + (size_t)m0 * a.K * esz;
        c.C = static_cast<uint8_t*>(a.C) + (size_t)m0 * a.N * csz;
        if (a.ep.residual) c.ep.residual = static_cast<const uint8_t*>(a.ep.residual) + (size_t)m0 * a.N * csz;
        c.splits = decode_splits(c.M, a.K, a.N, a.fmt, a.block);
        cudaError_t e = launch_one(c, s);
        if (e != cudaSuccess || c.splits <= 1) {
            if (e != cudaSuccess) return e;
            continue;
        }
        e = launch_splitk_reduce(c.partial, c.splits, (size_t)c.M * c.N, c.N, c.ep, c.C, c.c_dtype, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_splitk_reduce(const float* partial, int splits, size_t count, int N, const Epilogue& ep, void* C,
                                 int c_dtype, cudaStream_t s) {
    const int threads = 256;
    const size_t want = (count + threads - 1) / threads;
    const int blocks = (int)(want < 4096 ? want : 4096);
    switch (c_dtype) {
        case DT_F32: splitk_reduce_kernel<DT_F32><<<blocks, threads, 0, s>>>(partial, splits, count, N, ep, C); break;
        case DT_F16: splitk_reduce_kernel<DT_F16><<<blocks, threads, 0, s>>>(partial, splits, count, N, ep, C); break;
        default: splitk_reduce_kernel<DT_BF16><<<blocks, threads, 0, s>>>(partial, splits, count, N, ep, C); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_f32(const DecodeArgs& a, cudaStream_t s) {
    if (a.a_dtype == DT_F32) return launch_f32_a<DT_F32>(a, s);
    if (a.a_dtype == DT_F16) return launch_f32_a<DT_F16>(a, s);
    return launch_f32_a<DT_BF16>(a, s);
}

}  // namespace qg
