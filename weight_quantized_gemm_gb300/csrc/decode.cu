// Decode path (small M): the weight stream.
//
// C[m][n] = sum_k A[m][k] * (q[n][k] * s[n][b(k)] + o[n][b(k)])   (benchmark page
// "MNN GemmSpeed 基准测试实战", «为什么用 Conv1x1 来测 GEMM»; at small M the layer is bound by
// the weight read, «几个可以直接读出的规律»).
//
// Per 64-element K sub-block the sum is regrouped as  s * sum_k a*q + o * sum_k a, so the
// 4/8-bit codes only need an exact conversion to 16-bit integers-valued floats in registers
// (q <= 255 is exact in f16 and bf16), and both sums come out of 16x8x16 tensor-core MMAs
// with float32 accumulation:
//   - the weights (16 output channels x 16 k) are the MMA's A operand, built in registers
//     from 64-bit (INT4) / 128-bit (INT8, float) streaming loads;
//   - the activations (k x up to 8 rows of A per MMA column tile) are the B operand;
//   - an A operand of all ones gives sum_k a in the same register layout.
// The int4 -> f16 conversion is the magic-number method of Kim et al., "Who Says Elephants
// Can't Run: Bringing Large Scale MoE Models into Cloud Scale Production" (2022): OR the nibble
// into the mantissa of 1024.0 and subtract 1024 (for bf16: 128.0). Because the MMA only sums
// over k, the order in which k values are assigned to MMA slots is free as long as weights
// and activations agree; the assignment below is the one that makes the conversion cheapest.
//
// Work split: a thread block owns 16 output channels; its 8 warps interleave over the 64-wide
// K sub-blocks (warp w takes sub-blocks w, w+8, ...) so that one step of the block reads a
// contiguous 8 x 32 B (INT4) run of every weight row. Warps then reduce through shared memory
// in a fixed order. When N is small, K is also split across thread blocks (gridDim.y) and a
// second kernel sums the float32 partials in a fixed order, so results are deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace qg {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
    return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t bfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// streaming loads (each weight byte is read exactly once)
__device__ __forceinline__ uint2 ldg_stream64(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ldg_stream128(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ldg128(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ float2 ldg_f2(const float* p) {
    float2 v;
    asm volatile("ld.global.nc.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

template <bool BF>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    if constexpr (BF) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// 8 nibbles n0..n7 (n_i = bits 4i..4i+3) -> 4 pairs of exact 16-bit values
// p[0] = (n0, n4), p[1] = (n1, n5), p[2] = (n2, n6), p[3] = (n3, n7)   [(low half, high half)]
template <bool BF>
__device__ __forceinline__ void int4_pairs(uint32_t w, uint32_t (&p)[4]) {
    if constexpr (!BF) {
        const uint32_t w8 = w >> 8;
        p[0] = hsub2(lop3_and_or(w, 0x000F000Fu, 0x64006400u), 0x64006400u);                // 1024+n - 1024
        p[1] = hfma2(lop3_and_or(w, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD400D400u);   // (1024+16n)/16 - 64
        p[2] = hsub2(lop3_and_or(w8, 0x000F000Fu, 0x64006400u), 0x64006400u);
        p[3] = hfma2(lop3_and_or(w8, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD400D400u);
    } else {
        p[0] = bfma2(lop3_and_or(w, 0x000F000Fu, 0x43004300u), 0x3F803F80u, 0xC300C300u);   // (128+n)*1 - 128
        p[1] = bfma2(lop3_and_or(w >> 4, 0x000F000Fu, 0x43004300u), 0x3F803F80u, 0xC300C300u);
        p[2] = bfma2(lop3_and_or(w >> 8, 0x000F000Fu, 0x43004300u), 0x3F803F80u, 0xC300C300u);
        p[3] = bfma2(lop3_and_or(w >> 12, 0x000F000Fu, 0x43004300u), 0x3F803F80u, 0xC300C300u);
    }
}

// 4 bytes b0..b3 -> 2 pairs of exact 16-bit values: p[0] = (b0, b1), p[1] = (b2, b3)
template <bool BF>
__device__ __forceinline__ void int8_pairs(uint32_t w, uint32_t (&p)[2]) {
    if constexpr (!BF) {
        p[0] = hsub2(prmt(w, 0x64646464u, 0x4140u), 0x64006400u);
        p[1] = hsub2(prmt(w, 0x64646464u, 0x4342u), 0x64006400u);
    } else {
        // 8-bit integers are exact in bf16 but too wide for the bf16 magic number: go through
        // the float32 magic number 2^23 and round the (exact) values to bf16.
        const float f0 = __uint_as_float(prmt(w, 0x4B000000u, 0x7540u)) - 8388608.0f;
        const float f1 = __uint_as_float(prmt(w, 0x4B000000u, 0x7541u)) - 8388608.0f;
        const float f2 = __uint_as_float(prmt(w, 0x4B000000u, 0x7542u)) - 8388608.0f;
        const float f3 = __uint_as_float(prmt(w, 0x4B000000u, 0x7543u)) - 8388608.0f;
        p[0] = pack_bf16x2(f0, f1);
        p[1] = pack_bf16x2(f2, f3);
    }
}

template <int CDT>
__device__ __forceinline__ void store_out(void* C, size_t idx, float v) {
    if constexpr (CDT == DT_F32)
        static_cast<float*>(C)[idx] = v;
    else if constexpr (CDT == DT_F16)
        static_cast<__half*>(C)[idx] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(v);
}

// One thread block: 16 output channels x (8 * NT) rows of A x one K-split.
//   FMT: weight format; BF: bf16 (else f16) operands; NT: 8-row MMA column tiles (1 or 2);
//   U: sub-blocks in flight per warp; PERCH: one table entry per channel (block == K).
template <int FMT, bool BF, int NT, int U, bool PERCH, int CDT>
__global__ void __launch_bounds__(kWarps * 32) decode_mma_kernel(DecodeArgs p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int K = p.K, N = p.N, M = p.M;
    const int n0 = blockIdx.x * 16;
    const int m0 = blockIdx.z * (8 * NT);
    const int nsb = K >> 6;
    const int sb_begin = (int)((long long)nsb * blockIdx.y / gridDim.y);
    const int sb_end = (int)((long long)nsb * (blockIdx.y + 1) / gridDim.y);
    const int nb = K / p.block;
    const int sb_per_blk = p.block >> 6;

    // weight rows of this lane (clamped; rows >= N are computed but never stored)
    const int r0 = min(n0 + g, N - 1), r1 = min(n0 + g + 8, N - 1);
    const uint8_t* Bp = static_cast<const uint8_t*>(p.Bp);
    constexpr int kRowBytesPerSb = FMT == FMT_INT4 ? 32 : (FMT == FMT_INT8 ? 64 : 128);
    const size_t row_bytes = (size_t)nsb * kRowBytesPerSb;
    const uint8_t* w0p = Bp + (size_t)r0 * row_bytes + t * (kRowBytesPerSb / 4);
    const uint8_t* w1p = Bp + (size_t)r1 * row_bytes + t * (kRowBytesPerSb / 4);
    // activation rows of this lane for each column tile
    const uint16_t* A = static_cast<const uint16_t*>(p.A);
    bool arow_ok[NT];
    const uint16_t* ap[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int m = m0 + nt * 8 + g;
        arow_ok[nt] = m < M;
        ap[nt] = A + (size_t)(arow_ok[nt] ? m : 0) * K + t * 16;
    }
    const uint32_t kOne = BF ? 0x3F803F80u : 0x3C003C00u;

    float acc[NT][4], dp[NT][4], ds[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[nt][c] = dp[nt][c] = ds[nt][c] = 0.f;

    for (int sb0 = sb_begin + warp; sb0 < sb_end; sb0 += kWarps * U) {
        // ---- issue every load of U sub-blocks first
        uint32_t wr0[U][FMT == FMT_INT4 ? 2 : (FMT == FMT_INT8 ? 4 : 8)];
        uint32_t wr1[U][FMT == FMT_INT4 ? 2 : (FMT == FMT_INT8 ? 4 : 8)];
        uint4 act[U][NT][2];
        float2 ts0[U], ts1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int sb = sb0 + u * kWarps;
            if (sb < sb_end) {
                const size_t off = (size_t)sb * kRowBytesPerSb;
                if constexpr (FMT == FMT_INT4) {
                    const uint2 x0 = ldg_stream64(w0p + off), x1 = ldg_stream64(w1p + off);
                    wr0[u][0] = x0.x; wr0[u][1] = x0.y;
                    wr1[u][0] = x1.x; wr1[u][1] = x1.y;
                } else if constexpr (FMT == FMT_INT8) {
                    const uint4 x0 = ldg_stream128(w0p + off), x1 = ldg_stream128(w1p + off);
                    wr0[u][0] = x0.x; wr0[u][1] = x0.y; wr0[u][2] = x0.z; wr0[u][3] = x0.w;
                    wr1[u][0] = x1.x; wr1[u][1] = x1.y; wr1[u][2] = x1.z; wr1[u][3] = x1.w;
                } else {
                    const uint4 x0 = ldg_stream128(w0p + off), x1 = ldg_stream128(w0p + off + 16);
                    const uint4 y0 = ldg_stream128(w1p + off), y1 = ldg_stream128(w1p + off + 16);
                    wr0[u][0] = x0.x; wr0[u][1] = x0.y; wr0[u][2] = x0.z; wr0[u][3] = x0.w;
                    wr0[u][4] = x1.x; wr0[u][5] = x1.y; wr0[u][6] = x1.z; wr0[u][7] = x1.w;
                    wr1[u][0] = y0.x; wr1[u][1] = y0.y; wr1[u][2] = y0.z; wr1[u][3] = y0.w;
                    wr1[u][4] = y1.x; wr1[u][5] = y1.y; wr1[u][6] = y1.z; wr1[u][7] = y1.w;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (arow_ok[nt]) {
                        act[u][nt][0] = ldg128(ap[nt] + (size_t)sb * 64);
                        act[u][nt][1] = ldg128(ap[nt] + (size_t)sb * 64 + 8);
                    } else {
                        act[u][nt][0] = act[u][nt][1] = make_uint4(0, 0, 0, 0);
                    }
                }
                if constexpr (FMT != FMT_FLOAT && !PERCH) {
                    const int blk = sb / sb_per_blk;
                    ts0[u] = ldg_f2(p.T + ((size_t)r0 * nb + blk) * 2);
                    ts1[u] = ldg_f2(p.T + ((size_t)r1 * nb + blk) * 2);
                }
            }
        }
        // ---- convert, multiply, scale
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int sb = sb0 + u * kWarps;
            if (sb >= sb_end) break;
            // A operand (weights) for the 4 MMAs of this sub-block: for MMA j,
            // (fa0[2j], fa1[2j], fa0[2j+1], fa1[2j+1]) = (a0, a1, a2, a3)
            uint32_t fa0[8], fa1[8];
            if constexpr (FMT == FMT_INT4) {
                uint32_t q[4];
                int4_pairs<BF>(wr0[u][0], q); fa0[0] = q[0]; fa0[1] = q[1]; fa0[2] = q[2]; fa0[3] = q[3];
                int4_pairs<BF>(wr0[u][1], q); fa0[4] = q[0]; fa0[5] = q[1]; fa0[6] = q[2]; fa0[7] = q[3];
                int4_pairs<BF>(wr1[u][0], q); fa1[0] = q[0]; fa1[1] = q[1]; fa1[2] = q[2]; fa1[3] = q[3];
                int4_pairs<BF>(wr1[u][1], q); fa1[4] = q[0]; fa1[5] = q[1]; fa1[6] = q[2]; fa1[7] = q[3];
            } else if constexpr (FMT == FMT_INT8) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t q[2];
                    int8_pairs<BF>(wr0[u][i], q); fa0[2 * i] = q[0]; fa0[2 * i + 1] = q[1];
                    int8_pairs<BF>(wr1[u][i], q); fa1[2 * i] = q[0]; fa1[2 * i + 1] = q[1];
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) { fa0[i] = wr0[u][i]; fa1[i] = wr1[u][i]; }
            }
            if constexpr (!PERCH && FMT != FMT_FLOAT) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) dp[nt][c] = ds[nt][c] = 0.f;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t nw[8] = {act[u][nt][0].x, act[u][nt][0].y, act[u][nt][0].z, act[u][nt][0].w,
                                        act[u][nt][1].x, act[u][nt][1].y, act[u][nt][1].z, act[u][nt][1].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t b0, b1;
                    if constexpr (FMT == FMT_INT4) {
                        // MMA j = 2*uw + v uses k = 8uw + 2v + {0, 4 | 1, 5} of the lane's 16
                        const int uw = j >> 1, v = j & 1;
                        b0 = prmt(nw[4 * uw + v], nw[4 * uw + v + 2], 0x5410u);
                        b1 = prmt(nw[4 * uw + v], nw[4 * uw + v + 2], 0x7632u);
                    } else {
                        b0 = nw[2 * j];
                        b1 = nw[2 * j + 1];
                    }
                    if constexpr (FMT == FMT_FLOAT) {
                        mma16816<BF>(acc[nt], fa0[2 * j], fa1[2 * j], fa0[2 * j + 1], fa1[2 * j + 1], b0, b1);
                    } else {
                        mma16816<BF>(dp[nt], fa0[2 * j], fa1[2 * j], fa0[2 * j + 1], fa1[2 * j + 1], b0, b1);
                        mma16816<BF>(ds[nt], kOne, kOne, kOne, kOne, b0, b1);
                    }
                }
            }
            if constexpr (!PERCH && FMT != FMT_FLOAT) {
                // d[0], d[1]: channel row g, columns 2t, 2t+1; d[2], d[3]: channel row g + 8
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    acc[nt][0] += ts0[u].y * dp[nt][0] + ts0[u].x * ds[nt][0];
                    acc[nt][1] += ts0[u].y * dp[nt][1] + ts0[u].x * ds[nt][1];
                    acc[nt][2] += ts1[u].y * dp[nt][2] + ts1[u].x * ds[nt][2];
                    acc[nt][3] += ts1[u].y * dp[nt][3] + ts1[u].x * ds[nt][3];
                }
            }
        }
    }
    if constexpr (PERCH && FMT != FMT_FLOAT) {
        const float2 t0 = ldg_f2(p.T + (size_t)r0 * 2), t1 = ldg_f2(p.T + (size_t)r1 * 2);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            acc[nt][0] = t0.y * dp[nt][0] + t0.x * ds[nt][0];
            acc[nt][1] = t0.y * dp[nt][1] + t0.x * ds[nt][1];
            acc[nt][2] = t1.y * dp[nt][2] + t1.x * ds[nt][2];
            acc[nt][3] = t1.y * dp[nt][3] + t1.x * ds[nt][3];
        }
    }

    // ---- fixed-order reduction of the warps' partial sums
    __shared__ float red[kWarps][NT][32][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) red[warp][nt][lane][c] = acc[nt][c];
    __syncthreads();
    for (int idx = threadIdx.x; idx < NT * 32 * 4; idx += blockDim.x) {
        const int nt = idx >> 7, ln = (idx >> 2) & 31, c = idx & 3;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[w][nt][ln][c];
        const int row = n0 + (ln >> 2) + (c >= 2 ? 8 : 0);
        const int m = m0 + nt * 8 + 2 * (ln & 3) + (c & 1);
        if (row < N && m < M) {
            if (gridDim.y > 1)
                p.partial[((size_t)blockIdx.y * M + m) * N + row] = s;
            else
                store_out<CDT>(p.C, (size_t)m * N + row, s);
        }
    }
}

template <int CDT>
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int splits, size_t count, void* C) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count; i += (size_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int y = 0; y < splits; ++y) s += partial[(size_t)y * count + i];
        store_out<CDT>(C, i, s);
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
            o = p.T[((size_t)n * nb + blk) * 2 + 0];
            s = p.T[((size_t)n * nb + blk) * 2 + 1];
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
            if (m0 + r < p.M) store_out<CDT>(p.C, (size_t)(m0 + r) * p.N + n, acc[r]);
    }
    }
}

// ---------------------------------------------------------------- dispatch
template <int FMT, bool BF, int NT, int U, bool PERCH>
cudaError_t launch_mma_c(const DecodeArgs& a, cudaStream_t s, dim3 grid) {
    switch (a.splits > 1 ? DT_F32 : a.c_dtype) {
        case DT_F32: decode_mma_kernel<FMT, BF, NT, U, PERCH, DT_F32><<<grid, kWarps * 32, 0, s>>>(a); break;
        case DT_F16: decode_mma_kernel<FMT, BF, NT, U, PERCH, DT_F16><<<grid, kWarps * 32, 0, s>>>(a); break;
        default: decode_mma_kernel<FMT, BF, NT, U, PERCH, DT_BF16><<<grid, kWarps * 32, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

template <int FMT, bool BF>
cudaError_t launch_mma_fmt(const DecodeArgs& a, cudaStream_t s) {
    const int mt = a.M <= 8 ? 8 : 16;   // rows of A per thread block
    dim3 grid((a.N + 15) / 16, a.splits, (a.M + mt - 1) / mt);
    const bool perch = FMT != FMT_FLOAT && a.block == a.K;
    if (mt == 8) {
        return perch ? launch_mma_c<FMT, BF, 1, 4, true>(a, s, grid) : launch_mma_c<FMT, BF, 1, 4, false>(a, s, grid);
    }
    return perch ? launch_mma_c<FMT, BF, 2, 2, true>(a, s, grid) : launch_mma_c<FMT, BF, 2, 2, false>(a, s, grid);
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

int decode_splits(int M, int K, int N) {
    // Split K across thread blocks only when the channel groups alone cannot give every SM
    // two blocks; keep at least 8 sub-blocks (one per warp) per split.
    const int groups = ((N + 15) / 16) * ((M + 15) / 16);
    const int nsb = K / 64;
    int splits = 1;
    while (groups * splits < 2 * kTargetSms && nsb / (splits * 2) >= 8) splits *= 2;
    return splits;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    cudaError_t e;
    if (a.fmt == FMT_INT4)
        e = a.a_dtype == DT_BF16 ? launch_mma_fmt<FMT_INT4, true>(a, s) : launch_mma_fmt<FMT_INT4, false>(a, s);
    else if (a.fmt == FMT_INT8)
        e = a.a_dtype == DT_BF16 ? launch_mma_fmt<FMT_INT8, true>(a, s) : launch_mma_fmt<FMT_INT8, false>(a, s);
    else
        e = a.a_dtype == DT_BF16 ? launch_mma_fmt<FMT_FLOAT, true>(a, s) : launch_mma_fmt<FMT_FLOAT, false>(a, s);
    if (e != cudaSuccess || a.splits <= 1) return e;
    const size_t count = (size_t)a.M * a.N;
    const int threads = 256;
    const int blocks = (int)((count + threads - 1) / threads < 4096 ? (count + threads - 1) / threads : 4096);
    switch (a.c_dtype) {
        case DT_F32: splitk_reduce_kernel<DT_F32><<<blocks, threads, 0, s>>>(a.partial, a.splits, count, a.C); break;
        case DT_F16: splitk_reduce_kernel<DT_F16><<<blocks, threads, 0, s>>>(a.partial, a.splits, count, a.C); break;
        default: splitk_reduce_kernel<DT_BF16><<<blocks, threads, 0, s>>>(a.partial, a.splits, count, a.C); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_decode_f32(const DecodeArgs& a, cudaStream_t s) {
    if (a.a_dtype == DT_F32) return launch_f32_a<DT_F32>(a, s);
    if (a.a_dtype == DT_F16) return launch_f32_a<DT_F16>(a, s);
    return launch_f32_a<DT_BF16>(a, s);
}

}  // namespace qg
