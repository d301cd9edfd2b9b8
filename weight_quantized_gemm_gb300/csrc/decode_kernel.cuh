#pragma once
// The tensor-core decode kernel and its launch templates, instantiated once per weight format
// (decode_int4.cu, decode_int8.cu, decode_float.cu) so the instantiations compile in parallel.
// Decode path (small M): the weight stream.
//
// C[m][n] = sum_k A[m][k] * (q[n][k] * s[n][b(k)] + o[n][b(k)])   (benchmark page
// "MNN GemmSpeed 基准测试实战", «为什么用 Conv1x1 来测 GEMM»; at small M the layer is bound by
// the weight read, «几个可以直接读出的规律»).
//
// Arithmetic. Per 64-element K sub-block the sum is regrouped as s * sum_k a*q + o * sum_k a.
// The 4/8-bit codes are turned into exact integer-valued 16-bit floats in registers with the
// magic-number method of Kim et al., "Who Says Elephants Can't Run: Bringing Large Scale MoE
// Models into Cloud Scale Production" (2022): OR-ing the code into the mantissa of 1024.0
// (f16) or 128.0 (bf16) gives exactly bias + q. The bias is not subtracted per element: since
// sum_k a*(bias + q) = sum_k a*q + bias * sum_k a, it is folded into the offset,
// o' = o - bias * s, and the sub-block's contribution becomes s * P' + o' * S with
// P' = sum_k a*(bias + q) from a 16x8x16 tensor-core MMA (float32 accumulation; every product
// is exact) and S = sum_k a staged once per thread block. The weights (16 output channels x
// 16 k) are the MMA's A operand, the activations (up to 8 rows of A per column tile) its B
// operand. The MMA only sums over k, so the k order inside a sub-block is free as long as
// weights and activations agree; the activations are staged in shared memory already
// permuted into the order the cheap int4 conversion produces.
//
// Data movement. Persistent thread blocks (one per SM, 16 warps) walk over units of 16
// output channels; all 16 warps share a unit and interleave over its 64-wide K sub-blocks
// (warp w takes sub-blocks w, w+16, ...). Each warp streams its weight bytes (and the
// {offset, scale} pairs) through a private ring of cp.async stages several sub-blocks deep,
// so the bytes in flight per SM do not depend on registers, and the stream runs on across
// unit boundaries. At the end of a unit the 16 partial sums of each output are added in a
// fixed order in shared memory. When N is small, K is also split across thread blocks
// (gridDim.y) and a second kernel adds the float32 partials in a fixed order, so results are
// deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"

namespace qg {
namespace dec {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr size_t kMaxSmem = 232448;   // opt-in shared memory per thread block on sm_100-class GPUs
// cp.async stages per warp for the Int4 weight stream (build-time tuning constant, 2..5)
#ifndef QG_DEC_DEPTH_INT4
#define QG_DEC_DEPTH_INT4 3
#endif

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
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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

// Exact 16-bit values of the codes, offset by the format's bias (see above).
template <int FMT, bool BF>
struct Codes {
    static constexpr float kBias = FMT == FMT_INT4 ? (BF ? 128.f : 1024.f) : (FMT == FMT_INT8 && !BF ? 1024.f : 0.f);
};

// 8 nibbles n0..n7 (n_i = bits 4i..4i+3) -> p[0] = (n0, n4), p[1] = (n1, n5), p[2] = (n2, n6),
// p[3] = (n3, n7) as (low half, high half), each value bias + n.
template <bool BF>
__device__ __forceinline__ void int4_pairs(uint32_t w, uint32_t* p) {
    constexpr uint32_t kMagic = BF ? 0x43004300u : 0x64006400u;   // bf16 128.0 / f16 1024.0
    p[0] = lop3_and_or(w, 0x000F000Fu, kMagic);
    p[1] = lop3_and_or(w >> 4, 0x000F000Fu, kMagic);
    p[2] = lop3_and_or(w >> 8, 0x000F000Fu, kMagic);
    p[3] = lop3_and_or(w >> 12, 0x000F000Fu, kMagic);
}

// The A operand of MMA q is the quad {row g pair (2q), row g+8 pair (2q), row g pair (2q+1),
// row g+8 pair (2q+1)}. These helpers write conversions straight into such quads (a[q][0..3])
// so that no register moves are needed to assemble them.
template <bool BF>
__device__ __forceinline__ void int4_to_quads(uint32_t w, uint32_t (*a)[4], int row) {
    // word u of a row feeds MMAs 2u, 2u + 1; the caller passes a = &quads[2u], row 0 (g) or 1 (g + 8)
    constexpr uint32_t kMagic = BF ? 0x43004300u : 0x64006400u;
    a[0][row] = lop3_and_or(w, 0x000F000Fu, kMagic);            // (n0, n4)
    a[0][row + 2] = lop3_and_or(w >> 4, 0x000F000Fu, kMagic);   // (n1, n5)
    a[1][row] = lop3_and_or(w >> 8, 0x000F000Fu, kMagic);       // (n2, n6)
    a[1][row + 2] = lop3_and_or(w >> 12, 0x000F000Fu, kMagic);  // (n3, n7)
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// 4 bytes b0..b3 -> p[0] = (b0, b1), p[1] = (b2, b3). f16: 1024 + b. bf16: b itself (8-bit
// integers are exact in bf16 but too wide for its magic number, so they go through the
// float32 magic number 2^23 and are rounded, exactly, to bf16).
template <bool BF>
__device__ __forceinline__ void int8_pairs(uint32_t w, uint32_t* p) {
    if constexpr (!BF) {
        p[0] = prmt(w, 0x64646464u, 0x4140u);
        p[1] = prmt(w, 0x64646464u, 0x4342u);
    } else {
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

// Work split and ring geometry. A thread block's 16 warps share each unit of 16 output channels;
// each warp owns kSbw sub-blocks of the block's K-range per unit (sbl_of). One ring stage holds
// one warp's share of one unit, in copy groups:
//   Int4: a pair of adjacent sub-blocks, [16 rows][64 B] with the 16-byte chunk index XOR-ed
//         with (row & 3) (conflict-free 16-byte writes and 8-byte reads), then [16 rows][16 B]
//         of {offset, scale} for the two sub-blocks;
//   Int8, float: one sub-block, each lane's weight bytes for its two channel rows (g, g + 8) as
//         16-byte planes [plane][lane], then the 16 rows' {offset, scale} ordered (g, g + 8).
// A per-channel table (block == K) is stored once per stage instead.
template <int NT>
struct Share {
    static constexpr int kSbw = NT == 1 ? 4 : 2;            // sub-blocks per warp per unit
    static constexpr int kSbMaxNt = kSbw * kWarps;           // K-range per thread block (in sub-blocks)
};

template <int FMT, int NT, bool PERCH>
struct Ring {
    // Int4 rows are copied two adjacent sub-blocks (64 bytes) at a time with 16-byte cp.async.cg
    // (L2 only): smaller L1-allocating copies were measured to lose throughput as the ring grows.
    static constexpr bool kPair = FMT == FMT_INT4;
    static constexpr int kLaneBytes = FMT == FMT_INT4 ? 16 : (FMT == FMT_INT8 ? 32 : 64);   // per sub-block
    static constexpr int kGroupSb = kPair ? 2 : 1;                  // sub-blocks per copy group
    static constexpr int kGroups = Share<NT>::kSbw / kGroupSb;
    static constexpr int kGroupTable = (PERCH || FMT == FMT_FLOAT) ? 0 : (kPair ? 256 : 128);
    static constexpr int kGroupBytes = 32 * kLaneBytes * kGroupSb + kGroupTable;
    static constexpr int kStageBytes = kGroups * kGroupBytes + ((PERCH && FMT != FMT_FLOAT) ? 128 : 0);
    static constexpr int kDepth =
        FMT == FMT_INT4 ? (NT == 1 ? QG_DEC_DEPTH_INT4 : 3) : (FMT == FMT_INT8 ? (NT == 1 ? (PERCH ? 3 : 2) : 3) : 1);
    static constexpr int kRowBytesPerSb = FMT == FMT_INT4 ? 32 : (FMT == FMT_INT8 ? 64 : 128);
};

// Local index (within the thread block's K-range) of warp w's j-th sub-block: Int4 warps own
// pairs of adjacent sub-blocks (2w, 2w + 1), (2w + 32, 2w + 33); the others w, w + 16, ...
template <int FMT>
__device__ __forceinline__ int sbl_of(int warp, int j) {
    if constexpr (FMT == FMT_INT4) return 2 * warp + (j & 1) + 2 * kWarps * (j >> 1);
    else return warp + kWarps * j;
}

// Shared memory: [afrag [nsbc][NT][4][32] uint2, when the B operand is not kept in registers]
// asum [nsbc][NT*8] f32 | atot [NT*8] f32 | red [2][16][NT][32][4] f32 | ring [16][depth][stage].
template <int FMT, int NT, bool PERCH>
constexpr size_t smem_bytes(int nsbc) {
    using R = Ring<FMT, NT, PERCH>;
    return (NT == 1 ? 0 : (size_t)nsbc * NT * 1024) + (size_t)nsbc * NT * 32 + NT * 32 + 2 * (size_t)kWarps * NT * 512 +
           (size_t)kWarps * R::kDepth * R::kStageBytes;
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

template <bool BF>
__device__ __forceinline__ void mma16816_zc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
    const float z = 0.f;
    if constexpr (BF) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
    }
}

// B operand of the 4 MMAs of one sub-block from the lane's 16 consecutive activations
// (nw[i] = halves 2i, 2i+1), in the k order the weight conversion produces.
template <int FMT>
__device__ __forceinline__ void b_frags(const uint32_t (&nw)[8], uint32_t* b) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if constexpr (FMT == FMT_INT4) {
            // MMA j = 2u + v takes k = 8u + 2v + {0, 4} (b0) and 8u + 2v + {1, 5} (b1) of the lane's 16
            const int u = j >> 1, v = j & 1;
            b[2 * j] = prmt(nw[4 * u + v], nw[4 * u + v + 2], 0x5410u);
            b[2 * j + 1] = prmt(nw[4 * u + v], nw[4 * u + v + 2], 0x7632u);
        } else {
            b[2 * j] = nw[2 * j];
            b[2 * j + 1] = nw[2 * j + 1];
        }
    }
}

// Column sums of one sub-block's activations, sum_k a[m][k], in the MMA output layout:
// d[0] = column 2t, d[1] = column 2t + 1 (an A operand of all ones; products exact, f32 sums).
template <bool BF>
__device__ __forceinline__ float2 col_sums(const uint32_t* b) {
    const uint32_t one = BF ? 0x3F803F80u : 0x3C003C00u;
    float d[4];
    mma16816_zc<BF>(d, one, one, one, one, b[0], b[1]);
#pragma unroll
    for (int q = 1; q < 4; ++q) mma16816<BF>(d, one, one, one, one, b[2 * q], b[2 * q + 1]);
    return make_float2(d[0], d[1]);
}

// Everything one warp needs to issue the cp.async copies of one unit into one ring stage. All
// members are per-warp or per-lane constants, computed once, so issuing a unit costs only the
// row arithmetic and the copies themselves.
template <int FMT, int NT, bool PERCH, bool FULL>
struct Issuer {
    using R = Ring<FMT, NT, PERCH>;
    static constexpr int SBW = Share<NT>::kSbw;
    static constexpr bool kScaled = FMT != FMT_FLOAT && !PERCH;
    const uint8_t* bp;     // Bp + this lane's byte offset inside a row
    const float* T;
    size_t row_bytes;
    int N, nb, g, lane;
    int sb0;               // global index of the warp's first sub-block
    int sb_per_blk;        // sub-blocks per table block
    unsigned valid;        // bit j: the warp's sub-block j lies inside the K-range
    uint32_t wdst0, wdst1; // this lane's weight destinations inside a stage (rows g, g + 8)
    uint32_t tdst;         // this lane's table destination inside a stage (4-byte copies)
    int trow;              // the table row this lane copies (4-byte copies)

    __device__ __forceinline__ bool ok(int j) const { return FULL || ((valid >> j) & 1u); }
    // table column of the warp's sub-block j (j is a compile-time constant after unrolling)
    __device__ __forceinline__ int blk(int j) const {
        const int sb = sb0 + sbl_of<FMT>(0, j);
        return sb_per_blk == 1 ? sb : sb / sb_per_blk;
    }

    __device__ __forceinline__ void operator()(int n0, uint32_t st) const {
        const int r0 = min(n0 + g, N - 1), r1 = min(n0 + g + 8, N - 1);
        const uint8_t* w0 = bp + (size_t)r0 * row_bytes;
        const uint8_t* w1 = bp + (size_t)r1 * row_bytes;
        if constexpr (R::kPair) {
            const int t = lane & 3;
#pragma unroll
            for (int jp = 0; jp < R::kGroups; ++jp) {
                if (!ok(2 * jp)) continue;
                const uint32_t sg = st + jp * R::kGroupBytes;
                const size_t o = (size_t)jp * 2 * kWarps * R::kRowBytesPerSb;
                if (ok(2 * jp + 1) || t < 2) {
                    cp_async16(sg + wdst0, w0 + o);
                    cp_async16(sg + wdst1, w1 + o);
                }
                if constexpr (kScaled) {
                    // lanes 16 * q + r copy row r's {offset, scale} pairs of copy group q (all
                    // lanes copy group 0 when a stage holds one group)
                    const int q = R::kGroups == 2 ? (lane >> 4) : 0;
                    if (q == jp) {
                        const int rr = lane & 15;
                        const float* src = T + tab_index(n0 + rr, nb, blk(2 * jp)) * 2;
                        const uint32_t dst = sg + 1024 + rr * 16;
                        cp_async8(dst, src);
                        if (ok(2 * jp + 1)) cp_async8(dst + 8, src + 32 * (blk(2 * jp + 1) - blk(2 * jp)));
                    }
                }
            }
        } else {
            const int rt = min(n0 + trow, N - 1);
#pragma unroll
            for (int j = 0; j < SBW; ++j) {
                if (!ok(j)) continue;
                const uint32_t sj = st + j * R::kGroupBytes;
                const size_t o = (size_t)j * kWarps * R::kRowBytesPerSb;
                if constexpr (FMT == FMT_INT8) {
                    cp_async16(sj + wdst0, w0 + o);
                    cp_async16(sj + wdst1, w1 + o);
                } else {
                    cp_async16(sj + wdst0, w0 + o);
                    cp_async16(sj + wdst0 + 512, w0 + o + 16);
                    cp_async16(sj + wdst1, w1 + o);
                    cp_async16(sj + wdst1 + 512, w1 + o + 16);
                }
                if constexpr (kScaled)
                    cp_async4(sj + 32 * R::kLaneBytes + tdst, T + tab_index(rt, nb, blk(j)) * 2 + (lane & 1));
            }
        }
        if constexpr (PERCH && FMT != FMT_FLOAT) {
            const int rt = min(n0 + trow, N - 1);
            cp_async4(st + R::kGroups * R::kGroupBytes + tdst, T + tab_index(rt, 1, 0) * 2 + (lane & 1));
        }
    }
};

// One persistent thread block: units of 16 output channels (blockIdx.x, +gridDim.x, ...) over
// the K-range of split blockIdx.y, for at most 8 * NT rows of A.
//   ONECOL: M == 1, so only MMA column 0 carries data and only it is scaled.
//   FULL: every warp owns exactly kSbw sub-blocks (the K-range is 16 * kSbw sub-blocks).
template <int FMT, bool BF, int NT, bool PERCH, bool EP, bool ONECOL, bool FULL>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeArgs p) {
    using R = Ring<FMT, NT, PERCH>;
    constexpr int D = R::kDepth;
    constexpr int SBW = Share<NT>::kSbw;
    constexpr bool kScaled = FMT != FMT_FLOAT && !PERCH;   // scale per sub-block
    constexpr bool kRegB = NT == 1;                         // B operand kept in registers
    constexpr float kBias = Codes<FMT, BF>::kBias;
    extern __shared__ __align__(128) uint8_t smem[];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int K = p.K, N = p.N, M = p.M;
    const int nsb = K >> 6;
    const int sb_begin = (int)((long long)nsb * blockIdx.y / gridDim.y);
    const int sb_end = (int)((long long)nsb * (blockIdx.y + 1) / gridDim.y);
    const int nsbc = sb_end - sb_begin;
    const int groups = (N + 15) >> 4;
    const int nb = K / p.block;
    const int sb_per_blk = p.block >> 6;

    uint2* afrag = reinterpret_cast<uint2*>(smem);
    float* asum = reinterpret_cast<float*>(smem + (kRegB ? 0 : (size_t)nsbc * NT * 1024));
    float* atot = asum + (size_t)nsbc * NT * 8;
    float* red = atot + NT * 8;
    uint8_t* ring = reinterpret_cast<uint8_t*>(red + 2 * kWarps * NT * 128) + (size_t)warp * D * R::kStageBytes;
    const uint32_t ring_s = smem_u32(ring);

    Issuer<FMT, NT, PERCH, FULL> issue;
    issue.valid = 0;
#pragma unroll
    for (int j = 0; j < SBW; ++j) issue.valid |= (sbl_of<FMT>(warp, j) < nsbc ? 1u : 0u) << j;
    issue.sb0 = sb_begin + sbl_of<FMT>(warp, 0);
    issue.sb_per_blk = sb_per_blk;
    issue.row_bytes = (size_t)nsb * R::kRowBytesPerSb;
    issue.bp = static_cast<const uint8_t*>(p.Bp) + (size_t)(sb_begin + sbl_of<FMT>(warp, 0)) * R::kRowBytesPerSb +
               t * (R::kPair ? 16 : R::kRowBytesPerSb / 4);
    issue.T = p.T;
    issue.N = N;
    issue.nb = nb;
    issue.g = g;
    issue.lane = lane;
    if constexpr (R::kPair) {
        issue.wdst0 = (uint32_t)(g * 64 + ((t ^ (g & 3)) << 4));
        issue.wdst1 = issue.wdst0 + 512;
    } else {
        issue.wdst0 = (uint32_t)(lane * 16);
        issue.wdst1 = issue.wdst0 + (FMT == FMT_INT8 ? 512 : 1024);
    }
    // slot s = lane >> 1 holds row (s >> 1) + 8 * (s & 1), word lane & 1
    issue.trow = (lane >> 2) + 8 * ((lane >> 1) & 1);
    issue.tdst = (uint32_t)((lane >> 1) * 8 + (lane & 1) * 4);

    const int nu = (int)blockIdx.x < groups ? (groups - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    const int n_step = (int)gridDim.x * 16;

    // Let the next kernel on the stream launch (it only takes SMs as these blocks exit), start
    // the weight stream, then wait for the previous kernel's results before touching A or C.
    // Both griddepcontrol instructions are no-ops unless the launch carried the programmatic
    // serialization attribute.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int issue_ui = 0;
    uint32_t issue_st = ring_s;
#pragma unroll
    for (int i = 0; i < D - 1; ++i) {
        if (issue_ui < nu) issue((int)blockIdx.x * 16 + issue_ui * n_step, issue_st);
        cp_async_commit();
        ++issue_ui;
        issue_st = (i + 1 == D) ? ring_s : issue_st + R::kStageBytes;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const uint16_t* A = static_cast<const uint16_t*>(p.A);
    // B operand kept in registers (NT == 1): breg[j] for the warp's sub-block j; sreg[j] = the
    // sub-block's column sums for columns 2t, 2t + 1
    uint32_t breg[kRegB ? SBW : 1][8];
    float2 sreg[kRegB ? SBW : 1];
    if constexpr (kRegB) {
        uint32_t nw[SBW][8];
#pragma unroll
        for (int j = 0; j < SBW; ++j) {
#pragma unroll
            for (int q = 0; q < 8; ++q) nw[j][q] = 0u;
            if (issue.ok(j) && g < M) {
                const uint4* src = reinterpret_cast<const uint4*>(
                    A + (size_t)g * K + (size_t)(sb_begin + sbl_of<FMT>(warp, j)) * 64 + t * 16);
                const uint4 x = src[0], y = src[1];
                nw[j][0] = x.x; nw[j][1] = x.y; nw[j][2] = x.z; nw[j][3] = x.w;
                nw[j][4] = y.x; nw[j][5] = y.y; nw[j][6] = y.z; nw[j][7] = y.w;
            }
        }
#pragma unroll
        for (int j = 0; j < SBW; ++j) {
            b_frags<FMT>(nw[j], breg[j]);
            sreg[j] = col_sums<BF>(breg[j]);
            if (issue.ok(j) && g == 0) {
                asum[sbl_of<FMT>(warp, j) * 8 + 2 * t] = sreg[j].x;
                asum[sbl_of<FMT>(warp, j) * 8 + 2 * t + 1] = sreg[j].y;
            }
        }
    } else {
        for (int e = threadIdx.x; e < nsbc * NT * 32; e += kThreads) {   // a whole warp per (sub-block, tile)
            const int ln = e & 31, nt = (e >> 5) % NT, sbl = (e >> 5) / NT;
            const int m = nt * 8 + (ln >> 2), tt = ln & 3;
            uint32_t nw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (m < M) {
                const uint4* src = reinterpret_cast<const uint4*>(A + (size_t)m * K + (size_t)(sb_begin + sbl) * 64 + tt * 16);
                const uint4 x = src[0], y = src[1];
                nw[0] = x.x; nw[1] = x.y; nw[2] = x.z; nw[3] = x.w;
                nw[4] = y.x; nw[5] = y.y; nw[6] = y.z; nw[7] = y.w;
            }
            uint32_t b[8];
            b_frags<FMT>(nw, b);
            uint2* dst = afrag + (size_t)(sbl * NT + nt) * 4 * 32 + ln;
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j * 32] = make_uint2(b[2 * j], b[2 * j + 1]);
            const float2 S = col_sums<BF>(b);
            if (ln < 4) {
                asum[(sbl * NT + nt) * 8 + 2 * tt] = S.x;
                asum[(sbl * NT + nt) * 8 + 2 * tt + 1] = S.y;
            }
        }
    }
    __syncthreads();
    if constexpr (PERCH) {
        if (threadIdx.x < NT * 8) {
            float s = 0.f;
            for (int sbl = 0; sbl < nsbc; ++sbl) s += asum[sbl * NT * 8 + threadIdx.x];
            atot[threadIdx.x] = s;
        }
        __syncthreads();
    }

    // per-lane read offsets inside a stage
    int roff0 = 0, roff1 = 0, toff = 0;
    if constexpr (R::kPair) {
        roff0 = g * 64 + ((((t >> 1)) ^ (g & 3)) << 4) + ((t & 1) << 3);       // sub-block 0 of a pair
        roff1 = g * 64 + ((((2 + (t >> 1))) ^ (g & 3)) << 4) + ((t & 1) << 3); // sub-block 1 of a pair
        toff = 1024 + g * 16;
    } else {
        roff0 = lane * 16;
        toff = 32 * R::kLaneBytes + g * 16;
    }

    float acc[NT][4], dp[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[nt][c] = dp[nt][c] = 0.f;

    uint32_t cons = ring_s;   // stage being consumed (shared-space address)
    for (int ui = 0; ui < nu; ++ui) {
        const int n0 = (int)blockIdx.x * 16 + ui * n_step;
        if (issue_ui < nu) issue((int)blockIdx.x * 16 + issue_ui * n_step, issue_st);
        cp_async_commit();
        ++issue_ui;
        issue_st = (issue_st + R::kStageBytes == ring_s + D * R::kStageBytes) ? ring_s : issue_st + R::kStageBytes;
        cp_async_wait<D - 1>();
        __syncwarp();
        const uint32_t st = cons;
        cons = (cons + R::kStageBytes == ring_s + D * R::kStageBytes) ? ring_s : cons + R::kStageBytes;
        float4 tcc = make_float4(0.f, 0.f, 0.f, 0.f);   // per-channel {o_g, s_g, o_g+8, s_g+8}
        if constexpr (PERCH && FMT != FMT_FLOAT) tcc = lds128f(st + R::kGroups * R::kGroupBytes + g * 16);
        float4 tpair0 = make_float4(0.f, 0.f, 0.f, 0.f), tpair1 = tpair0;   // Int4: the current pair's table
#pragma unroll
        for (int j = 0; j < SBW; ++j) {
            if (!issue.ok(j)) continue;
            uint32_t a[4][4];   // A operand quads of the sub-block's 4 MMAs
            float s0 = 0.f, o0 = 0.f, s1 = 0.f, o1 = 0.f;
            if constexpr (FMT == FMT_INT4) {
                const uint32_t sg = st + (j >> 1) * R::kGroupBytes;
                const uint32_t off = (j & 1) ? (uint32_t)roff1 : (uint32_t)roff0;
                const uint2 x0 = lds64(sg + off);         // row g: 16 nibbles
                const uint2 x1 = lds64(sg + off + 512);   // row g + 8
                int4_to_quads<BF>(x0.x, &a[0], 0);
                int4_to_quads<BF>(x0.y, &a[2], 0);
                int4_to_quads<BF>(x1.x, &a[0], 1);
                int4_to_quads<BF>(x1.y, &a[2], 1);
                if constexpr (kScaled) {
                    if ((j & 1) == 0) {
                        tpair0 = lds128f(sg + toff);
                        tpair1 = lds128f(sg + toff + 128);
                    }
                    const float oa = (j & 1) ? tpair0.z : tpair0.x, sa = (j & 1) ? tpair0.w : tpair0.y;
                    const float ob = (j & 1) ? tpair1.z : tpair1.x, sbv = (j & 1) ? tpair1.w : tpair1.y;
                    s0 = sa; o0 = fmaf(-kBias, sa, oa);
                    s1 = sbv; o1 = fmaf(-kBias, sbv, ob);
                }
            } else {
                const uint32_t sj = st + j * R::kGroupBytes;
                if constexpr (FMT == FMT_INT8) {
                    const uint4 x = lds128(sj + roff0);         // row g: 16 bytes
                    const uint4 y = lds128(sj + roff0 + 512);   // row g + 8
                    const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {   // word q of a row holds MMA q's pairs
                        uint32_t pr[2];
                        int8_pairs<BF>(xw[q], pr); a[q][0] = pr[0]; a[q][2] = pr[1];
                        int8_pairs<BF>(yw[q], pr); a[q][1] = pr[0]; a[q][3] = pr[1];
                    }
                } else {
                    const uint4 x0 = lds128(sj + roff0), x1 = lds128(sj + roff0 + 512);
                    const uint4 y0 = lds128(sj + roff0 + 1024), y1 = lds128(sj + roff0 + 1536);
                    a[0][0] = x0.x; a[0][2] = x0.y; a[1][0] = x0.z; a[1][2] = x0.w;
                    a[2][0] = x1.x; a[2][2] = x1.y; a[3][0] = x1.z; a[3][2] = x1.w;
                    a[0][1] = y0.x; a[0][3] = y0.y; a[1][1] = y0.z; a[1][3] = y0.w;
                    a[2][1] = y1.x; a[2][3] = y1.y; a[3][1] = y1.z; a[3][3] = y1.w;
                }
                if constexpr (kScaled) {
                    const float4 tt4 = lds128f(sj + toff);
                    s0 = tt4.y; o0 = fmaf(-kBias, tt4.y, tt4.x);
                    s1 = tt4.w; o1 = fmaf(-kBias, tt4.w, tt4.z);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                uint32_t b[8];
                if constexpr (kRegB) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) b[q] = breg[j][q];
                } else {
                    const uint2* bf = afrag + (size_t)(sbl_of<FMT>(warp, j) * NT + nt) * 4 * 32 + lane;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint2 v = bf[q * 32];
                        b[2 * q] = v.x;
                        b[2 * q + 1] = v.y;
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (FMT == FMT_FLOAT) {
                        mma16816<BF>(acc[nt], a[q][0], a[q][1], a[q][2], a[q][3], b[2 * q], b[2 * q + 1]);
                    } else if constexpr (kScaled) {
                        if (q == 0)
                            mma16816_zc<BF>(dp[nt], a[0][0], a[0][1], a[0][2], a[0][3], b[0], b[1]);
                        else
                            mma16816<BF>(dp[nt], a[q][0], a[q][1], a[q][2], a[q][3], b[2 * q], b[2 * q + 1]);
                    } else {
                        mma16816<BF>(dp[nt], a[q][0], a[q][1], a[q][2], a[q][3], b[2 * q], b[2 * q + 1]);
                    }
                }
                if constexpr (kScaled) {
                    // d[0], d[1]: channel row g, columns 2t, 2t + 1; d[2], d[3]: channel row g + 8
                    float2 S;
                    if constexpr (kRegB) S = sreg[j];
                    else S = *reinterpret_cast<const float2*>(asum + (size_t)(sbl_of<FMT>(warp, j) * NT + nt) * 8 + 2 * t);
                    acc[nt][0] = fmaf(o0, S.x, fmaf(s0, dp[nt][0], acc[nt][0]));
                    acc[nt][2] = fmaf(o1, S.x, fmaf(s1, dp[nt][2], acc[nt][2]));
                    if constexpr (!ONECOL) {
                        acc[nt][1] = fmaf(o0, S.y, fmaf(s0, dp[nt][1], acc[nt][1]));
                        acc[nt][3] = fmaf(o1, S.y, fmaf(s1, dp[nt][3], acc[nt][3]));
                    }
                }
            }
        }
        __syncwarp();   // every lane has read the stage: it may be refilled by the next issue
        if constexpr (PERCH && FMT != FMT_FLOAT) {
            // the offset term o' * sum_k a belongs to the unit once: warp 0 adds it
            const float o0 = warp == 0 ? fmaf(-kBias, tcc.y, tcc.x) : 0.f;
            const float o1 = warp == 0 ? fmaf(-kBias, tcc.w, tcc.z) : 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float Sx = atot[nt * 8 + 2 * t], Sy = atot[nt * 8 + 2 * t + 1];
                acc[nt][0] = fmaf(o0, Sx, tcc.y * dp[nt][0]);
                acc[nt][1] = fmaf(o0, Sy, tcc.y * dp[nt][1]);
                acc[nt][2] = fmaf(o1, Sx, tcc.w * dp[nt][2]);
                acc[nt][3] = fmaf(o1, Sy, tcc.w * dp[nt][3]);
#pragma unroll
                for (int c = 0; c < 4; ++c) dp[nt][c] = 0.f;
            }
        }
        // fixed-order sum of the 16 warps' partials of this unit (double-buffered: one barrier)
        float* rb = red + (size_t)(ui & 1) * kWarps * NT * 128;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            *reinterpret_cast<float4*>(rb + ((size_t)(warp * NT + nt) * 32 + lane) * 4) =
                make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;
        }
        __syncthreads();
        if (threadIdx.x < NT * 128) {
            const int idx = threadIdx.x;
            const int nt = idx >> 7, ln = (idx >> 2) & 31, c = idx & 3;
            const int row = n0 + (ln >> 2) + (c >= 2 ? 8 : 0);
            const int m = nt * 8 + 2 * (ln & 3) + (c & 1);
            if (row < N && m < M) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) s += rb[((size_t)(w * NT + nt) * 32 + ln) * 4 + c];
                if (gridDim.y > 1)
                    p.partial[((size_t)blockIdx.y * M + m) * N + row] = s;
                else
                {
                    const size_t mn = (size_t)m * N + row;
                    if constexpr (EP) s = epilogue_apply_rt(p.ep, s, mn, row, p.c_dtype);
                    store_out_rt(p.C, mn, s, p.c_dtype);
                }
            }
        }
    }
    cp_async_wait<0>();
}

// ---------------------------------------------------------------- dispatch
// SMs of the device current at the first call (thread-safe one-time initialization).
inline int sm_count() {
    static const int count = [] {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = kTargetSms;
        return n;
    }();
    return count;
}

template <int FMT, bool BF, int NT, bool PERCH, bool EP, bool ONECOL, bool FULL>
cudaError_t launch_v(const DecodeArgs& a, cudaStream_t s) {
    const int nsb = a.K / 64;
    const int nsbc = (nsb + a.splits - 1) / a.splits;
    const size_t smem = smem_bytes<FMT, NT, PERCH>(nsbc);
    if (smem > kMaxSmem) return cudaErrorInvalidValue;
    auto kern = decode_kernel<FMT, BF, NT, PERCH, EP, ONECOL, FULL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int groups = (a.N + 15) / 16;
    const int per_split = sm_count() / a.splits > 0 ? sm_count() / a.splits : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(groups < per_split ? groups : per_split, a.splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int FMT, bool BF, int NT, bool PERCH, bool ONECOL>
cudaError_t launch_c(const DecodeArgs& a, cudaStream_t s) {
    // FULL: every split is exactly 16 warps x kSbw sub-blocks
    const bool full = (a.K / 64) == a.splits * Share<NT>::kSbMaxNt;
    // the fused epilogue gets its own instantiation (EP); split partials never take it
    if (a.splits == 1 && a.ep.any())
        return full ? launch_v<FMT, BF, NT, PERCH, true, ONECOL, true>(a, s)
                    : launch_v<FMT, BF, NT, PERCH, true, ONECOL, false>(a, s);
    return full ? launch_v<FMT, BF, NT, PERCH, false, ONECOL, true>(a, s)
                : launch_v<FMT, BF, NT, PERCH, false, ONECOL, false>(a, s);
}

// Shapes the TMA-fed kernel of decode_stream.cuh does not take: 9 <= M <= 16, or packed rows that
// are not a multiple of 128 bytes.
template <int FMT, bool BF>
cudaError_t launch_fmt(const DecodeArgs& a, cudaStream_t s) {
    const bool perch = FMT != FMT_FLOAT && a.block == a.K;
    if (a.M == 1) return perch ? launch_c<FMT, BF, 1, true, true>(a, s) : launch_c<FMT, BF, 1, false, true>(a, s);
    if (a.M <= 8) return perch ? launch_c<FMT, BF, 1, true, false>(a, s) : launch_c<FMT, BF, 1, false, false>(a, s);
    return perch ? launch_c<FMT, BF, 2, true, false>(a, s) : launch_c<FMT, BF, 2, false, false>(a, s);
}

}  // namespace dec
}  // namespace qg
