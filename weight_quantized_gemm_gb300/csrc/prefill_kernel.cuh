// Tensor-core kernel for larger M (prefill), W4A8 and Int8-Block0 codes: tcgen05 MMA with TMEM
// accumulators. The kernel template and its launch helpers; instantiated by prefill.cu
// (dequantizing forms) and prefill_codes.cu (W4A8 and Int8-Block0 codes).
//
// The layer C[M,N] = A[M,K] x dequant(B[K,N]) (benchmark page "MNN GemmSpeed 基准测试实战",
// «为什么用 Conv1x1 来测 GEMM») is computed transposed, D[n][m] = sum_k W[n][k] * A[m][k], so that
// the operand that needs work before it can be multiplied -- the packed weight -- is the MMA's
// A operand and lives in tensor memory, while the activations stream in by TMA:
//   - two TMA producer warps load, per pipeline stage, the stage's K slice of A (up to 256 rows,
//     128-byte swizzle) and the packed weight rows of the 128-channel tile with their {offset,
//     scale} table entries into shared memory; a stage is one or two 64-wide sub-stages of K;
//   - dequant warps rebuild w = q * scale + offset in float32 (one rounding to the activation's
//     16-bit type) and write them into a TMEM stage with tcgen05.st;
//   - one thread issues tcgen05.mma (kind::f16, M = 128, N = tile rows of A, K = 16 per
//     instruction) with A from TMEM and B from shared memory, accumulating in TMEM, and
//     commits each stage back to the producers;
//   - after the last stage the dequant warps read the accumulator with tcgen05.ld and stage the
//     tile in ring slots reserved for it; a store warp writes it out by TMA, 32 rows per store
//     as soon as they are staged (where the rows allow), then hands the slots back.
// Blocks are persistent where the staging leaves the ring a slot for the next tile: at most one
// per SM, each running through a sequence of tiles while the ring's stages and barrier phases run
// on (see the kernel's own comment).
// Shapes whose tiles fill less than one wave of SMs split K across blocks (grid z): each split
// writes float32 partial sums and a second kernel adds them in a fixed order.
// W4A8 ("W4 解包为 INT8 ... S8×S8→S32", «测试用例与注册机制») uses the same kernel with the 4-bit
// codes as exact f16 integers and the activation codes as exact f16 integers: every product is
// an integer below 2^11 and, over at most 8808 of K, every partial sum an integer below 2^24, so
// the float32 tensor-core accumulation is exact and equals the int32 sum; the epilogue then
// either stores it as int32 (or adds it into int32 accumulators, one K-chunk per split, for
// longer K) or applies as * (ws * acc + off * rowsum).
// Int8-Block0 (one {offset, scale} per channel, «为什么用 Conv1x1 来测 GEMM») takes the same route
// with float activations: sum_k a (q s + o) = s * sum_k a q + o * sum_k a, so the MMA multiplies
// the raw 8-bit codes (exact 16-bit integers, also in bf16: no hi/lo weight split) and the
// epilogue applies s and o with the row sums of A from a pre-pass.
//
// Every wait on an mbarrier is bounded: a wait that runs out sets the library's status word and
// an abort flag, all roles leave their loops, in-flight work is drained (bounded) and TMEM is
// freed before the kernel returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace qg {

namespace pf {

constexpr int kBM = 128;              // output channels per tile (MMA M)
constexpr int kBK = 64;               // K per pipeline stage
constexpr int kMaxBN = 256;           // rows of A per tile (MMA N), a multiple of 64
// warps: 0 TMA (activation boxes), 1 MMA + TMEM, 2..9 dequant + epilogue, 10 TMA (weight and
// table boxes), 11 the output tiles' TMA stores and the residual tiles' loads. Two producer lanes
// in different warps issue a stage's copies side by side: one lane issuing all of a stage's copies
// paced the Int4 prefill at ~440 ns per stage, above the MMA's ~320 ns (measured with per-stage
// timestamps).
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;   // dequant + epilogue threads (warps 2 .. 9)
constexpr int kWProdWarp = 2 + kEpiWarps;     // the weight / table producer warp
constexpr int kStoreWarp = kWProdWarp + 1;    // the store warp
constexpr int kTmemCols = 512;
constexpr int kAccCol = 0;            // accumulator columns [0, BN); the A stages follow

// Weight forms: INT4 / INT8 dequantized per K-block; FLOAT 16-bit weights; CODES4 / CODES8 the
// raw 4- / 8-bit codes as exact 16-bit integers (the per-channel scale and offset are applied in
// the epilogue: W4A8, and Int8-Block0 with C = s * sum(a q) + o * sum(a)).
enum Wf { WF_INT4 = 0, WF_INT8 = 1, WF_FLOAT = 2, WF_CODES4 = 3, WF_CODES8 = 4 };
enum Epi { EPI_STORE = 0, EPI_W4A8 = 1, EPI_ACC = 2 };

struct Params {
    int M, K, N, block, nb, BN;
    const uint8_t* Bp;
    const float* T;
    void* C;
    const float* a_scale;     // W4A8: per-row activation scale (none: 1)
    const int32_t* rowsum;    // W4A8: per-row sum of activation codes
    const float* rowsum_f;    // CODES8: per-row float32 sum of the activations (when rowsum is null)
    int32_t* acc;             // EPI_ACC output
    int acc_add;              // EPI_ACC: add the tile into acc (int32, exact) instead of storing it; the
                              // K-splits then all add into the one [M][N] array
    int c_tma;                // the output tile goes out by TMA stores of 32 rows (else 16-byte row stores)
    int r_tma;                // the epilogue's residual tile comes in by one TMA load (Maps::r)
    int splits;               // K-splits (grid z): split z writes float32 partial sums to C + z M N
    int tblocks;              // K-blocks per table box (min(SUB, nb))
    int m_tiles;              // row tiles (ceil(M / BN)); the grid's x enumerates (channel tile, row tile)
    int group_n;              // channel tiles per raster group (row tiles run fastest inside a group);
                              // 0: channel tiles fastest over the whole grid
    unsigned int* status;     // the library's device status word (bounded waits that gave up)
    Epilogue ep;              // bias / activation / residual (none when the output is split partials)
    long long wait_ns;        // bound of each pipeline wait (waits that drain issued work: ptx::kWaitNs)
    int stall;                // diagnostic: the MMA issuer first waits on a barrier nothing arrives at
    float* rowmax;            // when set (no K-split): rowmax[x * M + m] = max over the tile's channels of
                              // |C[m][n]| as rounded to C's type, x = the tile's channel tile (the next layer's
                              // activation quantization takes the row max from these)
};

// ---------------------------------------------------------------- PTX helpers
using ptx::mbar_arrive;
using ptx::mbar_expect_tx;
using ptx::mbar_init;
using ptx::smem_u32;
using ptx::tma_load_2d;
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (TMEM) (+)= A (TMEM) x B (shared memory, descriptor)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
            d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D (TMEM) (+)= A (shared memory, descriptor) x B (shared memory, descriptor)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
            d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ uint4 lds128u(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float2 lds64f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile stored with the 128-byte swizzle: rows of
// 128 bytes (64 16-bit elements), 8-row swizzle atoms 1024 bytes apart (stride byte offset),
// descriptor version 1, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: D float32, A and B both f16 (0) or both bf16 (1), both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t idesc_f16(bool bf16, int n, int m) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
    uint32_t d;
    if (bf16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Dequantized weights with bf16 activations are split as w = hi + lo with hi = bf16(w) and
// lo = bf16(w - hi): the MMA then multiplies both parts, which keeps the weight to about 2^-17
// relative instead of bf16's 2^-9 (f16 weights are kept to 2^-12 by one rounding).
template <int WF, bool BF>
struct Split {
    static constexpr bool kOn = BF && (WF == WF_INT4 || WF == WF_INT8);
    static constexpr int kStageCols = kOn ? 64 : 32;
};

__device__ __forceinline__ uint32_t pack2_split(float lo, float hi, uint32_t& rest) {
    const uint32_t h = pack2(lo, hi, true);
    const float l0 = lo - __uint_as_float(h << 16), l1 = hi - __uint_as_float(h & 0xFFFF0000u);
    rest = pack2(l0, l1, true);
    return h;
}

// Exact float32 values of 4- and 8-bit codes without an integer conversion: a code placed in
// mantissa bits 15..18 of the float 256.0 reads 256 + q, in bits 19..22 of 16.0 it reads 16 + q,
// and an 8-bit code in bits 15..22 of 256.0 reads 256 + q. The bias folds into the offset, so
// w = q * s + o = fma(bias + q, s, o - bias * s) is a single rounding of the exact value plus the
// rounding of o - bias * s (at most 2^-24 * (|o| + 256 s), which is negligible).
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
// (x0, x1) * (s, s) + (c0, c1) in one packed float32 instruction
__device__ __forceinline__ void fma2(float x0, float x1, float s, float c0, float c1, float& r0, float& r1) {
    asm("{\n\t.reg .b64 x, y, z, d;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\tmov.b64 z, {%5, %6};\n\t"
        "fma.rn.f32x2 d, x, y, z;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(x0), "f"(x1), "f"(s), "f"(c0), "f"(c1));
}
// (x0, x1) * (y0, y1) in one packed float32 instruction
__device__ __forceinline__ void mul2(float x0, float x1, float y0, float y1, float& r0, float& r1) {
    asm("{\n\t.reg .b64 x, y, d;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "mul.rn.f32x2 d, x, y;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}
// byte j of w moved to bits 15..22
template <int J>
__device__ __forceinline__ uint32_t byte_to_15(uint32_t w) {
    if constexpr (8 * J < 15) return w << (15 - 8 * J);
    else return w >> (8 * J - 15);
}

// The 32 weights (k = k0 .. k0 + 31 of one channel row) this thread converts for one stage,
// as 16 packed 16-bit pairs (low half = even k); with Split, rest gets the low parts. raw holds
// the packed bytes.
template <int WF, bool BF>
__device__ __forceinline__ void convert32(const uint4 (&raw)[4], float s, float o, uint32_t (&out)[16],
                                          uint32_t (&rest)[16]) {
    constexpr bool kSplit = Split<WF, BF>::kOn;
    auto emit = [&](int idx, float w0, float w1) {
        if constexpr (kSplit) out[idx] = pack2_split(w0, w1, rest[idx]);
        else out[idx] = pack2(w0, w1, BF);
    };
    if constexpr (WF == WF_INT4) {
        const uint32_t w[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};   // 32 nibbles, byte j = (k 2j, 2j+1)
        const float c_lo = fmaf(-256.f, s, o), c_hi = fmaf(-16.f, s, o);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t t[4] = {byte_to_15<0>(w[i]), byte_to_15<1>(w[i]), byte_to_15<2>(w[i]), byte_to_15<3>(w[i])};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float q0 = __uint_as_float(lop3_and_or(t[j], 0x00078000u, 0x43800000u));   // 256 + low nibble
                const float q1 = __uint_as_float(lop3_and_or(t[j], 0x00780000u, 0x41800000u));   // 16 + high nibble
                float w0, w1;
                fma2(q0, q1, s, c_lo, c_hi, w0, w1);
                emit(4 * i + j, w0, w1);
            }
        }
    } else if constexpr (WF == WF_CODES4) {
        // the codes themselves, exact in f16: (1024 + lo, 1024 + 16 hi) -> (lo, hi)
        const uint32_t w[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t v = lop3_and_or(prmt(w[i], w[i], 0x4040u + 0x0101u * j), 0x00F0000Fu, 0x64006400u);
                uint32_t d;
                asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(v), "r"(0x2C003C00u), "r"(0xD400E400u));
                out[4 * i + j] = d;
            }
        }
    } else if constexpr (WF == WF_INT8 || WF == WF_CODES8) {   // CODES8: s = 1, o = 0, exact
        const uint32_t w[8] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w};
        const float c8 = fmaf(-256.f, s, o);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float q0 = __uint_as_float(lop3_and_or(byte_to_15<0>(w[i]), 0x007F8000u, 0x43800000u));
            const float q1 = __uint_as_float(lop3_and_or(byte_to_15<1>(w[i]), 0x007F8000u, 0x43800000u));
            const float q2 = __uint_as_float(lop3_and_or(byte_to_15<2>(w[i]), 0x007F8000u, 0x43800000u));
            const float q3 = __uint_as_float(lop3_and_or(byte_to_15<3>(w[i]), 0x007F8000u, 0x43800000u));
            float w0, w1, w2, w3;
            fma2(q0, q1, s, c8, c8, w0, w1);
            fma2(q2, q3, s, c8, c8, w2, w3);
            emit(2 * i, w0, w1);
            emit(2 * i + 1, w2, w3);
        }
    } else {
        const uint32_t w[16] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w,
                                raw[2].x, raw[2].y, raw[2].z, raw[2].w, raw[3].x, raw[3].y, raw[3].z, raw[3].w};
#pragma unroll
        for (int i = 0; i < 16; ++i) out[i] = w[i];
    }
}

template <int CDT>
__device__ __forceinline__ float load_s(const void* C, size_t idx) {   // element of a staged tile
    if constexpr (CDT == DT_F32)
        return static_cast<const float*>(C)[idx];
    else if constexpr (CDT == DT_F16)
        return __half2float(static_cast<const __half*>(C)[idx]);
    else
        return __bfloat162float(static_cast<const __nv_bfloat16*>(C)[idx]);
}
template <int CDT>
__device__ __forceinline__ void store_c(void* C, size_t idx, float v) {
    if constexpr (CDT == DT_F32)
        static_cast<float*>(C)[idx] = v;
    else if constexpr (CDT == DT_F16)
        static_cast<__half*>(C)[idx] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(v);
}

// Shared-memory stage of SUB sub-stages (SUB x 64 of K), at a multiple of 1024 bytes:
//   [SUB activation boxes, each [BN rows][128 B] with the 128-byte swizzle]
//   [weights: one box [128 rows][SUB x row bytes of a sub-stage] for the quantized formats, or
//    (float mode, SUB = 1) the 16-bit weights [128 rows][128 B] with the 128-byte swizzle, read by
//    the MMA directly as its A operand]
//   [formats with a table: the {offset, scale} entries of the stage's (up to) SUB K-blocks for the
//    tile's 128 channels, [8 groups of 16][SUB x 32 floats] in the grouped table layout]
// One stage is one round of the pipeline's barriers, so SUB = 2 halves the waits, arrivals and
// commits per unit of K; the ring holds as many stages as shared and tensor memory allow.
constexpr size_t kSmemMax = 232448;                 // opt-in shared memory per block
constexpr int kTail = 512 + kMaxBN * 8;              // barriers + W4A8 row factors after the ring
constexpr int kSlabRows = 32;                         // rows of A per TMA store of a staged tile
constexpr int kMaxSlabs = kMaxBN / kSlabRows;
constexpr int kRing = (int)kSmemMax - kTail;         // bytes for the stages
constexpr int kMaxStages = 8;
constexpr size_t kL2GroupBytes = 64u << 20;         // weights above this take the grouped raster
template <int WF>
struct WBox {   // bytes of one channel row of one 64-wide sub-stage
    static constexpr int kRowBytes =
        (WF == WF_INT4 || WF == WF_CODES4) ? kBK / 2 : ((WF == WF_INT8 || WF == WF_CODES8) ? kBK : 2 * kBK);
};
template <int WF, bool BF, int SUB>
struct Geo {
    static constexpr bool kTable = WF == WF_INT4 || WF == WF_INT8;
    static constexpr int kWBytes = kBM * SUB * WBox<WF>::kRowBytes;
    static constexpr int kTBytes = kTable ? SUB * (kBM / 16) * 128 : 0;
    static constexpr int kCols = SUB * Split<WF, BF>::kStageCols;   // TMEM columns of one A stage
    static constexpr int stage_bytes(int BN) { return SUB * BN * kBK * 2 + kWBytes + kTBytes; }
    // stages in the ring for tile height BN: what shared memory holds, and what tensor memory
    // holds beside the BN accumulator columns
    static constexpr int stages(int BN) {
        return kRing / stage_bytes(BN) < (kTmemCols - BN) / kCols
                   ? (kRing / stage_bytes(BN) < kMaxStages ? kRing / stage_bytes(BN) : kMaxStages)
                   : ((kTmemCols - BN) / kCols < kMaxStages ? (kTmemCols - BN) / kCols : kMaxStages);
    }
};
// The kernel's shape for tile height BN, fixed at compile time: two 64-wide sub-stages per stage
// (half the barrier rounds per unit of K) where the ring still holds at least kMinSub2Stages of
// them. The MMA issuer's per-stage work (barrier wait, commit) leaves the tensor pipe idle for a
// moment each stage, so fewer, larger stages keep it busier (measured on 256-row tiles: three
// 128-wide stages ran the W4A8 and Int4 prefill GEMMs 4-9% faster than six 64-wide ones).
constexpr int kMinSub2Stages = 3;
template <int WF, bool BF, int BN>
struct Plan {
    static constexpr int kSub = (WF != WF_FLOAT && Geo<WF, BF, 2>::stages(BN) >= kMinSub2Stages) ? 2 : 1;
    using G = Geo<WF, BF, kSub>;
    static constexpr int kStages = G::stages(BN);
    static constexpr int kStageBytes = G::stage_bytes(BN);
    static_assert(WF != WF_FLOAT || kSub == 1, "float mode loads one swizzled weight box per stage");
    static_assert(kStages >= 2 && kStages <= kMaxStages, "ring of at least two stages");
    static_assert(kStages * kStageBytes <= kRing, "ring fits in shared memory");
    static_assert(BN + kStages * G::kCols <= kTmemCols, "accumulator and A stages fit in TMEM");
    static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned (128-byte swizzle atoms)");
};
// The staged output tile [BN rows][128 channels] in C's type (int32 accumulators: 4 bytes) takes
// kSlots consecutive ring slots. Persistent form, where a tile's staging leaves the ring at least
// one slot for the next tile (2 kSlots - 1 <= stages: the reserved slots may have to skip the
// ring's last ones to stay contiguous): at most one block per SM runs through a sequence of tiles.
// After a tile's last stage the pipeline takes kSlots "staging positions" (plus skipped ones) in
// ring order: the producers put no copies there until the tile's TMA store has read them, while
// they already fill the other slots with the next tile's stages, so the store drains and the next
// tile's loads, dequantization and MMAs start behind the epilogue, and the block's setup (barriers,
// tensor memory, the first copies) is paid once. Otherwise (float32 or int32 tiles of 256 rows)
// the tile is staged over the first slots, idle after the tile's last MMA, and the grid holds one
// block per tile.
template <int WF, bool BF, int EPI, int CDT, int BN>
struct Tiling {
    using P = Plan<WF, BF, BN>;
    static constexpr int kTileBytes = BN * kBM * ((EPI == EPI_ACC || CDT == DT_F32) ? 4 : 2);
    static constexpr int kSlots = (kTileBytes + P::kStageBytes - 1) / P::kStageBytes;
    static constexpr bool kPersistent = 2 * kSlots - 1 <= P::kStages;
    static_assert(kSlots <= P::kStages, "the staged tile fits in the ring");
};
struct Maps {                 // the kernel's tensor maps
    CUtensorMap a;            // activations
    CUtensorMap w;            // packed weights
    CUtensorMap t;            // grouped {offset, scale} table (formats with a table)
    CUtensorMap c;            // the output, when Params::c_tma (stored by TMA from the staged tile)
    CUtensorMap r;            // the epilogue's residual, when Params::r_tma (same layout as c)
};

// OR of v over the dequant / epilogue warps (named barrier 1): the same answer in every thread.
__device__ __forceinline__ bool epi_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kEpiThreads)
        : "memory");
    return r != 0;
}

// One thread block runs the output tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... (one tile per
// block unless Tiling::kPersistent): tile t covers output channels [128 x, 128 x + 128) x rows of
// A [BN y, BN y + BN) (the raster below maps t to x, y) over the stages of K-split z (all of K
// when p.splits == 1). Every role walks the same sequence of ring positions: per tile its stages,
// then (persistent form) its staging positions; position g uses ring slot g % S, and every
// position completes one phase of each of the slot's barriers.
template <int WF, bool BF, int EPI, int CDT, int BN>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ Maps maps, Params p) {
    using T = Tiling<WF, BF, EPI, CDT, BN>;
    using P = typename T::P;
    using G = typename P::G;
    constexpr int SUB = P::kSub, S = P::kStages;
    constexpr uint32_t SB = P::kStageBytes;
    constexpr bool kDequant = WF != WF_FLOAT;          // weights go through the dequant warps into TMEM
    constexpr int kRowB = WBox<WF>::kRowBytes;
    constexpr int kLo = SUB * 32;                      // TMEM column of the low parts in an A stage (Split)
    // The packed weight box ([128 channel rows][SUB * kRowB bytes]) lands with the TMA swizzle whose
    // span is one row (32, 64 or 128 bytes): the 16-byte chunk index is XOR-ed with address bits
    // 7 and up, so the dequant warps' 16-byte reads of consecutive rows spread over all banks
    // instead of 4 rows sharing each 128-byte line's banks.
    constexpr uint32_t kWSwMask = (uint32_t)(SUB * kRowB) / 16u - 1u;
    auto wbox_swizzle = [](uint32_t a) { return a ^ (((a >> 7) & kWSwMask) << 4); };
    extern __shared__ __align__(1024) uint8_t smem[];
    // bounded pipeline wait reporting to the library's status word
    auto mbar_wait = [&](uint32_t bar, uint32_t parity, volatile int* abort) {
        return ptx::mbar_wait(bar, parity, abort, p.status, p.wait_ns);
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr uint32_t kABytes = (uint32_t)BN * kBK * 2;   // one activation box
    constexpr uint32_t w_off = SUB * kABytes, t_off = w_off + G::kWBytes;
    // Raster. Weights larger than the L2 share: groups of group_n channel tiles with the row tiles
    // fastest inside a group, so the tiles running at the same time share each weight tile (read
    // from HBM once) and re-read only the activations, which stay in L2. Otherwise channel tiles
    // fastest (group_n == 0): the weights stay in L2 and each activation tile is read by a run of
    // consecutive tiles.
    const int n_tiles = (p.N + kBM - 1) / kBM;
    const int total = n_tiles * p.m_tiles;
    auto tile_of = [&](int t) {   // {channel tile, row tile} of tile t
        if (p.group_n > 0) {
            const int per_group = p.group_n * p.m_tiles;
            const int grp = t / per_group, in_grp = t - grp * per_group;
            // (the last group may hold fewer channel tiles; the tiles cover exactly n_tiles x m_tiles)
            return make_int2(grp * p.group_n + in_grp / p.m_tiles, in_grp % p.m_tiles);
        }
        return make_int2(t % n_tiles, t / n_tiles);
    };
    const int nsub = p.K / kBK;                        // 64-wide sub-stages of K
    const int nst = (nsub + SUB - 1) / SUB;            // stages (the last may be half past K: reads 0)
    // split z covers stages [ks0, ks0 + nks) of every tile
    const int ks0 = (int)((long long)nst * blockIdx.z / p.splits);
    const int nks = (int)((long long)nst * (blockIdx.z + 1) / p.splits) - ks0;
    const int bpb = p.block / kBK;                     // sub-stages per table block

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRing);
    // bars: full[S] (the stage's boxes landed) | full_a[S] (TMEM A stage written) |
    //       empty[S] (MMAs of the stage done) | acc_full (the tile's MMAs done) |
    //       res_full (the residual tile landed, Params::r_tma) | stall (Params::stall: never
    //       arrived at) | acc_empty (the epilogue warps have read the accumulator) |
    //       staged (the output tile is staged) | taken (the store warp has taken it) |
    //       wt_staged (the weight producer has passed the tile's staging positions) |
    //       slab[BN / 32] (rows [32 k, 32 k + 32) of the tile are staged: one arrival per warp
    //       of the epilogue's column half that writes them)
    // A barrier's waiter must never fall two phases behind it (a parity wait would then pass on
    // the wrong phase): every wait below is on a phase that cannot complete twice without the
    // waiter's own progress.
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kMaxStages + 7 + kMaxSlabs);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // W4A8: per row m of the tile as[m] and as[m] * rowsum[m] (the row factors of the epilogue),
    // as two arrays so that two rows' factors load as one pair
    float* rf_as = reinterpret_cast<float*>(smem + kRing + 512);
    float* rf_ars = rf_as + kMaxBN;
    const uint32_t st_s = smem_u32(smem);
    auto full_x = [&](int s) { return smem_u32(bars + s); };
    auto full_a = [&](int s) { return smem_u32(bars + kMaxStages + s); };
    auto empty = [&](int s) { return smem_u32(bars + 2 * kMaxStages + s); };
    const uint32_t acc_full = smem_u32(bars + 3 * kMaxStages);
    const uint32_t res_full = smem_u32(bars + 3 * kMaxStages + 1);
    const uint32_t stall_bar = smem_u32(bars + 3 * kMaxStages + 2);
    const uint32_t acc_empty = smem_u32(bars + 3 * kMaxStages + 3);
    const uint32_t staged = smem_u32(bars + 3 * kMaxStages + 4);
    const uint32_t taken = smem_u32(bars + 3 * kMaxStages + 5);
    const uint32_t wt_staged = smem_u32(bars + 3 * kMaxStages + 6);
    auto slab = [&](int k) { return smem_u32(bars + 3 * kMaxStages + 7 + k); };
    constexpr int kSlabs = BN / kSlabRows;
    static_assert((3 * kMaxStages + 7 + kMaxSlabs) * 8 + 8 <= 512, "barriers, TMEM slot and abort flag fit the tail");
    constexpr uint32_t kTileBytes = (uint32_t)T::kTileBytes;
    // Staging positions after a tile whose stages end at position g_end: returns their count and
    // sets *slot to the first of the kSlots contiguous slots where the tile is staged (the
    // positions before it, if any, skip the ring's last slots). Not persistent: none; the tile is
    // staged from slot 0.
    auto staging_of = [](int g_end, int* slot) {
        if constexpr (!T::kPersistent) {
            *slot = 0;
            return 0;
        } else {
            const int a = g_end % S;
            *slot = a + T::kSlots > S ? 0 : a;
            return a + T::kSlots > S ? S - a + T::kSlots : T::kSlots;
        }
    };

    // Stage i of this split (ks0 + i) of tile tc into ring slot s, all copies completing
    // full_x(s): the SUB activation boxes with the expected bytes of the whole stage (issue_act,
    // warp 0), and the weight box and (formats with a table) the {offset, scale} entries of the
    // stage's K-blocks (issue_wt, warp kWProdWarp). A copy may complete before the expect_tx
    // arrival; the phase still waits for that arrival.
    const uint32_t stage_tx = SUB * kABytes + (uint32_t)G::kWBytes + (G::kTable ? (uint32_t)p.tblocks * 1024u : 0u);
    auto issue_act = [&](int2 tc, int i, int s) {
        const int ks = ks0 + i;
        const uint32_t st = st_s + (uint32_t)s * SB;
        mbar_expect_tx(full_x(s), stage_tx);
#pragma unroll
        for (int j = 0; j < SUB; ++j) tma_load_2d(st + j * kABytes, &maps.a, (ks * SUB + j) * kBK, tc.y * BN, full_x(s));
    };
    auto issue_wt = [&](int2 tc, int i, int s) {
        const int ks = ks0 + i;
        const uint32_t st = st_s + (uint32_t)s * SB;
        // weight box: x in bytes for the packed formats, in elements for float mode
        tma_load_2d(st + w_off, &maps.w, WF == WF_FLOAT ? ks * kBK : ks * SUB * kRowB, tc.x * kBM, full_x(s));
        if constexpr (G::kTable)   // 8 groups of 16 channels: x = 32 floats per K-block, y = group
                                   // (the box holds tblocks K-blocks, the stage's first one first)
            tma_load_2d(st + t_off, &maps.t, 32 * ((ks * SUB) / bpb), tc.x * (kBM / 16), full_x(s));
    };
    // A producer lane's walk over the block's ring positions (the first one leaves before the
    // block barrier): at every position it waits for the slot's previous use, then at a stage it
    // `issue`s, at a staging position the activation producer (act) arrives on full_x without
    // copies. The staging positions are released by the store warp, which does not wait for the
    // weight producer otherwise: so that this producer never falls two phases behind a slot's
    // empty barrier, it waits for the previous tile to be taken before the tile's staging
    // positions and reports passing them (wt_staged), which the store warp waits for before it
    // releases them. The activation producer also brings in the residual tile (Params::r_tma)
    // where the tile is staged, as soon as the staging slots' previous uses are done, so that its
    // latency hides behind the tile's last stages. After an abort, the copies issued land before
    // the block exits.
    auto produce = [&](auto&& issue, bool act) {
        const bool res = act && EPI != EPI_ACC && p.r_tma;
        int g = 0, s = 0, tj = 0, res_issued = 0;
        uint32_t ph = 0, real = 0;                     // real: bit s = the last use of slot s had copies
        bool stop = false;
        auto load_res = [&](int2 tc, int slot) {
            mbar_expect_tx(res_full, kTileBytes);
            ptx::tma_load_3d(st_s + (uint32_t)slot * SB, &maps.r, tc.x * kBM, tc.y * BN, 0, res_full);
            ++res_issued;
        };
        for (int t = blockIdx.x; t < total && !stop; t += gridDim.x, ++tj) {
            const int2 tc = tile_of(t);
            int slot;
            const int np = nks + staging_of(g + nks, &slot);
            for (int i = 0; i < np; ++i) {
                if (!act && i == nks && tj > 0 && !mbar_wait(taken, (uint32_t)(tj - 1) & 1u, abort_flag)) {
                    stop = true;
                    break;
                }
                if (g > 0) {
                    if (*abort_flag || !mbar_wait(empty(s), ph ^ 1u, abort_flag)) {
                        stop = true;
                        break;
                    }
                    if (i < nks) issue(tc, i, s);
                    else if (act) mbar_arrive(full_x(s));
                }
                real = i < nks ? real | (1u << s) : real & ~(1u << s);
                ++g;
                if (++s == S) { s = 0; ph ^= 1u; }
                // the last staging position: every staging slot's previous use is done; the
                // previous tile's residual has been read (its staged tile was taken)
                if (res && i == np - 1 && np > nks) {
                    if (tj > 0 && !mbar_wait(taken, (uint32_t)(tj - 1) & 1u, abort_flag)) {
                        stop = true;
                        break;
                    }
                    load_res(tc, slot);
                }
            }
            if (!act && !stop) {
                // (a tile without staging positions: still after the previous tile was taken)
                if (np == nks && tj > 0 && !mbar_wait(taken, (uint32_t)(tj - 1) & 1u, abort_flag)) break;
                mbar_arrive(wt_staged);
            }
        }
        if constexpr (!T::kPersistent) {
            // one tile, staged over the first slots: the residual comes in once the last use of
            // each slot under the staged tile is done
            if (res && !stop && !*abort_flag && total > (int)blockIdx.x) {
                bool free = true;
                for (int sl = 0; sl < T::kSlots && sl < nks && free; ++sl) {
                    const int last = sl + ((nks - 1 - sl) / S) * S;   // its last use
                    free = mbar_wait(empty(sl), (uint32_t)(last / S) & 1u, abort_flag);
                }
                if (free) load_res(tile_of(blockIdx.x), 0);
            }
        }
        if (*abort_flag) {
            for (int gg = g - S < 0 ? 0 : g - S; gg < g; ++gg) {
                if (!act && !((real >> (gg % S)) & 1u)) continue;   // no copies of this lane there
                volatile int never = 0;
                ptx::mbar_wait(full_x(gg % S), (uint32_t)(gg / S) & 1u, &never, p.status);
            }
            if (res_issued > 0) {   // a residual tile still in flight
                volatile int never = 0;
                ptx::mbar_wait(res_full, (uint32_t)(res_issued - 1) & 1u, &never, p.status);
            }
        }
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_x(s), 1);
            mbar_init(full_a(s), kEpiWarps);   // one arrival per dequant warp
            mbar_init(empty(s), 1);            // one tcgen05.commit per use
        }
        mbar_init(acc_full, 1);
        mbar_init(res_full, 1);
        mbar_init(stall_bar, 1);
        mbar_init(acc_empty, kEpiWarps);
        mbar_init(staged, 1);
        mbar_init(taken, 1);
        mbar_init(wt_staged, 1);
        for (int k = 0; k < kSlabs; ++k) mbar_init(slab(k), 4);   // the 4 warps of a column half
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        ptx::prefetch_tmap(&maps.a);
        ptx::prefetch_tmap(&maps.w);
        if constexpr (G::kTable) ptx::prefetch_tmap(&maps.t);
        // the first stage leaves before the block barrier and the tensor-memory allocation (its
        // ring slot starts free)
        if (nks > 0 && (int)blockIdx.x < total) {
            const int2 tc = tile_of(blockIdx.x);
            issue_act(tc, 0, 0);
            issue_wt(tc, 0, 0);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t a_col = tmem + (uint32_t)BN;        // A stages follow the BN accumulator columns

    if (warp == kWProdWarp) {
        // ---------------- TMA producer of the weight and table boxes
        if (lane == 0) produce(issue_wt, false);
    } else if (warp == 0) {
        // ---------------- TMA producer of the activation boxes
        if (lane == 0) produce(issue_act, true);
    } else if (warp == kStoreWarp) {
        // ---------------- the staged tiles out, 32 rows per TMA store as soon as they are staged
        // (the stores read shared memory while the epilogue still works on later rows), then
        // the staging positions released to the producers
        if (lane == 0) {
            constexpr uint32_t kEsz = (EPI == EPI_ACC || CDT == DT_F32) ? 4u : 2u;
            int g = 0;
            bool stop = false;
            for (int t = blockIdx.x, tj = 0; t < total && !stop; t += gridDim.x, ++tj) {
                int slot;
                const int g_end = g + nks;
                g = g_end + staging_of(g_end, &slot);
                const uint32_t stile = st_s + (uint32_t)slot * SB;
                if (p.c_tma) {
                    const int2 tc = tile_of(t);
                    // the two column halves of the epilogue stage their slabs side by side
                    for (int kk = 0; kk < kSlabs / 2 && !stop; ++kk) {
                        for (int hh = 0; hh < 2; ++hh) {
                            const int k = hh * (kSlabs / 2) + kk;
                            if (!mbar_wait(slab(k), (uint32_t)tj & 1u, abort_flag)) {
                                stop = true;
                                break;
                            }
                            // rows and channels past the end are not written
                            const uint32_t src = stile + (uint32_t)k * kSlabRows * kBM * kEsz;
                            if (EPI == EPI_ACC && p.acc_add)
                                ptx::tma_reduce_add_3d(&maps.c, tc.x * kBM, tc.y * BN + k * kSlabRows, 0, src);
                            else
                                ptx::tma_store_3d(&maps.c, tc.x * kBM, tc.y * BN + k * kSlabRows, blockIdx.z, src);
                            ptx::bulk_commit();
                        }
                    }
                    if (stop) break;
                }
                if (!mbar_wait(staged, (uint32_t)tj & 1u, abort_flag) ||
                    !mbar_wait(wt_staged, (uint32_t)tj & 1u, abort_flag))
                    break;
                mbar_arrive(taken);
                ptx::bulk_wait_read();
                for (int k = g_end; k < g; ++k) mbar_arrive(empty(k % S));   // the staging positions
            }
            ptx::bulk_wait_read();   // (after an abort: the stores issued have read shared memory)
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer. tcgen05.mma issue stalls while the tensor pipe's queue is
        // full, so the instructions between one stage's last MMA and the next stage's first one
        // leave the pipe idle: the next stage's barrier is tested before the stage's last MMA (with
        // MMAs still queued) and, when already complete, not waited for again.
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(BF, BN, kBM);
            int g = 0, s = 0, commits = 0;
            uint32_t ph = 0;
            bool stop = false;
            if (p.stall) mbar_wait(stall_bar, 0u, abort_flag);   // diagnostic: runs out, raises the abort flag
            // With dequant warps the MMAs wait on full_a only: every dequant warp waited for the
            // stage's TMA barrier (activations included) before it arrived on full_a, so acquiring
            // full_a orders the landed boxes before these MMAs.
            auto ready_bar = [&](int sl) { return kDequant ? full_a(sl) : full_x(sl); };
            for (int t = blockIdx.x, tj = 0; t < total && !stop && !*abort_flag; t += gridDim.x, ++tj) {
                int slot, skip = staging_of(g + nks, &slot);   // the tile's staging positions: no MMAs
                // the accumulator is free once the epilogue warps have read the previous tile
                if (tj > 0 && !mbar_wait(acc_empty, (uint32_t)(tj - 1) & 1u, abort_flag)) break;
                bool ready = false;                            // stage i's barrier was seen complete
#pragma unroll 2
                for (int i = 0; i < nks; ++i) {
                    if (!ready && !mbar_wait(ready_bar(s), ph, abort_flag)) { stop = true; break; }
                    tc_fence_after();
                    const uint32_t st = st_s + (uint32_t)s * SB;
                    const uint32_t as = a_col + (uint32_t)(s * G::kCols);
#pragma unroll
                    for (int j = 0; j < SUB; ++j) {
                        const uint64_t bdesc = sw128_desc(st + j * kABytes);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            if (j == SUB - 1 && kk == kBK / 16 - 1)   // before the stage's last MMA
                                ready = i + 1 < nks && ptx::mbar_try_wait(ready_bar(s + 1 == S ? 0 : s + 1),
                                                                          s + 1 == S ? ph ^ 1u : ph);
                            const uint32_t acc = (i | j | kk) != 0;   // the tile's first MMA overwrites
                            if constexpr (kDequant) {
                                mma_ts(tmem, as + 32 * j + kk * 8, bdesc + (uint64_t)(2 * kk), idesc, acc);
                                if constexpr (Split<WF, BF>::kOn)   // the low parts of the same weights
                                    mma_ts(tmem, as + kLo + 32 * j + kk * 8, bdesc + (uint64_t)(2 * kk), idesc, 1u);
                            } else {
                                const uint64_t adesc = sw128_desc(st + w_off);
                                mma_ss(tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc, acc);
                            }
                        }
                    }
                    mma_commit(empty(s));
                    ++g;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                mma_commit(acc_full);   // also after an abort: completes once every issued MMA has finished
                ++commits;
                for (; skip > 0; --skip) {
                    ++g;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            if (*abort_flag && commits > 0) {
                // the MMAs already issued finish before their tensor memory is released
                volatile int never = 0;
                ptx::mbar_wait(acc_full, (uint32_t)(commits - 1) & 1u, &never, p.status);
            }
        }
    } else {
        // ---------------- dequant warps (8): TMEM lane quarter q = warp % 4, K half h of each
        // 64-wide sub-stage; after a tile's last stage, its epilogue
        const int q = warp & 3, h = (warp - 2) >> 2;
        const int r = 32 * q + lane;                 // row inside the tile
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        constexpr int kEsz = (EPI == EPI_ACC || CDT == DT_F32) ? 4 : 2;
        int g = 0, s = 0;
        uint32_t ph = 0;
        // W4A8: per row m of a tile {as[m], as[m] * rowsum[m]} (row ri = this thread's row, BN <= 256)
        const int ri = threadIdx.x - 64;
        auto row_factors = [&](int m_tile) {
            const int m = min(m_tile + ri, p.M - 1);
            const float as = p.a_scale ? __ldg(p.a_scale + m) : 1.f;
            const float rs = p.rowsum ? (float)__ldg(p.rowsum + m) : __ldg(p.rowsum_f + m);
            return make_float2(as, as * rs);
        };
        for (int t = blockIdx.x, tj = 0; t < total; t += gridDim.x, ++tj) {
            const int2 tc = tile_of(t);
            const int n_idx = tc.x, n_tile = tc.x * kBM, m_tile = tc.y * BN;
            int slot;
            const int nstg = staging_of(g + nks, &slot);
            uint8_t* const tile = smem + (size_t)slot * SB;   // where the tile is staged
            const int row = n_tile + r;
            const int rc = row < p.N ? row : p.N - 1;
            if constexpr (EPI == EPI_W4A8) {
                // the first tile's row factors while its first stages are in flight (later tiles'
                // were stored after the previous epilogue's barrier)
                if (tj == 0 && ri < BN) {
                    const float2 f = row_factors(m_tile);
                    rf_as[ri] = f.x;
                    rf_ars[ri] = f.y;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");   // the epilogue warps only
            }
            if constexpr (kDequant) {
                int pos = (ks0 * SUB) % bpb;         // the first stage's first sub-stage in its K-block
                for (int i = 0; i < nks; ++i) {
                    if (!mbar_wait(full_x(s), ph, abort_flag)) break;
                    const uint32_t st = st_s + (uint32_t)s * SB;
                    uint32_t out[SUB][16], rest[SUB][16];
#pragma unroll
                    for (int j = 0; j < SUB; ++j) {
                        uint4 raw[4];
                        const uint32_t wsrc = st + w_off + r * (SUB * kRowB) + j * kRowB + h * (kRowB / 2);
                        raw[0] = lds128u(wbox_swizzle(wsrc));
                        if constexpr (WF == WF_INT8 || WF == WF_CODES8) raw[1] = lds128u(wbox_swizzle(wsrc + 16));
                        float2 e = make_float2(0.f, 1.f);   // {offset, scale} of this row and sub-stage
                        if constexpr (G::kTable) {
                            // K-block of the sub-stage in the box (the box starts at the stage's
                            // first block); a sub-stage past K (its weights and activations read 0)
                            // keeps the last block of the box
                            const int d = (j == 0 || pos + j < bpb) ? 0 : min(1, p.tblocks - 1);
                            e = lds64f(st + t_off + (r >> 4) * (p.tblocks * 128) + d * 128 + (r & 15) * 8);
                        }
                        convert32<WF, BF>(raw, e.y, e.x, out[j], rest[j]);
                    }
                    if (!mbar_wait(empty(s), ph ^ 1u, abort_flag)) break;
                    tc_fence_after();
                    const uint32_t dst = a_col + lane_base + (uint32_t)(s * G::kCols) + 16 * h;
#pragma unroll
                    for (int j = 0; j < SUB; ++j) {
                        tmem_st16(dst + 32 * j, out[j]);
                        if constexpr (Split<WF, BF>::kOn) tmem_st16(dst + kLo + 32 * j, rest[j]);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full_a(s));
                    ++g;
                    if (++s == S) { s = 0; ph ^= 1u; }
                    if (SUB > 1 || bpb > 1) {
                        pos += SUB;
                        while (pos >= bpb) pos -= bpb;
                    }
                }
            } else {
                for (int i = 0; i < nks; ++i) {   // the MMA reads the weights from shared memory
                    ++g;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            // The tile's staging positions: the producers stopped at them (full_x), and the MMAs of
            // the slots' previous uses are done (empty), so the slots are free for the staged tile;
            // with dequant warps, full_a keeps its one phase per position.
            for (int k = 0; k < nstg; ++k) {
                const bool here = mbar_wait(full_x(s), ph, abort_flag) && mbar_wait(empty(s), ph ^ 1u, abort_flag);
                if (!__all_sync(0xffffffffu, here)) break;
                if constexpr (kDequant)
                    if (lane == 0) mbar_arrive(full_a(s));
                ++g;
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            // W4A8: the next tile's row factors, loaded now so that their latency hides behind this
            // epilogue; stored after its barrier, once every thread has read this tile's
            const bool next_rf = EPI == EPI_W4A8 && t + (int)gridDim.x < total && ri < BN;
            const float2 nrf = next_rf ? row_factors(tile_of(t + gridDim.x).y * BN) : make_float2(0.f, 0.f);
            // ---------------- epilogue: this warp's lane quarter, columns [h BN/2, (h+1) BN/2).
            // The tile is written transposed into its staging slots as [m][128 n], then stored by
            // TMA stores of 32 rows (the store warp) or copied out row by row with 16-byte stores.
            bool ok = mbar_wait(acc_full, (uint32_t)tj & 1u, abort_flag) && !*abort_flag;
            tc_fence_after();
            const bool has_ep = EPI != EPI_ACC && p.ep.any();
            const bool has_res = has_ep && p.ep.residual != nullptr;
            // the residual tile, when it comes in by TMA, sits where this thread stages its outputs:
            // each element is read and then overwritten by the same thread
            const bool res_smem = has_res && p.r_tma;
            const bool res_glob = has_res && !p.r_tma;
            if (ok && res_smem) ok = mbar_wait(res_full, (uint32_t)tj & 1u, abort_flag);
            ok = __all_sync(0xffffffffu, ok);   // the tensor-memory loads below are warp-collective
            if (ok) {
                float ws = 0.f, wo = 0.f;
                if constexpr (EPI == EPI_W4A8) {
                    if constexpr (G::kTable) {   // block-quantized W4A8 weights: dequantized per block already
                        ws = 1.f;
                        wo = 0.f;
                    } else {                     // raw codes: the per-channel {offset, scale} here
                        const float2 tt = __ldg(reinterpret_cast<const float2*>(p.T + tab_index(rc, 1, 0) * 2));
                        wo = tt.x;
                        ws = tt.y;
                    }
                }
                // The fused epilogue: this thread's channel bias once, and per 32-column chunk the 32
                // residual values (32 independent loads, one 64-byte segment of a residual row per
                // warp each) before any of them is used; the activation is chosen once per chunk.
                const float bias_r = (p.ep.bias && row < p.N) ? __ldg(p.ep.bias + row) : 0.f;
                // (the store warp took the previous tile: the slab barriers never run two phases
                // ahead of it)
                if (p.c_tma && tj > 0 && lane == 0) mbar_wait(taken, (uint32_t)(tj - 1) & 1u, abort_flag);
                for (int c0 = h * (BN / 2); c0 < (h + 1) * (BN / 2); c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + kAccCol + c0, v);
                    float rv[32];
                    if (res_glob) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int m = m_tile + c0 + i;
                            rv[i] = (row < p.N && m < p.M) ? load_c<CDT>(p.ep.residual, (size_t)m * p.N + row) : 0.f;
                        }
                    }
                    tmem_ld_wait();
                    if constexpr (EPI == EPI_ACC) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            reinterpret_cast<int32_t*>(tile)[(size_t)(c0 + i) * kBM + r] = __float2int_rn(__uint_as_float(v[i]));
                    } else {
                        float y[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(v[i]);
                        if constexpr (EPI == EPI_W4A8) {
                            // per-channel rescale, as * (ws * acc + wo * rowsum) =
                            // fma(ws, as * acc, wo * (as * rowsum)): W4A8 (acc the exact integer sum,
                            // see the file comment) and CODES8 (as = 1, rowsum = sum of a); two rows
                            // per packed instruction, each rounded as the scalar steps would be. The
                            // row factors are the same for the whole warp: broadcast loads. With K
                            // split across blocks (CODES8), the offset term goes to split 0.
                            const bool off = blockIdx.z == 0;
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const float2 a2 = *reinterpret_cast<const float2*>(rf_as + c0 + i);
                                const float2 r2 = *reinterpret_cast<const float2*>(rf_ars + c0 + i);
                                float t0, t1, u0 = 0.f, u1 = 0.f;
                                mul2(a2.x, a2.y, y[i], y[i + 1], t0, t1);
                                if (off) mul2(wo, wo, r2.x, r2.y, u0, u1);
                                fma2(t0, t1, ws, u0, u1, y[i], y[i + 1]);
                            }
                        }
                        if (has_ep) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) y[i] += bias_r;
                            switch (p.ep.act) {
                                case ACT_RELU:
#pragma unroll
                                    for (int i = 0; i < 32; ++i) y[i] = act_fixed<ACT_RELU>(y[i]);
                                    break;
                                case ACT_SILU:
#pragma unroll
                                    for (int i = 0; i < 32; ++i) y[i] = act_fixed<ACT_SILU>(y[i]);
                                    break;
                                case ACT_GELU_TANH:
#pragma unroll
                                    for (int i = 0; i < 32; ++i) y[i] = act_fixed<ACT_GELU_TANH>(y[i]);
                                    break;
                                default: break;
                            }
                            if (res_glob) {
#pragma unroll
                                for (int i = 0; i < 32; ++i) y[i] += rv[i];
                            } else if (res_smem) {
#pragma unroll
                                for (int i = 0; i < 32; ++i) y[i] += load_s<CDT>(tile, (size_t)(c0 + i) * kBM + r);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i) store_c<CDT>(tile, (size_t)(c0 + i) * kBM + r, y[i]);
                    }
                    if (p.c_tma) {   // these 32 rows are staged by this warp: visible to the store
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(slab(c0 / kSlabRows));
                    }
                }
                // the accumulator has been read (tcgen05.wait::ld above): the next tile's MMAs may
                // overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
            // the staged tile (and this thread's reads of the residual in it) before the store
            // warp's TMA store and the copies that later reuse the slots
            ptx::fence_proxy_async_smem();
            // one decision for all epilogue warps: after an abort they leave the tile loop together
            if (epi_any(!ok || *abort_flag != 0)) break;
            if (next_rf) {
                rf_as[ri] = nrf.x;
                rf_ars[ri] = nrf.y;
            }
            if (!p.c_tma) {
                const int nvalid = min(kBM, p.N - n_tile), mvalid = min(BN, p.M - m_tile);
                constexpr int kPer = 16 / kEsz;                   // elements per 16-byte chunk
                constexpr int kChunks = kBM / kPer;               // chunks per tile row
                const bool add = EPI == EPI_ACC && p.acc_add;
                uint8_t* out = (EPI == EPI_ACC ? reinterpret_cast<uint8_t*>(p.acc) : static_cast<uint8_t*>(p.C)) +
                               (add ? 0 : (size_t)blockIdx.z * p.M * p.N * kEsz);
                const bool vec = ((size_t)p.N * kEsz) % 16 == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
                for (int idx = threadIdx.x - 64; idx < mvalid * kChunks; idx += kEpiThreads) {
                    const int ml = idx / kChunks, c = idx - ml * kChunks;
                    const int n0 = c * kPer;
                    if (n0 >= nvalid) continue;
                    const uint8_t* src = tile + ((size_t)ml * kBM + n0) * kEsz;
                    uint8_t* dst = out + ((size_t)(m_tile + ml) * p.N + n_tile + n0) * kEsz;
                    if (add) {   // int32 accumulators of one K-chunk added in (exact, any order)
                        for (int e = 0; e < kPer && n0 + e < nvalid; ++e)
                            atomicAdd(reinterpret_cast<int*>(dst) + e, reinterpret_cast<const int*>(src)[e]);
                    } else if (vec && n0 + kPer <= nvalid) {
                        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
                    } else {
                        for (int e = 0; e < kPer && n0 + e < nvalid; ++e)
                            for (int b = 0; b < kEsz; ++b) dst[e * kEsz + b] = src[e * kEsz + b];
                    }
                }
            }
            // Params::rowmax: the max over the tile's channels of each staged row (the values as
            // stored in C's type), read back from the staged tile. Each lane owns one row and visits
            // its 128 channels in 32 groups of 4, starting at group `lane` (the lanes of a warp then
            // read different banks); the loads are independent, so the pass is a few hundred cycles.
            if constexpr (EPI != EPI_ACC) {
                const int ml = (warp - 2) * 32 + lane;
                if (p.rowmax && warp - 2 < BN / 32 && ml < min(BN, p.M - m_tile)) {
                    const int nvalid = min(kBM, p.N - n_tile);
                    float mx = 0.f;
#pragma unroll 8
                    for (int j = 0; j < 32; ++j) {
                        const int c = 4 * ((j + lane) & 31);
                        float v[4];
                        if constexpr (kEsz == 4) {
                            const float4 x = *reinterpret_cast<const float4*>(tile + ((size_t)ml * kBM + c) * 4);
                            v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
                        } else {
                            const uint2 x = *reinterpret_cast<const uint2*>(tile + ((size_t)ml * kBM + c) * 2);
                            const uint32_t w[2] = {x.x, x.y};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const unsigned short b = (unsigned short)(w[e >> 1] >> (16 * (e & 1)));
                                v[e] = CDT == DT_F16 ? __half2float(__ushort_as_half(b)) : __uint_as_float((uint32_t)b << 16);
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (c + e < nvalid) mx = fmaxf(mx, fabsf(v[e]));
                    }
                    p.rowmax[(size_t)n_idx * p.M + m_tile + ml] = mx;
                }
            }
            // threads that read the staged tile above are done before the store warp hands its
            // slots back to the producers
            if (!p.c_tma || (EPI != EPI_ACC && p.rowmax)) asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
            // (the store warp took the previous tile: staged never runs two phases ahead of it)
            if (threadIdx.x == 64 && (tj == 0 || mbar_wait(taken, (uint32_t)(tj - 1) & 1u, abort_flag)))
                mbar_arrive(staged);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
// [M][K] 16-bit activations, box of 64 (K) x BN (rows), 128-byte swizzle; rows past M read 0.
inline cudaError_t make_tmap(CUtensorMap* map, const void* A, bool bf16, int M, int K, int BN) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)BN};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                           const_cast<void*>(A), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Rows of A per tile (the MMA's N): 64, 128 or 256.
inline int pick_bn(int M) {
    return M <= 64 ? 64 : (M <= 128 ? 128 : 256);
}


// The packed weight rows [N][row bytes] as a 2-D byte (quantized formats) or 16-bit (float mode,
// 128-byte swizzle) tensor; box = one stage (sub sub-stages of 64) of 128 rows; rows past N and
// bytes past K read 0.
inline cudaError_t make_wmap(CUtensorMap* map, const void* Bp, int wf, bool bf16, int N, int K, int sub) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    CUresult r;
    if (wf == WF_FLOAT) {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
        const cuuint32_t estr[2] = {1, 1};
        r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(Bp),
                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const bool byte_codes = wf == WF_INT8 || wf == WF_CODES8;
        const int row_bytes = byte_codes ? K : K / 2;
        const int box_bytes = sub * (byte_codes ? kBK : kBK / 2);
        const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
        const cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)kBM};
        const cuuint32_t estr[2] = {1, 1};
        // swizzle span = the box row (32, 64 or 128 bytes); the kernel reads with the same XOR
        const CUtensorMapSwizzle sw = box_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                      : (box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(Bp), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The grouped {offset, scale} table [ceil(N/16)][nb][16][2] as a 2-D float tensor: x = 32 floats
// per K-block of a group (16 channels x 2), y = group (stride nb * 128 bytes); box = tblocks
// consecutive K-blocks of 8 groups (the tile's 128 channels); entries past the end read 0.
inline cudaError_t make_table_map(CUtensorMap* map, const float* T, int N, int nb, int tblocks) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)32 * nb, (cuuint64_t)((N + 15) / 16)};
    const cuuint64_t strides[1] = {(cuuint64_t)nb * 128};
    const cuuint32_t box[2] = {(cuuint32_t)(32 * tblocks), (cuuint32_t)(kBM / 16)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(T), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The output [depth][M][N] (bf16 / f16 / f32, or int32 accumulators; depth = the K-splits' partial
// sums, else 1) as a 3-D tensor; box = 128 channels x box_rows rows of one slice, matching the staged
// [rows][128] tile (the output: one 32-row slab per store; the residual: the whole tile). Only when
// a row is a whole number of 16-byte units (TMA strides) and the base is 16-byte aligned; else
// returns false.
inline bool make_out_map(CUtensorMap* map, void* out, int kind, int M, int N, int box_rows, int depth) {
    const size_t esz = kind == DT_F32 || kind < 0 ? 4 : 2;
    if (((size_t)N * esz) % 16 != 0 || (reinterpret_cast<uintptr_t>(out) & 15) != 0) return false;
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const CUtensorMapDataType dt = kind < 0 ? CU_TENSOR_MAP_DATA_TYPE_INT32
                                   : (kind == DT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : (kind == DT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16));
    const cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)depth};
    const cuuint64_t strides[2] = {(cuuint64_t)N * esz, (cuuint64_t)M * N * esz};
    const cuuint32_t box[3] = {(cuuint32_t)kBM, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, dt, 3, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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

// The weight and table maps for the plan's sub-stages per stage, then the launch: one block per
// tile, or (persistent form) at most one block per SM, each taking every gridDim.x-th tile.
template <int WF, bool BF, int EPI, int CDT, int BN>
cudaError_t launch_k(Maps maps, Params p, cudaStream_t s) {
    using T = Tiling<WF, BF, EPI, CDT, BN>;
    using P = typename T::P;
    cudaError_t e = make_wmap(&maps.w, p.Bp, WF, BF, p.N, p.K, P::kSub);
    if (e != cudaSuccess) return e;
    p.tblocks = P::kSub < p.nb ? P::kSub : p.nb;
    if constexpr (P::G::kTable) e = make_table_map(&maps.t, p.T, p.N, p.nb, p.tblocks);
    else maps.t = maps.w;   // unused
    if (e != cudaSuccess) return e;
    auto kern = prefill_kernel<WF, BF, EPI, CDT, BN>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax);
    if (e != cudaSuccess) return e;
    const int tiles = ((p.N + kBM - 1) / kBM) * p.m_tiles;
    const int blocks = T::kPersistent && tiles > sm_count() ? sm_count() : tiles;
    dim3 grid(blocks, 1, p.splits);
    kern<<<grid, kThreads, kSmemMax, s>>>(maps, p);
    return cudaGetLastError();
}

// The raster for tile height BN, then the launch for the output type c_dtype (EPI_ACC: int32).
template <int WF, bool BF, int EPI, int BN>
cudaError_t launch_bn(Maps maps, Params p, int c_dtype, cudaStream_t s) {
    p.m_tiles = (p.M + BN - 1) / BN;
    // weights beyond half the L2 (measured: the 117 MB f16 weights of a 4096 x 14336 layer were read
    // about six times over with channel tiles fastest): row tiles fastest in groups of about two
    // waves of blocks
    const size_t wbytes = (size_t)p.N * p.K * WBox<WF>::kRowBytes / kBK;   // packed weight bytes
    p.group_n = wbytes > kL2GroupBytes ? ((2 * kTargetSms) / p.m_tiles > 1 ? (2 * kTargetSms) / p.m_tiles : 1) : 0;
    if constexpr (EPI == EPI_ACC) return launch_k<WF, BF, EPI, DT_F32, BN>(maps, p, s);
    switch (c_dtype) {
        case DT_F32: return launch_k<WF, BF, EPI, DT_F32, BN>(maps, p, s);
        case DT_F16: return launch_k<WF, BF, EPI, DT_F16, BN>(maps, p, s);
        default: return launch_k<WF, BF, EPI, DT_BF16, BN>(maps, p, s);
    }
}

template <int WF, bool BF, int EPI>
cudaError_t launch_wf(const Maps& maps, const Params& p, int c_dtype, cudaStream_t s) {
    switch (p.BN) {
        case 64: return launch_bn<WF, BF, EPI, 64>(maps, p, c_dtype, s);
        case 128: return launch_bn<WF, BF, EPI, 128>(maps, p, c_dtype, s);
        default: return launch_bn<WF, BF, EPI, 256>(maps, p, c_dtype, s);
    }
}

}  // namespace pf

// Int8-Block0 with bf16 activations on the codes path (prefill_codes.cu); p.rowsum_f set.
cudaError_t launch_prefill_codes8(const pf::Maps& maps, const pf::Params& p, int kdt, cudaStream_t s);

}  // namespace qg
