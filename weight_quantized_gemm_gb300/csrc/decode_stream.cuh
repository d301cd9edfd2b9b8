#pragma once
// Decode kernel for up to 8 rows of A, with the weight stream fed by TMA. The arithmetic is the
// one of decode_kernel.cuh: per 64-wide K sub-block, s * P' + o' * S, with P' from 16x8x16
// tensor-core MMAs on exact integer-valued 16-bit codes (weights as the A operand, the rows of A
// as the B operand) and S the sub-block's column sums of A.
//
// Data movement. A thread block is 16 consumer warps and one producer warp; it walks over units
// of 16 output channels (blockIdx.x, + gridDim.x, ...) within the K-range of split blockIdx.y,
// which is a whole number of 128-byte slices of the packed weight rows (rows are a multiple of
// 128 bytes long). One stage of the shared-memory ring holds up to 16 slices of the unit's 16
// rows (32 KB), loaded by a single TMA copy: the weights are described as a 3-D tensor
// {128 bytes, rows (stride: row bytes), slices (stride: 128 bytes)}, so that the box lands as
// [slice][row][128 bytes] and the 128-byte swizzle (16-byte chunk index XOR row % 8) makes the
// lanes' 8- and 16-byte reads of 8 rows at once free of bank conflicts. Few large copies matter:
// the copy engine of an SM holds only a limited number of copies in flight, and one copy per row
// left it short of the bytes in flight HBM needs. Consumer warp w owns slice w of every stage.
// Behind the weights the stage holds the unit's {offset,
// scale} entries for the stage's K-range, one more bulk copy thanks to the table's 16-channel
// grouping ([entry][16 channels][2]: a lane's reads of rows g cover 8 distinct banks). A stage's
// "full" mbarrier completes on the bulk-copy bytes, its "empty" mbarrier on one arrival per
// consumer warp. A unit takes one
// stage per 16 slices (1 for Int4, up to 2 for Int8 and 4 for 16-bit weights: a split's K-range
// is at most 64 sub-blocks, whose activations stay in registers).
//
// Consumers keep a unit's partial sums in registers and park them in a reduction slot; every
// kRed units the 16 consumer warps meet at a named barrier and add the slots up in a fixed
// order, so results do not depend on timing and no block-wide barrier sits in the weight stream.
// All mbarrier waits are bounded (see ptx.cuh); every role runs the same loop structure after an
// abort, so the named barriers are always reached by all consumer warps.
#include "decode_kernel.cuh"
#include "ptx.cuh"

namespace qg {
namespace dstream {

using dec::b_frags;
using dec::Codes;
using dec::col_sums;
using dec::int4_to_quads;
using dec::int8_pairs;
using dec::lds128;
using dec::lds64;
using dec::mma16816;
using dec::mma16816_zc;
using dec::store_out;
using ptx::smem_u32;

constexpr int kCWarps = 16;                          // consumer warps
constexpr int kThreads = (kCWarps + 1) * 32;         // + the producer warp
constexpr int kRows = 16;                            // output channels per unit (the MMA's M)
constexpr int kSliceBytes = 128;
constexpr int kSliceTile = kRows * kSliceBytes;      // one slice of a unit in shared memory (2 KB)
constexpr int kWStage = kCWarps * kSliceTile;        // weight region of a stage (32 KB)
constexpr int kMaxDepth = 6;
constexpr size_t kMaxSmem = 232448;                  // opt-in shared memory per block (sm_100 class)
constexpr unsigned kStatusMisaligned = 2u;          // status bit: shared memory not 1024-byte aligned
constexpr int kNJ = 4;                               // sub-blocks per consumer warp and unit (64 per unit)

// Shared memory besides the ring, for NT column tiles of 8 rows of A. One tile (M <= 8) keeps the
// B fragments in registers and reduces 4 units at a time. Two tiles (9 <= M <= 16) would need
// 64 fragment registers per thread, so the fragments of the warp's 4 sub-blocks x 2 tiles go to
// shared memory (1 KB per sub-block and tile, as two 16-byte planes per lane so that reads are
// conflict-free, plus the 8 column sums), and partial sums are reduced after every unit.
template <int NT>
struct Budget {
    static constexpr int kRed = NT == 1 ? 4 : 1;                           // units per reduction round
    static constexpr int kRedBytes = kRed * kCWarps * NT * 32 * 16;       // a float4 per lane, tile, warp, unit
    static constexpr int kFragBytes = NT == 1 ? 0 : kCWarps * kNJ * NT * 1024;
    static constexpr int kSumBytes = NT == 1 ? 0 : kCWarps * kNJ * NT * 32;
    static constexpr int kFixedBytes = kRedBytes + kCWarps * NT * 32 + kFragBytes + kSumBytes + (2 * kMaxDepth + 1) * 8 + 16;
};

template <int FMT>
struct Geo {
    static constexpr int kSbBytes = FMT == FMT_INT4 ? 32 : (FMT == FMT_INT8 ? 64 : 128);   // row bytes per sub-block
    static constexpr int kSps = kSliceBytes / kSbBytes;   // sub-blocks per slice
    static constexpr int kChunks = 4 / kSps;              // stages per unit at most
};

struct Params {
    int M, K, N;
    int nsb;            // 64-wide sub-blocks per row
    int nsl;            // 128-byte slices per row
    int sb_per_blk;     // sub-blocks per table entry
    int nb;             // table entries per row
    int bz;             // slices per stage (the TMA box depth, at most 16)
    int chunks;         // stages per unit in the largest split (at most Geo::kChunks)
    int depth;          // ring stages
    int row_bytes;      // packed bytes per weight row
    int stage_bytes;    // weights, then the table entries [entry][16 rows][2]; a multiple of 1024
    const void* A;
    const uint8_t* Bp;
    const float* T;
    void* C;
    float* partial;     // [splits][M][N] when gridDim.y > 1
    unsigned int* status;
    Epilogue ep;        // applied to the final sums (not to split partials) by the EP kernels
    int cdt;            // C's type
    long long wait_ns;  // bound of each pipeline wait (the producer's drain: ptx::kWaitNs)
    int stall;          // diagnostic: consumer warp 0 first waits on a barrier nothing arrives at
};

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCWarps * 32) : "memory");
}

template <int FMT, bool BF, bool PERCH, bool EP, bool ONECOL, int NT>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const __grid_constant__ CUtensorMap wmap, Params p) {
    using G = Geo<FMT>;
    using Bu = Budget<NT>;
    constexpr int SPS = G::kSps, CH = G::kChunks, NJ = kNJ, kRed = Bu::kRed;
    static_assert(SPS * CH == kNJ, "64 sub-blocks per unit over 16 warps");
    static_assert(NT == 1 || !ONECOL, "one column is one tile");
    constexpr bool kRegB = NT == 1;   // B fragments in registers
    constexpr bool kTable = FMT != FMT_FLOAT;
    constexpr bool kScaled = kTable && !PERCH;   // scale per sub-block
    constexpr float kBias = Codes<FMT, BF>::kBias;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int sl_begin = (int)((long long)p.nsl * blockIdx.y / gridDim.y);
    const int sl_end = (int)((long long)p.nsl * (blockIdx.y + 1) / gridDim.y);
    const int sb_end = min(sl_end * SPS, p.nsb);
    const int chunks = (sl_end - sl_begin + p.bz - 1) / p.bz;   // stages per unit in this split
    const int groups = (p.N + kRows - 1) / kRows;
    const int nu = (int)blockIdx.x < groups ? (groups - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    const int n_step = (int)gridDim.x * kRows;

    float* red = reinterpret_cast<float*>(smem + (size_t)p.depth * p.stage_bytes);   // [unit][warp][tile][lane] float4
    float* wsum = red + Bu::kRedBytes / 4;                                            // [warp][tile][8] column sums
    uint8_t* fragp = reinterpret_cast<uint8_t*>(wsum + kCWarps * NT * 8);   // [warp][jj][tile][plane][lane] 16 B
    float2* fsum = reinterpret_cast<float2*>(fragp + Bu::kFragBytes);       // [warp][jj][tile][t] column sums
    uint64_t* bars = reinterpret_cast<uint64_t*>(fragp + Bu::kFragBytes + Bu::kSumBytes);   // full | empty | stall
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kMaxDepth + 1);
    const uint32_t s_base = smem_u32(smem);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + kMaxDepth + s); };
    const uint32_t stall_bar = smem_u32(bars + 2 * kMaxDepth);

    // Stage idx of the block's stream (unit idx / chunks, K-chunk idx % chunks) into ring slot s:
    // the weights as one TMA box and the unit's table entries for the stage's K-range as one bulk
    // copy, both completing full(s). Issued by the producer's lane 0 only.
    const int total = nu * chunks;
    auto issue = [&](int idx, int s) {
        const int ui = idx / chunks, c = idx - ui * chunks;
        const int n0 = (int)blockIdx.x * kRows + ui * n_step;
        const int sl0 = sl_begin + c * p.bz;
        const int nsl_c = min(p.bz, sl_end - sl0);
        const uint32_t st = s_base + (uint32_t)(s * p.stage_bytes);
        uint32_t tbytes = 0;   // table bytes of the stage
        int e0 = 0;
        if constexpr (kTable) {
            // entries of sub-blocks [sb_c0, sb_c1) for the unit's 16 channels: one range
            const int sb_c0 = sl0 * SPS, sb_c1 = min((sl0 + nsl_c) * SPS, sb_end);
            e0 = sb_c0 / p.sb_per_blk;
            tbytes = (uint32_t)(((sb_c1 - 1) / p.sb_per_blk + 1 - e0) * 128);
        }
        ptx::mbar_expect_tx(full(s), (uint32_t)(p.bz * kSliceTile) + tbytes);
        ptx::tma_load_3d(st, &wmap, 0, n0, sl0, full(s));
        if constexpr (kTable) ptx::bulk_load(st + kWStage, p.T + tab_index(n0, p.nb, e0) * 2, tbytes, full(s));
    };
    // The producer's lane 0 initializes the barriers and at once issues the first stage, before the
    // block-wide barrier, so that the weight stream starts as early as the block does (the first
    // copy otherwise left ~1.3 us after block start). Only one: every copy issued here delays the
    // consumers' own set-up behind the barrier (measured on the 1 x 4096 x 11008 Int4 GEMV: one
    // stage 7.0 us, two 7.2, the whole ring 7.8, none 7.3).
    const int pre = total < 1 ? total : 1;
    if (warp == kCWarps && lane == 0) {
        for (int s = 0; s < p.depth; ++s) {
            ptx::mbar_init(full(s), 1);   // the producer's expect_tx arrival
            ptx::mbar_init(empty(s), kCWarps);
        }
        ptx::mbar_init(stall_bar, 1);
        // the swizzled TMA boxes need 1024-byte aligned stages
        *abort_flag = (s_base & 1023u) != 0;
        if (*abort_flag) atomicOr(p.status, kStatusMisaligned);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!*abort_flag) {
            ptx::prefetch_tmap(&wmap);
            for (int i = 0; i < pre; ++i) issue(i, i);
        }
    }
    __syncthreads();
    if (*abort_flag) return;
    // Let the next kernel on the stream launch (it takes SMs only as these blocks exit). The
    // weight stream does not depend on earlier kernels; A and C are touched after
    // griddepcontrol.wait. Both are no-ops without the programmatic serialization attribute.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kCWarps) {
        // ---------------- producer (lane 0): the remaining stages, each once its slot is free
        if (lane == 0) {
            int s = pre % p.depth, issued = pre;
            uint32_t ph = (uint32_t)(pre / p.depth) & 1u;
            for (int idx = pre; idx < total; ++idx) {
                // no stage is issued after an abort (consumers then stop releasing slots)
                if (*abort_flag || !ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, p.status, p.wait_ns)) break;
                issue(idx, s);
                ++issued;
                if (++s == p.depth) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // Every copy this warp started lands before the block can exit: in normal operation
            // the consumers have already seen all stages complete; after an abort the waits are
            // bounded.
            volatile int never = 0;
            const int first = issued > p.depth ? issued - p.depth : 0;
            for (int i = first; i < issued; ++i)
                ptx::mbar_wait(full(i % p.depth), (uint32_t)(i / p.depth) & 1u, &never, p.status);
        }
        return;
    }

    // ---------------- consumers
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint16_t* A = static_cast<const uint16_t*>(p.A);
    // the warp's sub-block jj = c * SPS + j (stage c of a unit): global index
    // (sl_begin + c * bz + warp) * SPS + j; B operand fragments and column sums in registers
    uint32_t breg[kRegB ? NJ : 1][8];
    float2 sreg[kRegB ? NJ : 1];
    uint32_t toff[NJ];   // byte offset of the sub-block's entry (16 rows x 8 bytes) in a stage's table
    float2 stot[NT];     // PERCH: column sums over the split's whole K-range, per tile
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) stot[nt] = make_float2(0.f, 0.f);
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
        const int c = jj / SPS, j = jj % SPS;
        const int sb = (sl_begin + c * p.bz + warp) * SPS + j;
        const bool valid = c < chunks && warp < p.bz && sb < sb_end;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int m = nt * 8 + g;   // the row of A this lane's fragment column holds
            uint32_t nw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (valid && m < p.M) {
                const uint4* src = reinterpret_cast<const uint4*>(A + (size_t)m * p.K + (size_t)sb * 64 + t * 16);
                const uint4 x = src[0], y = src[1];
                nw[0] = x.x; nw[1] = x.y; nw[2] = x.z; nw[3] = x.w;
                nw[4] = y.x; nw[5] = y.y; nw[6] = y.z; nw[7] = y.w;
            }
            uint32_t bt[8];
            b_frags<FMT>(nw, bt);
            const float2 S = col_sums<BF>(bt);
            if constexpr (kRegB) {
#pragma unroll
                for (int q = 0; q < 8; ++q) breg[jj][q] = bt[q];
                sreg[jj] = S;
            } else {
                uint4* plane = reinterpret_cast<uint4*>(fragp + (size_t)((warp * NJ + jj) * NT + nt) * 1024);
                plane[lane] = make_uint4(bt[0], bt[1], bt[2], bt[3]);
                plane[32 + lane] = make_uint4(bt[4], bt[5], bt[6], bt[7]);
                if (g == 0) fsum[((warp * NJ + jj) * NT + nt) * 4 + t] = S;
            }
            if constexpr (PERCH) {
                stot[nt].x += S.x;
                stot[nt].y += S.y;
            }
        }
        toff[jj] = 0;
        if constexpr (kTable) {
            const int sb_c0 = (sl_begin + c * p.bz) * SPS;
            const int sbv = valid ? sb : sb_c0;   // a copied entry even when the sub-block is unused
            toff[jj] = (uint32_t)((sbv / p.sb_per_blk - sb_c0 / p.sb_per_blk) * 128);
        }
    }
    if constexpr (!kRegB) __syncwarp();   // a warp reads only its own fragments
    if constexpr (PERCH) {
        if (g == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                wsum[(warp * NT + nt) * 8 + 2 * t] = stot[nt].x;
                wsum[(warp * NT + nt) * 8 + 2 * t + 1] = stot[nt].y;
            }
        }
        consumer_sync();
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            stot[nt] = make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kCWarps; ++w) {
                stot[nt].x += wsum[(w * NT + nt) * 8 + 2 * t];
                stot[nt].y += wsum[(w * NT + nt) * 8 + 2 * t + 1];
            }
        }
    }
    const uint32_t frag_s = smem_u32(fragp) + (uint32_t)(warp * NJ * NT * 1024 + lane * 16);
    const uint32_t fsum_s = smem_u32(fsum) + (uint32_t)(warp * NJ * NT * 32 + t * 8);

    // per-lane read offset inside the warp's slice of a stage: row g, the 16-byte chunk holding
    // the lane's 16 k of sub-block 0 (bytes 8t (Int4), 16t (Int8) or 32t (16-bit) of it), chunk
    // index XOR g; sub-block j is chunk-index XOR 2j (Int4) or 4j (Int8); row g + 8 is 1024 bytes
    // on with the same swizzle phase
    constexpr uint32_t kRow8 = 8 * kSliceBytes;
    uint32_t woff;
    if constexpr (FMT == FMT_INT4) woff = (uint32_t)(g * 128 + (((t >> 1) ^ g) << 4) + ((t & 1) << 3));
    else if constexpr (FMT == FMT_INT8) woff = (uint32_t)(g * 128 + ((t ^ g) << 4));
    else woff = (uint32_t)(g * 128 + (((2 * t) ^ g) << 4));
    const uint32_t trow0 = (uint32_t)(g * 8), trow1 = (uint32_t)((g + 8) * 8);   // rows g, g + 8 of an entry

    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    if (p.stall && warp == 0)   // diagnostic: runs out and raises the abort flag
        ok = ptx::mbar_wait(stall_bar, 0u, abort_flag, p.status, p.wait_ns);
    for (int ui0 = 0; ui0 < nu; ui0 += kRed) {
        const int nr = min(kRed, nu - ui0);
        for (int r = 0; r < nr; ++r) {
            float acc[NT][4], dp[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[nt][q] = dp[nt][q] = 0.f;
            float2 tp0 = make_float2(0.f, 0.f), tp1 = tp0;   // PERCH: {offset, scale} of rows g, g + 8
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                if (c >= chunks) break;
                ok = ok && ptx::mbar_wait(full(s), ph, abort_flag, p.status, p.wait_ns);
                // the stage holds slices [0, sl_end - first slice): a warp past them has nothing
                // loaded (stale bytes could even read as non-finite 16-bit weights)
                if (ok && warp < sl_end - (sl_begin + c * p.bz)) {
                    const uint32_t st = s_base + (uint32_t)(s * p.stage_bytes);
                    const uint32_t ws = st + warp * kSliceTile, ts = st + kWStage;
                    if constexpr (PERCH) {
                        if (c == 0) {
                            tp0 = lds64f(ts + trow0);
                            tp1 = lds64f(ts + trow1);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < SPS; ++j) {
                        const int jj = c * SPS + j;
                        uint32_t a[4][4];   // A operand quads of the sub-block's 4 MMAs
                        if constexpr (FMT == FMT_INT4) {
                            const uint32_t o = woff ^ (uint32_t)(32 * j);
                            const uint2 x0 = lds64(ws + o);           // row g: 16 nibbles
                            const uint2 x1 = lds64(ws + o + kRow8);   // row g + 8
                            int4_to_quads<BF>(x0.x, &a[0], 0);
                            int4_to_quads<BF>(x0.y, &a[2], 0);
                            int4_to_quads<BF>(x1.x, &a[0], 1);
                            int4_to_quads<BF>(x1.y, &a[2], 1);
                        } else if constexpr (FMT == FMT_INT8) {
                            const uint32_t o = woff ^ (uint32_t)(64 * j);
                            const uint4 x = lds128(ws + o);           // row g: 16 bytes
                            const uint4 y = lds128(ws + o + kRow8);   // row g + 8
                            const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {   // word q of a row holds MMA q's pairs
                                uint32_t pr[2];
                                int8_pairs<BF>(xw[q], pr);
                                a[q][0] = pr[0];
                                a[q][2] = pr[1];
                                int8_pairs<BF>(yw[q], pr);
                                a[q][1] = pr[0];
                                a[q][3] = pr[1];
                            }
                        } else {
                            const uint4 x0 = lds128(ws + woff), x1 = lds128(ws + (woff ^ 16u));
                            const uint4 y0 = lds128(ws + woff + kRow8), y1 = lds128(ws + (woff ^ 16u) + kRow8);
                            a[0][0] = x0.x; a[0][2] = x0.y; a[1][0] = x0.z; a[1][2] = x0.w;
                            a[2][0] = x1.x; a[2][2] = x1.y; a[3][0] = x1.z; a[3][2] = x1.w;
                            a[0][1] = y0.x; a[0][3] = y0.y; a[1][1] = y0.z; a[1][3] = y0.w;
                            a[2][1] = y1.x; a[2][3] = y1.y; a[3][1] = y1.z; a[3][3] = y1.w;
                        }
                        float2 e0 = make_float2(0.f, 0.f), e1 = e0;   // {o, s} of rows g, g + 8
                        if constexpr (kScaled) {
                            e0 = lds64f(ts + trow0 + toff[jj]);
                            e1 = lds64f(ts + trow1 + toff[jj]);
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            uint32_t b[8];
                            float2 S;
                            if constexpr (kRegB) {
#pragma unroll
                                for (int q = 0; q < 8; ++q) b[q] = breg[jj][q];
                                S = sreg[jj];
                            } else {
                                const uint32_t fa = frag_s + (uint32_t)((jj * NT + nt) * 1024);
                                const uint4 b0 = lds128(fa), b1 = lds128(fa + 512);
                                b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
                                b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
                                S = lds64f(fsum_s + (uint32_t)((jj * NT + nt) * 32));
                            }
                            if constexpr (kScaled) {
                                mma16816_zc<BF>(dp[nt], a[0][0], a[0][1], a[0][2], a[0][3], b[0], b[1]);
#pragma unroll
                                for (int q = 1; q < 4; ++q)
                                    mma16816<BF>(dp[nt], a[q][0], a[q][1], a[q][2], a[q][3], b[2 * q], b[2 * q + 1]);
                                const float o0 = fmaf(-kBias, e0.y, e0.x), o1 = fmaf(-kBias, e1.y, e1.x);
                                // dp[0], dp[1]: channel row g, columns 2t, 2t + 1; dp[2], dp[3]: row g + 8
                                acc[nt][0] = fmaf(o0, S.x, fmaf(e0.y, dp[nt][0], acc[nt][0]));
                                acc[nt][2] = fmaf(o1, S.x, fmaf(e1.y, dp[nt][2], acc[nt][2]));
                                if constexpr (!ONECOL) {
                                    acc[nt][1] = fmaf(o0, S.y, fmaf(e0.y, dp[nt][1], acc[nt][1]));
                                    acc[nt][3] = fmaf(o1, S.y, fmaf(e1.y, dp[nt][3], acc[nt][3]));
                                }
                            } else {
                                // one accumulation for the unit: per-channel scale (applied at the
                                // unit's end) or no scale at all (16-bit weights)
                                float(&d)[4] = PERCH ? dp[nt] : acc[nt];
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    mma16816<BF>(d, a[q][0], a[q][1], a[q][2], a[q][3], b[2 * q], b[2 * q + 1]);
                            }
                        }
                    }
                }
                __syncwarp();   // every lane has read the stage
                // A slot is released only once its copy has landed (lane 0 saw it complete): after an
                // abort no slot whose copy may still be in flight is handed back to the producer.
                if (lane == 0 && ok) ptx::mbar_arrive(empty(s));
                if (++s == p.depth) {
                    s = 0;
                    ph ^= 1u;
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if constexpr (PERCH) {
                    // the offset term o' * sum_k a belongs to the unit once: warp 0 adds it
                    const float o0 = warp == 0 ? fmaf(-kBias, tp0.y, tp0.x) : 0.f;
                    const float o1 = warp == 0 ? fmaf(-kBias, tp1.y, tp1.x) : 0.f;
                    acc[nt][0] = fmaf(o0, stot[nt].x, tp0.y * dp[nt][0]);
                    acc[nt][1] = fmaf(o0, stot[nt].y, tp0.y * dp[nt][1]);
                    acc[nt][2] = fmaf(o1, stot[nt].x, tp1.y * dp[nt][2]);
                    acc[nt][3] = fmaf(o1, stot[nt].y, tp1.y * dp[nt][3]);
                }
                *reinterpret_cast<float4*>(red + (((size_t)(r * kCWarps + warp) * NT + nt) * 32 + lane) * 4) =
                    make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
            }
        }
        // fixed-order sum of the 16 warps' partials of the round's units
        consumer_sync();
        for (int idx = threadIdx.x; idx < kRed * NT * 128; idx += kCWarps * 32) {   // (unit r, tile nt, lane ln, element cc)
            const int r = idx / (NT * 128), nt = (idx / 128) % NT, ln = (idx >> 2) & 31, cc = idx & 3;
            const int row = (int)blockIdx.x * kRows + (ui0 + r) * n_step + (ln >> 2) + (cc >= 2 ? 8 : 0);
            const int m = nt * 8 + 2 * (ln & 3) + (cc & 1);
            if (r < nr && row < p.N && m < p.M && ok) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kCWarps; ++w) sum += red[(((size_t)(r * kCWarps + w) * NT + nt) * 32 + ln) * 4 + cc];
                if (gridDim.y > 1)
                    p.partial[((size_t)blockIdx.y * p.M + m) * p.N + row] = sum;
                else
                {
                    const size_t mn = (size_t)m * p.N + row;
                    if constexpr (EP) sum = epilogue_apply_rt(p.ep, sum, mn, row, p.cdt);
                    store_out_rt(p.C, mn, sum, p.cdt);
                }
            }
        }
        consumer_sync();
    }
}

// ---------------------------------------------------------------- host side
struct Plan {
    Params p;
    size_t smem;
};

// Packed bytes per 64-wide sub-block of a row.
inline int sb_bytes(int fmt) { return fmt == FMT_INT4 ? 32 : (fmt == FMT_INT8 ? 64 : 128); }

// Bytes of one ring stage: the weight box plus the table entries a stage can need.
inline int stage_bytes_for(int fmt, int K, int block) {
    int table = 0;
    if (fmt != FMT_FLOAT) {
        const int sps = kSliceBytes / sb_bytes(fmt), spb = block / 64, nb = K / block;
        const int ent_bound = (kCWarps * sps - 1) / spb + 2;
        table = 128 * (nb < ent_bound ? nb : ent_bound);
    }
    return (kWStage + table + 1023) / 1024 * 1024;
}

// Ring depth that fits beside the fixed shared memory of NT column tiles (0 if fewer than 2).
template <int NT>
inline int ring_depth(int fmt, int K, int block) {
    const int d = (int)((kMaxSmem - Budget<NT>::kFixedBytes) / (size_t)stage_bytes_for(fmt, K, block));
    return d < 2 ? 0 : (d < kMaxDepth ? d : kMaxDepth);
}

// True if this kernel takes the shape: at most 16 rows of A, packed rows a multiple of 128 bytes,
// and (for two column tiles) at least two ring stages beside the fragments. Shapes it takes run
// with at most 64 sub-blocks per thread block (the split-K rule in decode.cu uses this).
inline bool stream_takes(int M, int K, int fmt, int block) {
    if (M < 1 || M > 16 || ((long long)(K / 64) * sb_bytes(fmt)) % kSliceBytes != 0) return false;
    return M <= 8 ? ring_depth<1>(fmt, K, block) > 0 : ring_depth<2>(fmt, K, block) > 0;
}


// Ring geometry for a launch with `splits` K-splits; false if the shape does not fit.
template <int FMT, int NT>
bool make_plan(const DecodeArgs& a, Plan* out) {
    using G = Geo<FMT>;
    Params& p = out->p;
    p = Params{};
    p.M = a.M; p.K = a.K; p.N = a.N;
    p.nsb = a.K / 64;
    p.nsl = (p.nsb + G::kSps - 1) / G::kSps;
    p.sb_per_blk = a.block / 64;
    p.nb = a.K / a.block;
    const int sl_split = (p.nsl + a.splits - 1) / a.splits;
    p.bz = sl_split < kCWarps ? sl_split : kCWarps;
    p.chunks = (sl_split + p.bz - 1) / p.bz;
    if (p.chunks > G::kChunks) return false;
    p.row_bytes = p.nsb * G::kSbBytes;
    if (p.row_bytes % kSliceBytes != 0) return false;
    p.stage_bytes = stage_bytes_for(FMT, a.K, a.block);
    p.depth = ring_depth<NT>(FMT, a.K, a.block);
    if (p.depth < 2) return false;
    out->smem = (size_t)p.depth * p.stage_bytes + Budget<NT>::kFixedBytes;
    return true;
}

// The packed weights [N][row bytes] as the 3-D byte tensor {128, N (stride row bytes), row bytes /
// 128 (stride 128)}; box {128, 16, bz} with the 128-byte swizzle; rows past N read 0.
inline cudaError_t make_wmap(CUtensorMap* map, const void* Bp, int row_bytes, int N, int bz) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)kSliceBytes, (cuuint64_t)N, (cuuint64_t)(row_bytes / kSliceBytes)};
    const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)kSliceBytes};
    const cuuint32_t box[3] = {(cuuint32_t)kSliceBytes, (cuuint32_t)kRows, (cuuint32_t)bz};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(Bp), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int FMT>
inline bool supported(const DecodeArgs& a) {
    return stream_takes(a.M, a.K, FMT, a.block);
}

template <int FMT, bool BF, bool PERCH, bool EP, bool ONECOL, int NT>
cudaError_t launch_v(const DecodeArgs& a, cudaStream_t s) {
    Plan plan;
    if (!make_plan<FMT, NT>(a, &plan)) return cudaErrorInvalidValue;
    plan.p.A = a.A;
    plan.p.Bp = static_cast<const uint8_t*>(a.Bp);
    plan.p.T = a.T;
    plan.p.C = a.C;
    plan.p.partial = a.partial;
    plan.p.ep = a.ep;
    plan.p.cdt = a.c_dtype;
    plan.p.status = status_word_address();
    if (!plan.p.status) return cudaErrorInvalidValue;
    plan.p.wait_ns = option_wait_ns();
    plan.p.stall = option_stall();
    CUtensorMap wmap;
    cudaError_t e = make_wmap(&wmap, a.Bp, plan.p.row_bytes, a.N, plan.p.bz);
    if (e != cudaSuccess) return e;
    auto kern = stream_kernel<FMT, BF, PERCH, EP, ONECOL, NT>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem);
    if (e != cudaSuccess) return e;
    const int groups = (a.N + kRows - 1) / kRows;
    const int sms = dec::sm_count();
    const int per_split = sms / a.splits > 0 ? sms / a.splits : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(groups < per_split ? groups : per_split, a.splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, wmap, plan.p);
}

// The fused epilogue gets its own instantiation (EP), so that the plain store path is unchanged;
// split partials never take it (the reduction applies it).
template <int FMT, bool BF, bool PERCH, bool ONECOL, int NT>
cudaError_t launch_c(const DecodeArgs& a, cudaStream_t s) {
    if (a.splits == 1 && a.ep.any()) return launch_v<FMT, BF, PERCH, true, ONECOL, NT>(a, s);
    return launch_v<FMT, BF, PERCH, false, ONECOL, NT>(a, s);
}

// Shapes stream_takes accepts (M <= 16)
template <int FMT, bool BF>
cudaError_t launch_fmt(const DecodeArgs& a, cudaStream_t s) {
    constexpr bool kPerch = FMT != FMT_FLOAT;   // the per-channel specialization exists for tabled formats
    const bool perch = kPerch && a.block == a.K;
    if (a.M == 1) return perch ? launch_c<FMT, BF, kPerch, true, 1>(a, s) : launch_c<FMT, BF, false, true, 1>(a, s);
    if (a.M <= 8) return perch ? launch_c<FMT, BF, kPerch, false, 1>(a, s) : launch_c<FMT, BF, false, false, 1>(a, s);
    return perch ? launch_c<FMT, BF, kPerch, false, 2>(a, s) : launch_c<FMT, BF, false, false, 2>(a, s);
}

}  // namespace dstream
}  // namespace qg
