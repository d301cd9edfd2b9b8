// Internal launch interface between the C ABI (qgemm_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qg {

enum Fmt { FMT_FLOAT = 0, FMT_INT4 = 1, FMT_INT8 = 2 };
enum Dt { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

inline size_t dt_size(int dt) { return dt == DT_F32 ? 4 : 2; }

// Output epilogue (epilogue.cuh): C = act(acc + bias) + residual, applied in float32 before the
// one rounding to C's type. The activation codes are the C ABI's QGEMM_ACT_* values.
enum Act { ACT_NONE = 0, ACT_RELU = 1, ACT_SILU = 2, ACT_GELU_TANH = 3 };
struct Epilogue {
    const float* bias = nullptr;        // [N] float32, or none
    const void* residual = nullptr;     // [M][N] in C's type, or none (may be C itself)
    int act = ACT_NONE;
    __host__ __device__ bool any() const { return bias || residual || act != ACT_NONE; }
};

// The {offset, scale} table T holds one float32 pair per (output channel n, K-block b), stored in
// groups of 16 channels: [ceil(N / 16)][nb][16][2]. The entries of a 16-channel group for a run
// of K-blocks are then one contiguous, 128-byte aligned range (one bulk copy), and the 16
// channels of one K-block are 128 contiguous bytes. Channels past N (up to the next multiple of
// 16) hold zeros. tab_index gives the pair's index (in pairs).
__host__ __device__ __forceinline__ size_t tab_index(int n, int nb, int b) {
    return (((size_t)(n >> 4) * nb + b) << 4) + (n & 15);
}
inline size_t table_pairs(int N, int nb) { return (size_t)((N + 15) / 16) * 16 * nb; }

// SM count the grid heuristics are sized for (GB300: 152 SMs). A constant, so that host-side
// size queries (workspace bytes) give the same answer with or without a GPU present.
constexpr int kTargetSms = 152;

// ---------------------------------------------------------------- pack
cudaError_t launch_quant_pack(const float* W, int K, int N, int block, int nbits, uint8_t* Bp, float* T,
                              cudaStream_t s);
cudaError_t launch_float_pack(const float* W, int K, int N, int w_dtype, void* Bp, cudaStream_t s);

// ---------------------------------------------------------------- decode (M small)
struct DecodeArgs {
    int M, K, N;
    int block;        // K-group size of the table (multiple of 64; == K for per-channel)
    int fmt;          // Fmt
    int a_dtype;      // DT_F16 / DT_BF16 for the tensor-core decode; any for the f32 kernel
    int c_dtype;
    const void* A;
    const void* Bp;
    const float* T;
    void* C;
    float* partial;   // [splits][M][N] f32 partial sums when splits > 1
    int splits;       // number of K-splits across thread blocks (>= 1)
    int overlap;      // launch with a programmatic dependency on the previous kernel
    Epilogue ep;
};
// K-splits the decode kernels use for this shape, at most 16 rows of A (1 = none); block is the
// table's K-group (K for per-channel).
int decode_splits(int M, int K, int N, int fmt, int block);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
// C[i] = epilogue(sum over y = 0 .. splits-1, in that order, of partial[y * count + i]) (float32),
// rounded once to c_dtype; i = m * N + n.
cudaError_t launch_splitk_reduce(const float* partial, int splits, size_t count, int N, const Epilogue& ep, void* C,
                                 int c_dtype, cudaStream_t s);
// Exact float32 CUDA-core kernel (any activation dtype, any M); used for f32 activations.
cudaError_t launch_decode_f32(const DecodeArgs& a, cudaStream_t s);

// ---------------------------------------------------------------- prefill / W4A8
struct PrefillArgs {
    int M, K, N, block, fmt, a_dtype, c_dtype;
    const void* A;
    const void* Bp;
    const float* T;
    void* C;
    float* partial;   // [splits][M][N] f32 partial sums when splits > 1
    int splits;       // K-splits across thread blocks (>= 1), from prefill_splits
    Epilogue ep;
    float* rowsum;    // [M] scratch for the row sums of A (Int8-Block0 on the codes path)
    float* rowmax = nullptr;   // [ceil(N/128)][M] per-tile row maxima of |C| (no K-split), or none
};
// Int8-Block0 (per-channel) layers with bf16 activations and M >= 256 run on the tensor cores as
// raw codes with the scale and offset applied in the epilogue (they need [M] float32 row sums of A
// as scratch): the codes are exact in bf16, so the hi/lo weight split and its second MMA go away
// (measured at M = 1024: 33 us against 44). With f16 activations, or fewer rows, the row-sum
// pre-pass costs more than it saves and the dequantizing path stays.
inline bool prefill_codes_path(int fmt, int K, int block, int M, int a_dtype) {
    return fmt == FMT_INT8 && block == K && a_dtype == DT_BF16 && M >= 256;
}
// K-splits the tensor-core kernel uses for this shape (1 = none); host-only, no GPU needed.
int prefill_splits(int M, int K, int N, int fmt);
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);
bool prefill_supported(int M, int K, int N, int fmt, int a_dtype);

// Per-row activation codes: qa (int8) and/or qa16 (the same codes as exact f16 values; either
// may be null), the row scales and the row sums of the codes.
cudaError_t launch_act_quant(int M, int K, const void* A, int a_dtype, int8_t* qa, void* qa16, float* as,
                             int32_t* rowsum, cudaStream_t s);
cudaError_t launch_codes_to_f16(const int8_t* qa, void* out, size_t n, cudaStream_t s);
// The activation step of a next W4A8 layer applied to C [M][N] (c_dtype) when the row maxima of
// |C| are known per 128-channel tile (rowmax [ntiles][M], from the tensor-core epilogue): codes as
// exact f16 [M][N], scales and code sums; the same codes as launch_act_quant on C. N % 8 == 0.
cudaError_t launch_quant_rows(int M, int N, const void* C, int c_dtype, const float* rowmax, int ntiles,
                              void* qa16, float* as, int32_t* rowsum, cudaStream_t s);
// out[m] = sum_k A[m][k] in float32 (the Int8-Block0 tensor-core path's row sums)
cudaError_t launch_row_sums(int M, int K, const void* A, int a_dtype, float* out, cudaStream_t s);
// acc (int32 [M][N]) = qa x q^T; or, when acc == nullptr, the rescaled output into C.
struct W4A8Args {
    int M, K, N;
    const void* qa16;    // activation codes as f16 [M][K]
    const float* as;
    const int32_t* rowsum;
    const void* Bp;
    const float* T;
    int32_t* acc;   // int32 accumulators out (or nullptr)
    void* C;        // rescaled output (or nullptr)
    int c_dtype;
    Epilogue ep;    // applied to the rescaled output
    int block = 0;  // K-block of the weights' {offset, scale} (0 or K: per channel)
    int splits = 1; // K-chunks (grid z); with acc_add each chunk adds its int32 sums into acc
    int acc_add = 0;
    float* rowmax = nullptr;   // [ceil(N/128)][M] per-tile row maxima of |C| (rescaled output only)
};
cudaError_t launch_w4a8_gemm(const W4A8Args& a, cudaStream_t s);
// The integer sums of the W4A8 tensor-core GEMM are exact while every float32 partial sum is an
// integer below 2^24: |qa| <= 127 and q <= 15 bound a K-chunk's sum by 1905 * chunk, so chunks of
// at most 8808 (8192 used, a multiple of 64) stay exact. Longer K runs as K-chunks whose int32
// sums are added in int32 (exact, in any order).
constexpr int kW4A8ExactK = 8808;
constexpr int kW4A8ChunkK = 8192;
inline int w4a8_exact_splits(int K) { return K <= kW4A8ExactK ? 1 : (K + kW4A8ChunkK - 1) / kW4A8ChunkK; }
// C = epilogue(as[m] * (ws[n] * acc[m][n] + off[n] * rowsum[m])) from int32 accumulators (W4A8 with
// per-channel weights when K was split into exact chunks); T is the grouped table (one block).
cudaError_t launch_w4a8_rescale(int M, int N, const int32_t* acc, const float* as, const int32_t* rowsum,
                                const float* T, const Epilogue& ep, void* C, int c_dtype, cudaStream_t s);

// library options (qgemm_set_option)
int option_overlap();
long long option_wait_ns();   // bound of each pipeline wait in the TMA-fed kernels
int option_stall();           // diagnostic stall of the next launches (QGEMM_OPT_DEBUG_STALL)
// Records `detail` as the thread's last error and returns `code` (the C ABI's error path).
int api_fail(int code, const char* detail);
// Bp bytes of a shape (0 if the shape is invalid) and, in *table_bytes, its T bytes (0 in FLOAT).
size_t api_packed_bytes(int K, int N, int mode, int block, int w_dtype, size_t* table_bytes);

// device status word (bounded waits that gave up); read and cleared by qgemm_status
cudaError_t read_and_clear_status(int* value, cudaStream_t s);
// Device address of the status word on the current device (nullptr if it cannot be had), for
// kernels compiled in other translation units.
unsigned int* status_word_address();

// cuTensorMapEncodeTiled, taken from the driver once (nullptr if the driver lacks it)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

}  // namespace qg
