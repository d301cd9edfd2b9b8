// The C ABI of include/qgemm.h: argument checks, workspace sizing and kernel choice.
// Every check runs before the first launch, so a rejected call enqueues nothing.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "../../include/qgemm.h"
#include "internal.h"

namespace {

thread_local char g_last_error[256] = "";
std::atomic<int> g_opt_overlap{0};
std::atomic<int> g_opt_decode_max_m{16};
std::atomic<int> g_opt_split_k{1};
std::atomic<int> g_opt_wait_us{1000000};
std::atomic<int> g_opt_stall{0};

// QGEMM_OPT_FAULT_INJECT: the n-th compute call from now reports a simulated launch failure.
int fault_from_env() {
    const char* v = getenv("QGEMM_FAULT_INJECT");
    if (!v || !*v) return 0;
    const long n = strtol(v, nullptr, 10);
    return n > 0 && n < 1000000000L ? (int)n : 0;
}
std::atomic<int> g_fault{fault_from_env()};

// Counts one compute call down; true for the call the countdown selected.
bool inject_fault() {
    int v = g_fault.load();
    while (v > 0)
        if (g_fault.compare_exchange_weak(v, v - 1)) return v == 1;
    return false;
}

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(QGEMM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_dtype(int d) { return d == QGEMM_F32 || d == QGEMM_F16 || d == QGEMM_BF16; }
bool valid_mode(int m) { return m >= QGEMM_MODE_FLOAT && m <= QGEMM_MODE_W4A8; }

// Checks shared by pack and run; `block` is normalised (0 -> K). Returns QGEMM_OK or a code.
int check_shape(int K, int N, int mode, int* block) {
    if (!valid_mode(mode)) return fail(QGEMM_ERR_ARG, "unknown mode %d", mode);
    if (K <= 0 || N < 0) return fail(QGEMM_ERR_ARG, "invalid sizes K=%d N=%d", K, N);
    if (K % 64 != 0) return fail(QGEMM_ERR_UNSUPPORTED, "K=%d is not a multiple of 64", K);
    if (*block < 0) return fail(QGEMM_ERR_ARG, "negative block %d", *block);
    if (*block == 0) *block = K;
    if (mode == QGEMM_MODE_FLOAT) return QGEMM_OK;
    if (*block % 64 != 0 || K % *block != 0)
        return fail(QGEMM_ERR_UNSUPPORTED, "block %d must be a multiple of 64 dividing K=%d", *block, K);
    return QGEMM_OK;
}

size_t packed_bytes(int K, int N, int mode, int w_dtype) {
    switch (mode) {
        case QGEMM_MODE_FLOAT: return (size_t)K * N * qg::dt_size(w_dtype);
        case QGEMM_MODE_INT8: return (size_t)K * N;
        default: return (size_t)K * N / 2;
    }
}

// W4A8 workspace: the activation codes as f16 [M][K] (exact integers, the tensor cores' operand
// type), then as [M] f32 and rowsum [M] int32, each 256-byte aligned; with per-channel weights and
// K beyond the exact range of one float32 accumulation (qg::w4a8_exact_splits), then the int32
// accumulators [M][N] that the K-chunks add into.
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
bool w4a8_chunked(int K, int block) { return block == K && qg::w4a8_exact_splits(K) > 1; }
size_t w4a8_ws(int M, int K, int N, int block) {
    return align256((size_t)M * K * 2) + align256((size_t)M * 4) * 2 +
           (w4a8_chunked(K, block) ? align256((size_t)M * N * 4) : 0);
}
// Largest K whose int32 accumulators cannot overflow: |qa| * q <= 127 * 15 per term.
constexpr int kW4A8MaxK = 2147483647 / (127 * 15);

int fmt_of(int mode) {
    return mode == QGEMM_MODE_FLOAT ? qg::FMT_FLOAT : (mode == QGEMM_MODE_INT8 ? qg::FMT_INT8 : qg::FMT_INT4);
}

// Kernel choice by shape (one backend: these are all this library's CUDA kernels).
enum Path { PATH_F32, PATH_DECODE, PATH_PREFILL };
Path choose_path(int M, int K, int N, int mode, int a_dtype) {
    if (a_dtype == QGEMM_F32) return PATH_F32;
    if (M > g_opt_decode_max_m.load(std::memory_order_relaxed) && qg::prefill_supported(M, K, N, fmt_of(mode), a_dtype))
        return PATH_PREFILL;
    return PATH_DECODE;
}

// K-splits of the tensor-core path for this call: the shape's choice, lowered until the float32
// partial sums [splits][M][N] fit in ws_bytes of scratch.
int prefill_splits_for(int M, int K, int N, int mode, size_t ws_bytes) {
    if (!g_opt_split_k.load(std::memory_order_relaxed)) return 1;
    int splits = qg::prefill_splits(M, K, N, fmt_of(mode));
    const size_t per = (size_t)M * N * sizeof(float);
    while (splits > 1 && (size_t)splits * per > ws_bytes) --splits;
    return splits;
}

// Row-sum scratch of the tensor-core path for Int8-Block0 (float32 [M], 256-byte aligned), in
// front of any split-K partials.
size_t rowsum_ws(int M, int K, int mode, int block, int a_dtype) {
    return qg::prefill_codes_path(fmt_of(mode), K, block, M, a_dtype) ? align256((size_t)M * sizeof(float)) : 0;
}

// Scratch bytes of a call. The decode split-K partials, the W4A8 codes and the Int8-Block0 row
// sums are required; the tensor-core path's split-K partials are optional (with less scratch it
// splits less), so `required` leaves them out.
size_t run_ws(int M, int K, int N, int mode, int block, int a_dtype, bool required) {
    if (mode == QGEMM_MODE_W4A8) return w4a8_ws(M, K, N, block);
    const Path path = choose_path(M, K, N, mode, a_dtype);
    if (path == PATH_PREFILL) {
        const size_t rows = rowsum_ws(M, K, mode, block, a_dtype);
        if (required) return rows;
        const int splits = prefill_splits_for(M, K, N, mode, SIZE_MAX);
        return rows + (splits > 1 ? (size_t)splits * M * N * sizeof(float) : 0);
    }
    if (path != PATH_DECODE) return 0;
    // the decode kernel runs 16 rows of A at a time; split-K partials are per 16-row launch
    const int mc = M < 16 ? M : 16;
    const int splits = qg::decode_splits(mc, K, N, fmt_of(mode), block == 0 ? K : block);
    return splits > 1 ? (size_t)splits * mc * N * sizeof(float) : 0;
}

// Checks shared by the layer calls (block normalised); QGEMM_OK for an empty call too.
int check_run(int M, int K, int N, int mode, int* block, const void* A, int a_dtype, const void* Bp, const float* T,
              const float* bias, int act, const void* residual, const void* C, int c_dtype, const void* workspace) {
    int rc = check_shape(K, N, mode, block);
    if (rc != QGEMM_OK) return rc;
    if (M < 0) return fail(QGEMM_ERR_ARG, "negative M=%d", M);
    if (!valid_dtype(a_dtype) || !valid_dtype(c_dtype))
        return fail(QGEMM_ERR_ARG, "unknown dtype (a_dtype %d, c_dtype %d)", a_dtype, c_dtype);
    if (act < QGEMM_ACT_NONE || act > QGEMM_ACT_GELU_TANH) return fail(QGEMM_ERR_ARG, "unknown activation %d", act);
    if (M == 0 || N == 0) return QGEMM_OK;
    if (!A || !Bp || !C) return fail(QGEMM_ERR_ARG, "null A, Bp or C");
    if (mode != QGEMM_MODE_FLOAT && !T) return fail(QGEMM_ERR_ARG, "null T");
    if (!aligned16(A) || !aligned16(Bp) || !aligned16(C) || (T && !aligned16(T)) ||
        (workspace && !aligned16(workspace)) || (bias && !aligned16(bias)) || (residual && !aligned16(residual)))
        return fail(QGEMM_ERR_ALIGN, "A, Bp, T, C, bias, residual and workspace must be 16-byte aligned");
    if ((M + 15) / 16 > 65535) return fail(QGEMM_ERR_UNSUPPORTED, "M=%d exceeds the launch limit", M);
    if (mode == QGEMM_MODE_W4A8 && K > kW4A8MaxK)
        return fail(QGEMM_ERR_UNSUPPORTED, "W4A8 with K=%d could overflow the int32 accumulators", K);
    return QGEMM_OK;
}

qg::Epilogue make_ep(const float* bias, int act, const void* residual) {
    qg::Epilogue ep;
    ep.bias = bias;
    ep.residual = residual;
    ep.act = act;
    return ep;
}

// The W4A8 GEMM from activation codes (exact f16 [M][K]), row scales and code sums: one launch,
// or (per-channel weights, K past the exact range) int32 K-chunks added in acc_ws [M][N], then the
// rescale. rowmax (one launch only): the epilogue's per-tile row maxima of |C|.
int w4a8_from_codes(int M, int K, int N, int block, const void* qa16, const float* as, const int32_t* rs,
                    const void* Bp, const float* T, const qg::Epilogue& ep, void* C, int c_dtype, int32_t* acc_ws,
                    float* rowmax, cudaStream_t s) {
    cudaError_t e;
    if (w4a8_chunked(K, block)) {
        e = cudaMemsetAsync(acc_ws, 0, (size_t)M * N * sizeof(int32_t), s);
        if (e != cudaSuccess) return cuda_fail(e, "accumulator clear");
        qg::W4A8Args w{M, K, N, qa16, nullptr, nullptr, Bp, nullptr, acc_ws, nullptr, QGEMM_F32};
        w.splits = qg::w4a8_exact_splits(K);
        w.acc_add = 1;
        e = qg::launch_w4a8_gemm(w, s);
        if (e != cudaSuccess) return cuda_fail(e, "w4a8 gemm launch");
        e = qg::launch_w4a8_rescale(M, N, acc_ws, as, rs, T, ep, C, c_dtype, s);
        return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "w4a8 rescale launch");
    }
    qg::W4A8Args w{M, K, N, qa16, as, rs, Bp, T, nullptr, C, c_dtype, ep, block};
    w.rowmax = rowmax;
    e = qg::launch_w4a8_gemm(w, s);
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "w4a8 gemm launch");
}

// The launches of one layer call (every check done). rowmax: when set, the tensor-core epilogue
// writes its per-tile row maxima of |C| there, and the call does not split K.
int launch_layer(int M, int K, int N, int mode, int block, const void* A, int a_dtype, const void* Bp,
                 const float* T, const qg::Epilogue& ep, void* C, int c_dtype, void* workspace, size_t workspace_bytes,
                 float* rowmax, cudaStream_t s) {
    cudaError_t e;
    if (mode == QGEMM_MODE_W4A8) {
        void* qa16 = workspace;
        float* as = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256((size_t)M * K * 2));
        int32_t* rs = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(as) + align256((size_t)M * 4));
        e = qg::launch_act_quant(M, K, A, a_dtype, nullptr, qa16, as, rs, s);
        if (e != cudaSuccess) return cuda_fail(e, "act_quant launch");
        int32_t* acc = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(rs) + align256((size_t)M * 4));
        return w4a8_from_codes(M, K, N, block, qa16, as, rs, Bp, T, ep, C, c_dtype, acc, rowmax, s);
    }
    const int fmt = fmt_of(mode);
    const Path path = choose_path(M, K, N, mode, a_dtype);
    if (path == PATH_PREFILL) {
        const size_t rows = rowsum_ws(M, K, mode, block, a_dtype);   // [row sums][split-K partials]
        qg::PrefillArgs pa{M, K, N, block, fmt, a_dtype, c_dtype, A, Bp, T, C,
                           rows ? reinterpret_cast<float*>(static_cast<char*>(workspace) + rows)
                                : static_cast<float*>(workspace),
                           1, ep, static_cast<float*>(workspace)};
        pa.splits = rowmax ? 1 : prefill_splits_for(M, K, N, mode, workspace ? workspace_bytes - rows : 0);
        pa.rowmax = rowmax;
        e = qg::launch_prefill(pa, s);
        return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "prefill launch");
    }
    qg::DecodeArgs da{};
    da.M = M; da.K = K; da.N = N; da.block = block; da.fmt = fmt;
    da.a_dtype = a_dtype; da.c_dtype = c_dtype;
    da.A = A; da.Bp = Bp; da.T = T; da.C = C;
    da.ep = ep;
    if (path == PATH_F32) {
        da.splits = 1;
        e = qg::launch_decode_f32(da, s);
        return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "decode_f32 launch");
    }
    da.splits = 1;   // chosen per 16-row launch inside launch_decode
    da.overlap = qg::option_overlap();
    da.partial = static_cast<float*>(workspace);
    e = qg::launch_decode(da, s);
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "decode launch");
}

// Workspace of qgemm_run_fused_quant: the layer's own required scratch (no tensor-core K-split),
// then, where the layer runs on the tensor-core kernel in one launch, the per-tile row maxima
// [ceil(N/128)][M] float32 (256-byte aligned).
struct FqLayout {
    bool rowmax;
    size_t parts_off, total;
};
FqLayout fq_layout(int M, int K, int N, int mode, int block, int a_dtype) {
    FqLayout L{};
    L.rowmax = mode == QGEMM_MODE_W4A8 ? !w4a8_chunked(K, block)
                                       : choose_path(M, K, N, mode, a_dtype) == PATH_PREFILL;
    const size_t layer = run_ws(M, K, N, mode, block, a_dtype, true);
    if (!L.rowmax) {
        L.total = layer;
        return L;
    }
    L.parts_off = align256(layer);
    L.total = L.parts_off + align256((size_t)((N + 127) / 128) * M * sizeof(float));
    return L;
}

}  // namespace

int qg::option_overlap() { return g_opt_overlap.load(std::memory_order_relaxed); }
long long qg::option_wait_ns() { return 1000LL * g_opt_wait_us.load(std::memory_order_relaxed); }
int qg::option_stall() { return g_opt_stall.load(std::memory_order_relaxed); }

int qg::api_fail(int code, const char* detail) { return fail(code, "%s", detail); }
size_t qg::api_packed_bytes(int K, int N, int mode, int block, int w_dtype, size_t* table_bytes) {
    *table_bytes = 0;
    if (check_shape(K, N, mode, &block) != QGEMM_OK) return 0;
    if (mode == QGEMM_MODE_FLOAT && !valid_dtype(w_dtype)) return 0;
    if (mode != QGEMM_MODE_FLOAT) *table_bytes = qg::table_pairs(N, K / block) * 2 * sizeof(float);
    return packed_bytes(K, N, mode, w_dtype);
}

extern "C" {

int qgemm_set_option(int option, int value) {
    if (option == QGEMM_OPT_LAUNCH_OVERLAP) {
        if (value != 0 && value != 1) return fail(QGEMM_ERR_ARG, "option %d takes 0 or 1, got %d", option, value);
        return g_opt_overlap.exchange(value);
    }
    if (option == QGEMM_OPT_DECODE_MAX_M) {
        if (value < 16 || value > 1024) return fail(QGEMM_ERR_ARG, "option %d takes 16..1024, got %d", option, value);
        return g_opt_decode_max_m.exchange(value);
    }
    if (option == QGEMM_OPT_SPLIT_K) {
        if (value != 0 && value != 1) return fail(QGEMM_ERR_ARG, "option %d takes 0 or 1, got %d", option, value);
        return g_opt_split_k.exchange(value);
    }
    if (option == QGEMM_OPT_WAIT_LIMIT_US) {
        if (value < 1 || value > 1000000)
            return fail(QGEMM_ERR_ARG, "option %d takes 1..1000000 (microseconds), got %d", option, value);
        return g_opt_wait_us.exchange(value);
    }
    if (option == QGEMM_OPT_DEBUG_STALL) {
        if (value != 0 && value != 1) return fail(QGEMM_ERR_ARG, "option %d takes 0 or 1, got %d", option, value);
        return g_opt_stall.exchange(value);
    }
    if (option == QGEMM_OPT_FAULT_INJECT) {
        if (value < 0) return fail(QGEMM_ERR_ARG, "option %d takes a count >= 0, got %d", option, value);
        return g_fault.exchange(value);
    }
    return fail(QGEMM_ERR_ARG, "unknown option %d", option);
}

int qgemm_get_option(int option) {
    if (option == QGEMM_OPT_LAUNCH_OVERLAP) return g_opt_overlap.load();
    if (option == QGEMM_OPT_DECODE_MAX_M) return g_opt_decode_max_m.load();
    if (option == QGEMM_OPT_SPLIT_K) return g_opt_split_k.load();
    if (option == QGEMM_OPT_WAIT_LIMIT_US) return g_opt_wait_us.load();
    if (option == QGEMM_OPT_DEBUG_STALL) return g_opt_stall.load();
    if (option == QGEMM_OPT_FAULT_INJECT) return g_fault.load();
    return fail(QGEMM_ERR_ARG, "unknown option %d", option);
}

size_t qgemm_packed_bytes(int K, int N, int mode, int w_dtype) {
    int block = 0;
    if (check_shape(K, N, mode, &block) != QGEMM_OK) return 0;
    if (mode == QGEMM_MODE_FLOAT && !valid_dtype(w_dtype)) return 0;
    return packed_bytes(K, N, mode, w_dtype);
}

size_t qgemm_table_bytes(int K, int N, int mode, int block) {
    if (check_shape(K, N, mode, &block) != QGEMM_OK || mode == QGEMM_MODE_FLOAT) return 0;
    return qg::table_pairs(N, K / block) * 2 * sizeof(float);
}

size_t qgemm_workspace_bytes(int M, int K, int N, int mode, int block, int a_dtype, int c_dtype) {
    if (M <= 0 || check_shape(K, N, mode, &block) != QGEMM_OK || !valid_dtype(a_dtype) || !valid_dtype(c_dtype))
        return 0;
    return run_ws(M, K, N, mode, block, a_dtype, false);
}

int qgemm_pack(const float* W, int K, int N, int mode, int block, int w_dtype, void* Bp, float* T, void* stream) {
    int rc = check_shape(K, N, mode, &block);
    if (rc != QGEMM_OK) return rc;
    if (N == 0) return QGEMM_OK;
    if (!W || !Bp) return fail(QGEMM_ERR_ARG, "null W or Bp");
    if (!aligned16(W) || !aligned16(Bp)) return fail(QGEMM_ERR_ALIGN, "W and Bp must be 16-byte aligned");
    if (mode == QGEMM_MODE_FLOAT && !valid_dtype(w_dtype)) return fail(QGEMM_ERR_ARG, "unknown w_dtype %d", w_dtype);
    if (mode != QGEMM_MODE_FLOAT) {
        if (!T) return fail(QGEMM_ERR_ARG, "null T");
        if (!aligned16(T)) return fail(QGEMM_ERR_ALIGN, "T must be 16-byte aligned");
        if ((size_t)(K / block) > 65535) return fail(QGEMM_ERR_UNSUPPORTED, "too many blocks per channel");
    }
    if (inject_fault()) return fail(QGEMM_ERR_CUDA, "simulated launch failure (fault injection)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (mode == QGEMM_MODE_FLOAT) {
        e = qg::launch_float_pack(W, K, N, w_dtype, Bp, s);
    } else {
        e = qg::launch_quant_pack(W, K, N, block, mode == QGEMM_MODE_INT8 ? 8 : 4, static_cast<uint8_t*>(Bp), T, s);
    }
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "qgemm_pack launch");
}

int qgemm_run(int M, int K, int N, int mode, int block, const void* A, int a_dtype, const void* Bp, const float* T,
              void* C, int c_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    return qgemm_run_fused(M, K, N, mode, block, A, a_dtype, Bp, T, nullptr, QGEMM_ACT_NONE, nullptr, C, c_dtype,
                           workspace, workspace_bytes, stream);
}

int qgemm_run_fused(int M, int K, int N, int mode, int block, const void* A, int a_dtype, const void* Bp,
                    const float* T, const float* bias, int act, const void* residual, void* C, int c_dtype,
                    void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_run(M, K, N, mode, &block, A, a_dtype, Bp, T, bias, act, residual, C, c_dtype, workspace);
    if (rc != QGEMM_OK || M == 0 || N == 0) return rc;
    const size_t need = run_ws(M, K, N, mode, block, a_dtype, true);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(QGEMM_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (inject_fault()) return fail(QGEMM_ERR_CUDA, "simulated launch failure (fault injection)");
    return launch_layer(M, K, N, mode, block, A, a_dtype, Bp, T, make_ep(bias, act, residual), C, c_dtype, workspace,
                        workspace_bytes, nullptr, static_cast<cudaStream_t>(stream));
}

size_t qgemm_fused_quant_workspace_bytes(int M, int K, int N, int mode, int block, int a_dtype, int c_dtype) {
    if (M <= 0 || check_shape(K, N, mode, &block) != QGEMM_OK || !valid_dtype(a_dtype) || !valid_dtype(c_dtype) ||
        N % 64 != 0)
        return 0;
    return fq_layout(M, K, N, mode, block, a_dtype).total;
}

int qgemm_run_fused_quant(int M, int K, int N, int mode, int block, const void* A, int a_dtype, const void* Bp,
                          const float* T, const float* bias, int act, const void* residual, void* C, int c_dtype,
                          void* qa_next, float* as_next, int32_t* rowsum_next, void* workspace, size_t workspace_bytes,
                          void* stream) {
    int rc = check_run(M, K, N, mode, &block, A, a_dtype, Bp, T, bias, act, residual, C, c_dtype, workspace);
    if (rc != QGEMM_OK) return rc;
    if (N % 64 != 0)
        return fail(QGEMM_ERR_UNSUPPORTED, "N=%d: the next layer's K must be a multiple of 64", N);
    if (M == 0 || N == 0) return QGEMM_OK;
    if (!qa_next || !as_next || !rowsum_next) return fail(QGEMM_ERR_ARG, "null qa_next, as_next or rowsum_next");
    if (!aligned16(qa_next) || !aligned16(as_next) || !aligned16(rowsum_next))
        return fail(QGEMM_ERR_ALIGN, "qa_next, as_next and rowsum_next must be 16-byte aligned");
    const FqLayout L = fq_layout(M, K, N, mode, block, a_dtype);
    if (L.total > 0 && (!workspace || workspace_bytes < L.total))
        return fail(QGEMM_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", L.total,
                    workspace ? workspace_bytes : (size_t)0);
    if (inject_fault()) return fail(QGEMM_ERR_CUDA, "simulated launch failure (fault injection)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* parts = L.rowmax ? reinterpret_cast<float*>(static_cast<char*>(workspace) + L.parts_off) : nullptr;
    rc = launch_layer(M, K, N, mode, block, A, a_dtype, Bp, T, make_ep(bias, act, residual), C, c_dtype, workspace,
                      L.rowmax ? L.parts_off : workspace_bytes, parts, s);
    if (rc != QGEMM_OK) return rc;
    // the next layer's activation step on C: from the epilogue's row maxima (one read of C), or,
    // where the layer's kernel has no such epilogue, the standalone pass (same codes)
    const cudaError_t e =
        L.rowmax ? qg::launch_quant_rows(M, N, C, c_dtype, parts, (N + 127) / 128, qa_next, as_next, rowsum_next, s)
                 : qg::launch_act_quant(M, N, C, c_dtype, nullptr, qa_next, as_next, rowsum_next, s);
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "activation step launch");
}

size_t qgemm_w4a8_codes_workspace_bytes(int M, int K, int N, int block) {
    if (M <= 0 || check_shape(K, N, QGEMM_MODE_W4A8, &block) != QGEMM_OK) return 0;
    return w4a8_chunked(K, block) ? align256((size_t)M * N * 4) : 0;
}

int qgemm_run_w4a8_codes(int M, int K, int N, int block, const void* qa, const float* a_scale, const int32_t* rowsum,
                         const void* Bp, const float* T, const float* bias, int act, const void* residual, void* C,
                         int c_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_run(M, K, N, QGEMM_MODE_W4A8, &block, qa, QGEMM_F16, Bp, T, bias, act, residual, C, c_dtype,
                       workspace);
    if (rc != QGEMM_OK || M == 0 || N == 0) return rc;
    if (!a_scale || !rowsum) return fail(QGEMM_ERR_ARG, "null a_scale or rowsum");
    if (!aligned16(a_scale) || !aligned16(rowsum)) return fail(QGEMM_ERR_ALIGN, "a_scale and rowsum must be 16-byte aligned");
    const size_t need = w4a8_chunked(K, block) ? align256((size_t)M * N * 4) : 0;
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(QGEMM_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (inject_fault()) return fail(QGEMM_ERR_CUDA, "simulated launch failure (fault injection)");
    return w4a8_from_codes(M, K, N, block, qa, a_scale, rowsum, Bp, T, make_ep(bias, act, residual), C, c_dtype,
                           static_cast<int32_t*>(workspace), nullptr, static_cast<cudaStream_t>(stream));
}

int qgemm_act_quant(int M, int K, const void* A, int a_dtype, int8_t* qa, float* a_scale, int32_t* rowsum,
                    void* stream) {
    if (M < 0 || K <= 0) return fail(QGEMM_ERR_ARG, "invalid sizes M=%d K=%d", M, K);
    if (K % 64 != 0) return fail(QGEMM_ERR_UNSUPPORTED, "K=%d is not a multiple of 64", K);
    if (!valid_dtype(a_dtype)) return fail(QGEMM_ERR_ARG, "unknown a_dtype %d", a_dtype);
    if (M == 0) return QGEMM_OK;
    if (!A || !qa || !a_scale || !rowsum) return fail(QGEMM_ERR_ARG, "null pointer");
    if (!aligned16(A) || !aligned16(qa) || !aligned16(a_scale) || !aligned16(rowsum))
        return fail(QGEMM_ERR_ALIGN, "pointers must be 16-byte aligned");
    if (inject_fault()) return fail(QGEMM_ERR_CUDA, "simulated launch failure (fault injection)");
    cudaError_t e =
        qg::launch_act_quant(M, K, A, a_dtype, qa, nullptr, a_scale, rowsum, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "act_quant launch");
}

size_t qgemm_w4a8_acc_workspace_bytes(int M, int K) {
    if (M <= 0 || K <= 0) return 0;
    return (size_t)M * K * 2;
}

int qgemm_w4a8_acc(int M, int K, int N, const int8_t* qa, const void* Bp, int32_t* acc, void* workspace,
                   size_t workspace_bytes, void* stream) {
    int block = 0;
    int rc = check_shape(K, N, QGEMM_MODE_W4A8, &block);
    if (rc != QGEMM_OK) return rc;
    if (M < 0) return fail(QGEMM_ERR_ARG, "negative M=%d", M);
    if (K > kW4A8MaxK) return fail(QGEMM_ERR_UNSUPPORTED, "K=%d could overflow the int32 accumulators", K);
    if (M == 0 || N == 0) return QGEMM_OK;
    if (!qa || !Bp || !acc) return fail(QGEMM_ERR_ARG, "null pointer");
    if (!aligned16(qa) || !aligned16(Bp) || !aligned16(acc) || (workspace && !aligned16(workspace)))
        return fail(QGEMM_ERR_ALIGN, "pointers must be 16-byte aligned");
    const size_t need = qgemm_w4a8_acc_workspace_bytes(M, K);
    if (!workspace || workspace_bytes < need)
        return fail(QGEMM_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (inject_fault()) return fail(QGEMM_ERR_CUDA, "simulated launch failure (fault injection)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = qg::launch_codes_to_f16(qa, workspace, (size_t)M * K, s);
    if (e != cudaSuccess) return cuda_fail(e, "codes_to_f16 launch");
    qg::W4A8Args w{M, K, N, workspace, nullptr, nullptr, Bp, nullptr, acc, nullptr, QGEMM_F32};
    w.splits = qg::w4a8_exact_splits(K);
    if (w.splits > 1) {   // K-chunks, each exact in float32, added into acc in int32
        e = cudaMemsetAsync(acc, 0, (size_t)M * N * sizeof(int32_t), s);
        if (e != cudaSuccess) return cuda_fail(e, "accumulator clear");
        w.acc_add = 1;
    }
    e = qg::launch_w4a8_gemm(w, s);
    return e == cudaSuccess ? QGEMM_OK : cuda_fail(e, "w4a8 gemm launch");
}

int qgemm_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int v = 0;
    e = qg::read_and_clear_status(&v, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (v & 1) return fail(QGEMM_ERR_TIMEOUT, "a kernel gave up a bounded wait (status word 0x%x)", v);
    if (v != 0) return fail(QGEMM_ERR_CUDA, "a kernel found its shared memory misaligned and did no work (status word 0x%x)", v);
    return QGEMM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- the no-allocation variant
namespace {

// Scratch for qgemm_run_noalloc: one fixed array in every device that loads the library.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QGEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(QGEMM_ERR_UNSUPPORTED, "device %d beyond the supported %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the scratch array");
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return QGEMM_OK;
}

}  // namespace

extern "C" {

int qgemm_run_noalloc(int M, int K, int N, int mode, int block, const void* A, int a_dtype, const void* Bp,
                      const float* T, void* C, int c_dtype, void* stream) {
    // the same checks qgemm_run makes, so the size test below sees a valid shape
    int blk = block;
    int rc = check_shape(K, N, mode, &blk);
    if (rc != QGEMM_OK) return rc;
    if (M < 0) return fail(QGEMM_ERR_ARG, "negative M=%d", M);
    if (!valid_dtype(a_dtype) || !valid_dtype(c_dtype))
        return fail(QGEMM_ERR_ARG, "unknown dtype (a_dtype %d, c_dtype %d)", a_dtype, c_dtype);
    if (M == 0 || N == 0) return QGEMM_OK;
    const size_t need = run_ws(M, K, N, mode, blk, a_dtype, true);
    if (need > QGEMM_NOALLOC_SCRATCH_BYTES)
        return fail(QGEMM_ERR_WORKSPACE, "this call needs %zu bytes of scratch; the built-in scratch holds %u", need,
                    QGEMM_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != QGEMM_OK) return rc;
    return qgemm_run(M, K, N, mode, block, A, a_dtype, Bp, T, C, c_dtype, scratch, QGEMM_NOALLOC_SCRATCH_BYTES,
                     stream);
}

const char* qgemm_error_string(int code) {
    switch (code) {
        case QGEMM_OK: return "QGEMM_OK";
        case QGEMM_ERR_ARG: return "QGEMM_ERR_ARG";
        case QGEMM_ERR_UNSUPPORTED: return "QGEMM_ERR_UNSUPPORTED";
        case QGEMM_ERR_ALIGN: return "QGEMM_ERR_ALIGN";
        case QGEMM_ERR_WORKSPACE: return "QGEMM_ERR_WORKSPACE";
        case QGEMM_ERR_CUDA: return "QGEMM_ERR_CUDA";
        case QGEMM_ERR_TIMEOUT: return "QGEMM_ERR_TIMEOUT";
        case QGEMM_ERR_IO: return "QGEMM_ERR_IO";
        default: return "QGEMM_ERR_UNKNOWN";
    }
}

const char* qgemm_last_error(void) { return g_last_error; }

}  // extern "C"
