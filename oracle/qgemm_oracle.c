/*
 * CPU oracle for the weight-quantized linear layer C[M,N] = A[M,K] x dequant(B[K,N]).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's GPU path calls, links or includes this
 * file; only the test suite, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header or constant with the CUDA sources.
 *
 * Plain loops, written to be checked by eye against the pages:
 *   - "MNN GemmSpeed 基准测试实战" (the benchmark page), section «为什么用 Conv1x1 来测 GEMM»:
 *     the layer is C = A[M,K] x B[K,N] with weight shape {ic, oc} = {K, N}; the quantized
 *     modes are asymmetric, with an [offset, scale] pair per (output channel, K-block),
 *     laid out as oc x blockNum pairs; Int4-Block64 uses blocks of 64 along K, Int8-Block0
 *     one block covering all of K.
 *   - same page, section «测试用例与注册机制»: W4A8 unpacks per-channel INT4 weights to INT8,
 *     quantizes activations dynamically to INT8 and accumulates S8 x S8 -> S32.
 * Where the page is silent the plainest reading is taken (min/max asymmetric scheme,
 * unsigned codes, round half to even, f32 decisions, f64 accumulation); each reading is
 * stated at the function that uses it.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off (no fast-math), so every float expression below
 * is evaluated as written in IEEE single or double precision.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_OVERFLOW (-2)

int orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/*
 * Asymmetric block quantization (benchmark page, «为什么用 Conv1x1 来测 GEMM»: "非对称量化",
 * "[offset, scale] 交替对", oc x blockNum groups).
 * W is the row-major [K][N] float32 weight. For each output channel n and each block b of
 * `block` consecutive k, all in float32 round-to-nearest:
 *     lo = min w, hi = max w, scale = (hi - lo) / qmax, offset = lo,
 *     q  = clamp(rint((w - lo) / scale), 0, qmax), rint = round half to even,
 * and q = 0 for the whole block when scale == 0 (a constant block dequantizes to offset).
 * Outputs: q [N][K] one unsigned code per byte; T [N][K/block][2] = {offset, scale}.
 */
int orc_quantize(const float* W, int64_t K, int64_t N, int64_t block, int qmax, uint8_t* q, float* T) {
    if (!W || !q || !T || K <= 0 || N <= 0 || block <= 0 || K % block != 0 || qmax <= 0 || qmax > 255)
        return ORC_ERR_ARG;
    const int64_t nb = K / block;
    const float fq = (float)qmax;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const int64_t k0 = b * block;
            float lo = W[k0 * N + n], hi = lo;
            for (int64_t k = k0; k < k0 + block; ++k) {
                const float w = W[k * N + n];
                if (w < lo) lo = w;
                if (w > hi) hi = w;
            }
            const float d = hi - lo;
            const float scale = d / fq;
            T[(n * nb + b) * 2 + 0] = lo;
            T[(n * nb + b) * 2 + 1] = scale;
            for (int64_t k = k0; k < k0 + block; ++k) {
                int code = 0;
                if (scale != 0.0f) {
                    const float t = W[k * N + n] - lo;
                    const float u = t / scale;
                    const float r = nearbyintf(u); /* default rounding mode: ties to even */
                    code = (int)r;
                    if (code < 0) code = 0;
                    if (code > qmax) code = qmax;
                }
                q[n * K + k] = (uint8_t)code;
            }
        }
    }
    return ORC_OK;
}

/*
 * Packing of the codes (the page fixes only "nbit 4" / "nbit 8"; the layout is the stated
 * reading): Bp is [N][K*nbits/8], output-channel-major with K contiguous. For 4 bits,
 * byte j of a row holds q[2j] in its low nibble and q[2j+1] in its high nibble.
 */
int orc_pack(const uint8_t* q, int64_t K, int64_t N, int nbits, uint8_t* Bp) {
    if (!q || !Bp || K <= 0 || N <= 0) return ORC_ERR_ARG;
    if (nbits == 8) {
        memcpy(Bp, q, (size_t)(K * N));
        return ORC_OK;
    }
    if (nbits != 4 || K % 2 != 0) return ORC_ERR_ARG;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / 2; ++j) {
            const uint8_t lo = q[n * K + 2 * j], hi = q[n * K + 2 * j + 1];
            if (lo > 15 || hi > 15) return ORC_ERR_ARG;
            Bp[n * (K / 2) + j] = (uint8_t)(lo | (hi << 4));
        }
    return ORC_OK;
}

/* Inverse of orc_pack (used to read codes back out of a packed buffer). */
int orc_unpack(const uint8_t* Bp, int64_t K, int64_t N, int nbits, uint8_t* q) {
    if (!q || !Bp || K <= 0 || N <= 0) return ORC_ERR_ARG;
    if (nbits == 8) {
        memcpy(q, Bp, (size_t)(K * N));
        return ORC_OK;
    }
    if (nbits != 4 || K % 2 != 0) return ORC_ERR_ARG;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / 2; ++j) {
            const uint8_t byte = Bp[n * (K / 2) + j];
            q[n * K + 2 * j] = (uint8_t)(byte & 15);
            q[n * K + 2 * j + 1] = (uint8_t)(byte >> 4);
        }
    return ORC_OK;
}

/*
 * Dequantization w = q * scale + offset, evaluated in double: q * scale is exact in double
 * (a <= 8-bit integer times a 24-bit significand), so the only rounding is the final add.
 * Output Bt [N][K] float64, i.e. the transpose of the weight B[K][N].
 */
int orc_dequant(const uint8_t* q, const float* T, int64_t K, int64_t N, int64_t block, double* Bt) {
    if (!q || !T || !Bt || K <= 0 || N <= 0 || block <= 0 || K % block != 0) return ORC_ERR_ARG;
    const int64_t nb = K / block;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            const int64_t b = k / block;
            const double offset = (double)T[(n * nb + b) * 2 + 0];
            const double scale = (double)T[(n * nb + b) * 2 + 1];
            Bt[n * K + k] = (double)q[n * K + k] * scale + offset;
        }
    return ORC_OK;
}

/*
 * The GEMM of the linear layer (benchmark page, «为什么用 Conv1x1 来测 GEMM»: C = A[M,K] x B[K,N]):
 * R[m][n] = sum_k A[m][k] * B[k][n], summed in double with k increasing.
 * A is [M][K] float64 (exact copies of the stored activations), Bt is [N][K] float64.
 */
int orc_gemm(int64_t M, int64_t K, int64_t N, const double* A, const double* Bt, double* R) {
    if (!A || !Bt || !R || M <= 0 || K <= 0 || N <= 0) return ORC_ERR_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += A[m * K + k] * Bt[n * K + k];
            R[m * N + n] = acc;
        }
    return ORC_OK;
}

/*
 * The same dot products as orc_dequant + orc_gemm, for a list of (m, n) points only, with
 * the dequantization done on the fly (for full-size layers where the whole product is too
 * slow on a CPU). out[i] = sum_k A[m_i][k] * (q[n_i][k] * scale + offset).
 */
int orc_gemm_points(int64_t K, int64_t N, int64_t block, const double* A, const uint8_t* q, const float* T,
                    int64_t npts, const int64_t* m_idx, const int64_t* n_idx, double* out) {
    if (!A || !q || !T || !m_idx || !n_idx || !out || K <= 0 || N <= 0 || block <= 0 || K % block != 0)
        return ORC_ERR_ARG;
    const int64_t nb = K / block;
    for (int64_t i = 0; i < npts; ++i)
        if (n_idx[i] < 0 || n_idx[i] >= N || m_idx[i] < 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t m = m_idx[i], n = n_idx[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const int64_t b = k / block;
            const double w = (double)q[n * K + k] * (double)T[(n * nb + b) * 2 + 1] + (double)T[(n * nb + b) * 2 + 0];
            acc += A[m * K + k] * w;
        }
        out[i] = acc;
    }
    return ORC_OK;
}

/* Float-mode points: out[i] = sum_k A[m_i][k] * Bt[n_i][k] with Bt the [N][K] float64 weight. */
int orc_dense_points(int64_t K, const double* A, const double* Bt, int64_t npts, const int64_t* m_idx,
                     const int64_t* n_idx, double* out) {
    if (!A || !Bt || !m_idx || !n_idx || !out || K <= 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < npts; ++i) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += A[m_idx[i] * K + k] * Bt[n_idx[i] * K + k];
        out[i] = acc;
    }
    return ORC_OK;
}

/*
 * Float mode keeps the weight as a 16-bit copy, transposed to [N][K]. bfloat16 is the top
 * half of a float32, rounded to nearest with ties to even (the IEEE default), written out
 * here on the bit pattern. NaN is not handled (weights are finite).
 */
int orc_to_bf16_t(const float* W, int64_t K, int64_t N, uint16_t* out) {
    if (!W || !out || K <= 0 || N <= 0) return ORC_ERR_ARG;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            uint32_t u;
            memcpy(&u, &W[k * N + n], 4);
            const uint32_t lsb = (u >> 16) & 1u;
            out[n * K + k] = (uint16_t)((u + 0x7FFFu + lsb) >> 16);
        }
    return ORC_OK;
}

/*
 * Dynamic per-row activation quantization for W4A8 (benchmark page, «测试用例与注册机制»:
 * "激活动态量化为 INT8"; the page gives no formula, so the plainest symmetric reading is
 * used): per row, in float32, amax = max |a|, as = amax / 127, qa = clamp(rint(a / as),
 * -127, 127) with ties to even, all qa = 0 when as == 0, and rowsum = sum qa (integer).
 * A is [M][K] float32 holding the exact values of the stored activations.
 */
int orc_act_quant(int64_t M, int64_t K, const float* A, int8_t* qa, float* as, int32_t* rowsum) {
    if (!A || !qa || !as || !rowsum || M <= 0 || K <= 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            const float v = fabsf(A[m * K + k]);
            if (v > amax) amax = v;
        }
        const float s = amax / 127.0f;
        int64_t sum = 0;
        for (int64_t k = 0; k < K; ++k) {
            int code = 0;
            if (s != 0.0f) {
                const float u = A[m * K + k] / s;
                code = (int)nearbyintf(u);
                if (code < -127) code = -127;
                if (code > 127) code = 127;
            }
            qa[m * K + k] = (int8_t)code;
            sum += code;
        }
        as[m] = s;
        rowsum[m] = (int32_t)sum;
    }
    return ORC_OK;
}

/*
 * W4A8 integer accumulators ("S8xS8→S32", «测试用例与注册机制»): acc[m][n] = sum_k qa[m][k] * q[n][k]
 * where q in [0, 15] is the unpacked INT4 code used as a signed 8-bit value. Summed in int64;
 * returns ORC_ERR_OVERFLOW if a result does not fit int32.
 */
int orc_w4a8_acc(int64_t M, int64_t K, int64_t N, const int8_t* qa, const uint8_t* q, int32_t* acc) {
    if (!qa || !q || !acc || M <= 0 || K <= 0 || N <= 0) return ORC_ERR_ARG;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(static) reduction(| : bad)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)qa[m * K + k] * (int64_t)q[n * K + k];
            if (s > INT32_MAX || s < INT32_MIN) bad = 1;
            acc[m * N + n] = (int32_t)s;
        }
    return bad ? ORC_ERR_OVERFLOW : ORC_OK;
}

/* Point version of orc_w4a8_acc. */
int orc_w4a8_acc_points(int64_t K, const int8_t* qa, const uint8_t* q, int64_t npts, const int64_t* m_idx,
                        const int64_t* n_idx, int32_t* out) {
    if (!qa || !q || !m_idx || !n_idx || !out || K <= 0) return ORC_ERR_ARG;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t i = 0; i < npts; ++i) {
        int64_t s = 0;
        for (int64_t k = 0; k < K; ++k) s += (int64_t)qa[m_idx[i] * K + k] * (int64_t)q[n_idx[i] * K + k];
        if (s > INT32_MAX || s < INT32_MIN) bad = 1;
        out[i] = (int32_t)s;
    }
    return bad ? ORC_ERR_OVERFLOW : ORC_OK;
}

/*
 * W4A8 rescale. The integer GEMM sees a_q = qa * as and w = q * ws + off (per channel), so
 *   sum_k a_q w = as * (ws * sum_k qa q + off * sum_k qa) = as * (ws * acc + off * rowsum),
 * evaluated in double. T is [N][1][2] = {off, ws}.
 */
int orc_w4a8_out(int64_t M, int64_t N, const int32_t* acc, const float* as, const int32_t* rowsum,
                 const float* T, double* R) {
    if (!acc || !as || !rowsum || !T || !R || M <= 0 || N <= 0) return ORC_ERR_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            const double off = (double)T[n * 2 + 0], ws = (double)T[n * 2 + 1];
            R[m * N + n] = (double)as[m] * (ws * (double)acc[m * N + n] + off * (double)rowsum[m]);
        }
    return ORC_OK;
}

/*
 * Output epilogue (the pull request "vulkan: 在骁龙 8 Gen 3（Adreno 750，安卓）上跑通并调优无协作矩阵档"
 * keeps accumulators unrounded until bias, residual and activation are applied; the order
 * and the activations are this library's reading): in double, for every output,
 *   R[m][n] = act(R[m][n] + bias[n]) + residual[m][n]
 * with act 0 = identity, 1 = max(x, 0), 2 = x * sigmoid(x), 3 = the tanh form of GELU,
 * 0.5 x (1 + tanh(sqrt(2 / pi) (x + 0.044715 x^3))). bias and residual may be NULL.
 */
static double orc_act(int act, double x) {
    switch (act) {
        case 1: return x > 0.0 ? x : 0.0;
        case 2: return x / (1.0 + exp(-x));
        case 3: {
            const double c = sqrt(2.0 / 3.14159265358979323846);
            return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
        }
        default: return x;
    }
}

int orc_epilogue(int64_t M, int64_t N, double* R, const float* bias, int act, const double* residual) {
    if (!R || M <= 0 || N <= 0 || act < 0 || act > 3) return ORC_ERR_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double v = R[m * N + n];
            if (bias) v += (double)bias[n];
            v = orc_act(act, v);
            if (residual) v += residual[m * N + n];
            R[m * N + n] = v;
        }
    return ORC_OK;
}

/*
 * W4A8 with weights quantized per K-block (the page's block sizes, «为什么用 Conv1x1 来测 GEMM»,
 * applied to the W4A8 weights): each block b of K has its own {off_b, ws_b}, so the integer
 * GEMM runs per block and the rescale sums the blocks:
 *   R[m][n] = as[m] * sum_b (ws_b * sum_{k in b} qa q + off_b * sum_{k in b} qa)
 * with the block sums in int64 and the rescale in double. q is [N][K], T is [N][K/block][2].
 */
int orc_w4a8_block_out(int64_t M, int64_t K, int64_t N, int64_t block, const int8_t* qa, const float* as,
                       const uint8_t* q, const float* T, double* R) {
    if (!qa || !as || !q || !T || !R || M <= 0 || K <= 0 || N <= 0 || block <= 0 || K % block) return ORC_ERR_ARG;
    const int64_t nb = K / block;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double r = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                int64_t acc = 0, rs = 0;
                for (int64_t k = b * block; k < (b + 1) * block; ++k) {
                    acc += (int64_t)qa[m * K + k] * (int64_t)q[n * K + k];
                    rs += qa[m * K + k];
                }
                const double off = (double)T[(n * nb + b) * 2 + 0], ws = (double)T[(n * nb + b) * 2 + 1];
                r += ws * (double)acc + off * (double)rs;
            }
            R[m * N + n] = (double)as[m] * r;
        }
    return ORC_OK;
}
