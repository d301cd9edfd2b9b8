/*
 * qgemm: weight-quantized linear layer C[M,N] = A[M,K] x dequant(B[K,N]) on NVIDIA GB300
 * (sm_103a), behind a plain C ABI.
 *
 * The operation and its formats follow the benchmark page "MNN GemmSpeed 基准测试实战：多后端
 * LLM GEMM 吞吐评估与 GPU 时间戳剖析":
 *   - «为什么用 Conv1x1 来测 GEMM»: the LLM linear layer is C = A[M,K] x B[K,N] with the
 *     weight given as {ic, oc} = {K, N}; quantized weights are asymmetric with one
 *     [offset, scale] pair per (output channel, K-block), stored as oc x blockNum pairs;
 *     Int8-Block0 is 8-bit with one block over all of K, Int4-Block64 is 4-bit with blocks
 *     of 64 along K (K % 64 == 0 is required).
 *   - «测试用例与注册机制»: mode numbers 0 float, 1 Int4-Block64, 2 Int8-Block0, 3 W4A8
 *     (per-channel INT4 weights unpacked to INT8, activations dynamically quantized to
 *     INT8, S8 x S8 -> S32 accumulation).
 *   - «测量流程»: throughput is counted as 2*M*K*N flops per call.
 *
 * Conventions for every function below:
 *   - All buffer pointers are DEVICE pointers owned by the caller (allocate them with any
 *     allocator; the library never allocates, frees or retains them). Each must be 16-byte
 *     aligned; 128-byte alignment is recommended.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Compute
 *     calls only enqueue work and return; results are ready once the stream is synchronized.
 *   - Return value: QGEMM_OK (0) or a negative QGEMM_ERR_* code. Every argument is checked
 *     before anything is launched; on an error nothing is enqueued and no buffer is written.
 *     qgemm_last_error() gives a one-line description of the last error on this thread.
 *   - Sizes are int; products of sizes are computed in 64 bits.
 *
 * Layouts (row-major unless stated):
 *   W   float32 [K][N]            the unquantized weight, {ic, oc} = {K, N}
 *   Bp  packed weight, output-channel-major with K contiguous:
 *         INT4 / W4A8  uint8 [N][K/2], byte j of a row = q[2j] | q[2j+1] << 4
 *         INT8         uint8 [N][K]
 *         FLOAT        [N][K] in the activation dtype (f16, bf16 or f32)
 *   T   float32 {offset, scale} per (channel n, block b), absent in FLOAT mode, stored in groups
 *       of 16 channels: [ceil(N/16)][K/block][16][2], i.e. the pair of (n, b) at pair index
 *       ((n / 16) * (K/block) + b) * 16 + n % 16; channels N .. ceil(N/16)*16 - 1 hold zeros.
 *       (The page keeps oc x blockNum pairs; the grouping lets one 16-channel unit's pairs for
 *       a K-range be one contiguous copy.)
 *   A   [M][K] in a_dtype;  C  [M][N] in c_dtype
 * Dequantization: w[k][n] = q[n][k] * scale[n][k/block] + offset[n][k/block], with unsigned
 * codes q in [0, 15] (4-bit) or [0, 255] (8-bit).
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* weight formats (same numbering as the benchmark page's mode column) */
#define QGEMM_MODE_FLOAT 0 /* unquantized 16/32-bit weight                       */
#define QGEMM_MODE_INT4 1  /* asymmetric 4-bit, block = 64 (any multiple of 64)  */
#define QGEMM_MODE_INT8 2  /* asymmetric 8-bit, block = K (Block0) or multiple of 64 */
#define QGEMM_MODE_W4A8 3  /* per-channel 4-bit weight x dynamic per-row 8-bit activation */

/* element types */
#define QGEMM_F32 0
#define QGEMM_F16 1
#define QGEMM_BF16 2

/* status codes */
#define QGEMM_OK 0
#define QGEMM_ERR_ARG (-1)         /* null pointer, negative size, unknown mode or dtype        */
#define QGEMM_ERR_UNSUPPORTED (-2) /* K % 64 != 0, K % block != 0, block not a multiple of 64,
                                      W4A8 with block != K, FLOAT weights of another dtype,
                                      a size beyond the launch limits                          */
#define QGEMM_ERR_ALIGN (-3)       /* a pointer is not 16-byte aligned                          */
#define QGEMM_ERR_WORKSPACE (-4)   /* workspace smaller than qgemm_workspace_bytes()            */
#define QGEMM_ERR_CUDA (-5)        /* a CUDA call or launch failed (detail in qgemm_last_error) */
#define QGEMM_ERR_TIMEOUT (-6)     /* a kernel gave up a bounded wait (reported by qgemm_status) */
#define QGEMM_ERR_IO (-7)          /* a weight file could not be read or written, or is corrupt  */

/* ---------------------------------------------------------------- sizes (host only, no GPU needed) */

/* Bytes of the packed weight Bp for a K x N layer. FLOAT mode stores w_dtype elements; the
 * quantized modes ignore w_dtype. Returns 0 for invalid arguments. */
size_t qgemm_packed_bytes(int K, int N, int mode, int w_dtype);

/* Bytes of the {offset, scale} table T, including the zero channels that complete the last
 * group of 16 (0 in FLOAT mode or for invalid arguments). block = 0 means one block over all
 * of K. */
size_t qgemm_table_bytes(int K, int N, int mode, int block);

/* Bytes of scratch device memory qgemm_run uses for this call (0 if none). The decode path
 * needs it when it splits K across thread blocks (small N); W4A8 needs it for the quantized
 * activations (2*M*K bytes of codes as 16-bit values, M scales and M row sums), and with
 * per-channel weights and K > 8808 also for int32 accumulators [M][N] (4*M*N bytes: the sums are
 * formed in K-chunks of at most 8192, each exact, and added in int32). The tensor-core
 * path (M above QGEMM_OPT_DECODE_MAX_M) needs 4*M bytes (256-byte aligned) for the row sums of A
 * in INT8 mode with block = K, bf16 activations and M >= 256 (the per-channel scale and offset are
 * then applied in its epilogue), and
 * uses the rest for float32 partial sums when it splits K
 * (mid-sized M, few 128-channel tiles): splits*M*N*4 bytes. That part is optional: qgemm_run
 * given less scratch splits K fewer times (down to none), which changes only the float32
 * summation order of the result. */
size_t qgemm_workspace_bytes(int M, int K, int N, int mode, int block, int a_dtype, int c_dtype);

/* ---------------------------------------------------------------- weight preparation */

/* Quantize and pack a float32 weight W [K][N] (benchmark page «为什么用 Conv1x1 来测 GEMM»).
 * For each channel n and block b (block elements along K), in float32 round-to-nearest:
 *   lo = min w, hi = max w, scale = (hi - lo) / qmax, offset = lo,
 *   q = clamp(rint((w - lo) / scale), 0, qmax) with ties to even; q = 0 if scale == 0.
 * qmax = 15 for INT4 and W4A8, 255 for INT8. W4A8 weights may be per channel (block = 0) or
 * per K-block like INT4.
 * FLOAT mode instead writes W transposed to [N][K], rounded to nearest-even in w_dtype,
 * and T may be NULL. W must be finite. Writes Bp (qgemm_packed_bytes) and T
 * (qgemm_table_bytes). */
int qgemm_pack(const float* W, int K, int N, int mode, int block, int w_dtype, void* Bp, float* T,
               void* stream);

/* ---------------------------------------------------------------- the layer */

/* C = A x dequant(Bp, T) for modes 0-3 (the operation of the benchmark page's four test
 * cases, «测试用例与注册机制»).
 *   a_dtype: f32, f16 or bf16. FLOAT mode expects Bp in the same dtype as A.
 *   c_dtype: f32, f16 or bf16 (results are accumulated in f32 and rounded once).
 *   W4A8: A is quantized per row (as = max|a| / 127, qa = clamp(rint(a / as), -127, 127)),
 *   acc = sum_k qa * q in int32, and C = as * (ws * acc + off * sum_k qa); with block-quantized
 *   weights C = as * sum_b (ws_b * acc_b + off_b * sum_{k in b} qa) over the K-blocks b (the
 *   weights are then dequantized per block to f16 for the tensor cores, so acc_b is not formed
 *   exactly; the result is within the float bar).
 * Kernel choice is by shape only: f32 activations use an exact CUDA-core kernel; M <= 16
 * uses the weight-streaming decode kernel; larger M uses the tensor-core (tcgen05) kernel.
 * workspace may be NULL when qgemm_workspace_bytes() returns 0. M == 0 or N == 0 is a valid
 * empty call that launches nothing. */
int qgemm_run(int M, int K, int N, int mode, int block, const void* A, int a_dtype, const void* Bp,
              const float* T, void* C, int c_dtype, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- fused epilogue */

/* Activations of qgemm_run_fused. */
#define QGEMM_ACT_NONE 0
#define QGEMM_ACT_RELU 1        /* max(x, 0) */
#define QGEMM_ACT_SILU 2        /* x / (1 + exp(-x)) */
#define QGEMM_ACT_GELU_TANH 3   /* 0.5 x (1 + tanh(sqrt(2 / pi) (x + 0.044715 x^3))) */

/* qgemm_run with the layer's neighbours fused into its output store. The pull request
 * "vulkan: 在骁龙 8 Gen 3（Adreno 750，安卓）上跑通并调优无协作矩阵档" keeps the float32 accumulators
 * until bias, residual and activation are applied (note on the DIRECT build); here
 *   C[m][n] = act(acc[m][n] + bias[n]) + residual[m][n]
 * in float32, rounded once to c_dtype, where acc is what qgemm_run would round (for W4A8 the
 * rescaled result).
 *   bias: float32 [N], 16-byte aligned, or NULL for none.
 *   act: QGEMM_ACT_*.
 *   residual: [M][N] in c_dtype, 16-byte aligned, or NULL for none. It may be C itself (an
 *   in-place residual add: every element is read before it is written, by the same thread),
 *   but must not overlap C in any other way.
 * Kernels, workspace and errors as qgemm_run; an unknown act gives QGEMM_ERR_ARG. */
int qgemm_run_fused(int M, int K, int N, int mode, int block, const void* A, int a_dtype, const void* Bp,
                    const float* T, const float* bias, int act, const void* residual, void* C, int c_dtype,
                    void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- activation step fused into the producer */

/* A layer (as qgemm_run_fused) that also produces the next W4A8 layer's activation codes from its
 * own output, so that a W4A8 layer fed by it skips its activation pass (the step on either side
 * of the path: the W4A8 activation quantization of «测试用例与注册机制», applied where the previous
 * layer's accumulators are still in float32, the Vulkan pull request's note on the DIRECT build).
 * After C is written exactly as qgemm_run_fused writes it, the activation step of qgemm_act_quant
 * is applied to C's stored values (rows of N elements):
 *   as_next[m] = max_n |C[m][n]| / 127, qa_next[m][n] = clamp(rint(C[m][n] / as_next[m]), -127, 127),
 *   rowsum_next[m] = sum_n qa_next[m][n]
 * bit for bit what qgemm_act_quant gives for C. The codes are written as exact f16 integers
 * [M][N] (the form qgemm_run_w4a8_codes reads), as_next float32 [M], rowsum_next int32 [M].
 * Where the layer runs on the tensor-core kernel in one launch (M above QGEMM_OPT_DECODE_MAX_M
 * with 16-bit activations, and W4A8 with K <= 8808), its epilogue records each 128-channel tile's
 * row maxima of |C| in the workspace and one pass reads C once to write the codes; on the other
 * paths the activation pass runs on C after the layer. N must be a multiple of 64 (it is the next
 * layer's K). Workspace: qgemm_fused_quant_workspace_bytes (the tensor-core path does not split K
 * in this call). Errors as qgemm_run_fused; QGEMM_ERR_UNSUPPORTED for N % 64 != 0. */
int qgemm_run_fused_quant(int M, int K, int N, int mode, int block, const void* A, int a_dtype, const void* Bp,
                          const float* T, const float* bias, int act, const void* residual, void* C, int c_dtype,
                          void* qa_next, float* as_next, int32_t* rowsum_next, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Workspace bytes of qgemm_run_fused_quant (0 for invalid arguments or when none is needed). */
size_t qgemm_fused_quant_workspace_bytes(int M, int K, int N, int mode, int block, int a_dtype, int c_dtype);

/* A W4A8 layer from activation codes already computed (by qgemm_run_fused_quant): qa exact f16
 * integers [M][K] in [-127, 127], a_scale float32 [M], rowsum int32 [M] (their sum per row).
 * Computes what qgemm_run_fused computes in W4A8 mode after its activation pass:
 * C = act(a_scale * (ws * acc + off * rowsum) + bias) + residual with acc = sum_k qa * q (per-channel
 * weights, block = 0 or K; exact), or the per-block form for block-quantized weights. The workspace
 * (qgemm_w4a8_codes_workspace_bytes) holds int32 accumulators [M][N] when the weights are per channel
 * and K > 8808, and is otherwise not needed. */
int qgemm_run_w4a8_codes(int M, int K, int N, int block, const void* qa, const float* a_scale, const int32_t* rowsum,
                         const void* Bp, const float* T, const float* bias, int act, const void* residual, void* C,
                         int c_dtype, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of qgemm_run_w4a8_codes (0 if none). */
size_t qgemm_w4a8_codes_workspace_bytes(int M, int K, int N, int block);

/* The W4A8 activation step alone (same page and section: "激活动态量化为 INT8"): per row of
 * A [M][K], as[m] = max|a| / 127 (float32), qa = clamp(rint(a / as), -127, 127) with ties
 * to even (all 0 when as == 0), rowsum[m] = sum_k qa. Outputs qa int8 [M][K], as float32 [M],
 * rowsum int32 [M]. */
int qgemm_act_quant(int M, int K, const void* A, int a_dtype, int8_t* qa, float* a_scale, int32_t* rowsum,
                    void* stream);

/* The W4A8 integer GEMM alone ("S8×S8→S32"): acc[m][n] = sum_k qa[m][k] * q[n][k] with q the
 * 4-bit codes of Bp [N][K/2] read as int8 values 0..15. Writes acc int32 [M][N]. The sums are
 * exact for every accepted K: the tensor cores accumulate in float32, which is exact while every
 * partial sum is an integer below 2^24 (K <= 8808); longer K runs as K-chunks of at most 8192
 * whose sums are added into acc in int32 (acc is cleared first). K above 1127384, where
 * 127 * 15 * K could overflow int32, gives QGEMM_ERR_UNSUPPORTED (also for qgemm_run in W4A8
 * mode). Needs a workspace of qgemm_w4a8_acc_workspace_bytes(M, K) bytes (the codes as 16-bit
 * operands). */
int qgemm_w4a8_acc(int M, int K, int N, const int8_t* qa, const void* Bp, int32_t* acc, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Workspace bytes qgemm_w4a8_acc needs (0 for invalid sizes). */
size_t qgemm_w4a8_acc_workspace_bytes(int M, int K);

/* ---------------------------------------------------------------- no-allocation variant */

/* Size of the library's own scratch buffer used by qgemm_run_noalloc (4 MiB). */
#define QGEMM_NOALLOC_SCRATCH_BYTES (4u << 20)

/* qgemm_run without a caller workspace, for callers that cannot hand the library device memory
 * of their own: code whose execution path must not allocate (a plugin inside an inference
 * engine that owns all device memory, a real-time loop that cannot pay for an allocator call,
 * a C host with no device allocator at hand). The pages have no counterpart to this call; it is
 * a convenience of this library.
 * It computes exactly what qgemm_run computes, with the same kernels, but its scratch memory is
 * a fixed array inside the library (QGEMM_NOALLOC_SCRATCH_BYTES, 256-byte aligned) that every
 * GPU which loads the library keeps until the process exits. No call allocates or frees device
 * memory.
 *   - A call whose required scratch exceeds the array is rejected with QGEMM_ERR_WORKSPACE
 *     before anything is enqueued; calls that need no scratch always fit. The required part is
 *     qgemm_workspace_bytes less the tensor-core path's optional split-K partial sums, which
 *     are cut to what the array holds.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before capturing a stream into a graph.
 *   - All calls share the one array and leave their data in it. Every byte a call reads from it
 *     is written earlier by the same call, so nothing needs clearing; but two calls whose work
 *     overlaps on the GPU (different streams, or different host threads, without ordering)
 *     race on it and may produce wrong results. Order them on one stream. */
int qgemm_run_noalloc(int M, int K, int N, int mode, int block, const void* A, int a_dtype, const void* Bp,
                      const float* T, void* C, int c_dtype, void* stream);
/* (The array's device address is looked up once per device and kept for the life of the
 * process. A device reset or a torn-down and recreated primary context invalidates it: reload
 * the library, or do not call qgemm_run_noalloc again, after cudaDeviceReset.) */

/* ---------------------------------------------------------------- packed-weight files */

/* One packed layer per file, so that weights are quantized once (qgemm_pack) and later loaded
 * ready to run: a 64-byte little-endian header {magic "QGEMMW\0\1", version 1, header size 64,
 * K, N, mode, block, w_dtype, CRC-32 of the payload, Bp bytes, T bytes}, then Bp, then T (none
 * in FLOAT mode), byte for byte as qgemm_pack wrote them. The pages have no counterpart; this
 * is a convenience of this library.
 * on_device: 1 if Bp / T are device pointers (copied through a host staging buffer on `stream`,
 * synchronously), 0 if they are host pointers (no CUDA call is made). */

/* Writes Bp (qgemm_packed_bytes) and T (qgemm_table_bytes; NULL in FLOAT mode) of the shape to
 * `path`, replacing the file. QGEMM_ERR_ARG for an invalid shape or null buffer, QGEMM_ERR_IO if
 * the file cannot be written. */
int qgemm_save(const char* path, int K, int N, int mode, int block, int w_dtype, const void* Bp, const float* T,
               int on_device, void* stream);

/* Reads a file's header: the shape and format to pass to qgemm_packed_bytes / qgemm_table_bytes
 * and qgemm_run. QGEMM_ERR_IO for a missing, foreign or inconsistent file. */
int qgemm_load_info(const char* path, int* K, int* N, int* mode, int* block, int* w_dtype);

/* Reads a file's Bp and T into buffers of at least the file's sizes (QGEMM_ERR_ARG if smaller).
 * The whole payload is read and its CRC-32 checked before anything is written to Bp or T:
 * a truncated, extended or corrupt file gives QGEMM_ERR_IO and leaves them untouched. */
int qgemm_load(const char* path, void* Bp, size_t Bp_bytes, float* T, size_t T_bytes, int on_device, void* stream);

/* ---------------------------------------------------------------- options */

/* QGEMM_OPT_LAUNCH_OVERLAP (default 0). When 1, the decode kernel (M <= 16) is launched with a
 * programmatic dependency on the previous kernel in the stream: it may start while that
 * kernel is finishing, begins streaming Bp and T at once, and waits for the previous kernel
 * to complete before it reads A or writes C or the workspace. This hides the launch and
 * weight-fetch latency of back-to-back layer calls. CONTRACT while enabled: the kernel
 * launched immediately before qgemm_run on the same stream must not write Bp or T.
 * The setting is process-wide. */
#define QGEMM_OPT_LAUNCH_OVERLAP 1

/* QGEMM_OPT_DECODE_MAX_M (default 16, range 16..1024). Layers with M up to this value (and
 * 16-bit activations) run on the weight-streaming decode kernels, in launches of 16 rows of A;
 * larger M on the tensor-core kernel. A larger value trades extra weight reads (one per 16 rows)
 * for using every SM when N offers few 128-channel tiles. The setting is process-wide; it
 * changes qgemm_workspace_bytes for the shapes it moves. */
#define QGEMM_OPT_DECODE_MAX_M 2

/* QGEMM_OPT_SPLIT_K (default 1). When 1, the tensor-core kernel splits K across thread blocks
 * for shapes whose output tiles (128 channels x up to 256 rows) fill less than one wave of the
 * GPU's SMs; each split writes float32 partial sums to the workspace and a second kernel adds
 * them in a fixed order and rounds once. When 0, it never splits (no workspace needed). The
 * setting is process-wide; it changes qgemm_workspace_bytes for the shapes it affects. */
#define QGEMM_OPT_SPLIT_K 3

/* QGEMM_OPT_WAIT_LIMIT_US (default 1000000, range 1..1000000). The TMA-fed kernels (the decode
 * kernel for M <= 16 and the tensor-core kernel) bound every wait of their pipelines by this many
 * microseconds of the GPU's global timer: a wait that runs out sets the status word that
 * qgemm_status reports as QGEMM_ERR_TIMEOUT, every role of the thread block leaves its loop, the
 * copies and MMAs already issued are waited for (always with the full one-second bound) and the
 * tensor memory is released before the block exits; that call's outputs are then undefined. A
 * bound shorter than a normal wait makes healthy calls time out: the option exists to exercise
 * that recovery path, and production code keeps the default. Process-wide. */
#define QGEMM_OPT_WAIT_LIMIT_US 4

/* QGEMM_OPT_DEBUG_STALL (default 0). Diagnostic: when 1, every following launch of the TMA-fed
 * kernels has one role (the MMA issuer of the tensor-core kernel, the first consumer warp of the
 * decode kernel) wait first on a barrier that nothing arrives at, so that the wait runs out after
 * QGEMM_OPT_WAIT_LIMIT_US and the call ends with QGEMM_ERR_TIMEOUT as described above. It makes
 * the timeout path testable without a hang; production code keeps 0. Process-wide. */
#define QGEMM_OPT_DEBUG_STALL 5

/* QGEMM_OPT_FAULT_INJECT (default 0, or the value of the environment variable QGEMM_FAULT_INJECT
 * when the library loads). Host-side fault injection: when n > 0, the n-th compute call from now
 * (qgemm_pack, qgemm_run, qgemm_run_fused, qgemm_run_noalloc, qgemm_act_quant, qgemm_w4a8_acc)
 * passes its argument checks and then returns QGEMM_ERR_CUDA with the detail "simulated launch
 * failure" instead of launching, as a failed launch would; the count then stays 0. No GPU fault is
 * involved. For testing callers' error handling. Process-wide. */
#define QGEMM_OPT_FAULT_INJECT 6

/* Set an option; returns its previous value, or QGEMM_ERR_ARG for an unknown option or value. */
int qgemm_set_option(int option, int value);

/* Current value of an option, or QGEMM_ERR_ARG for an unknown option. */
int qgemm_get_option(int option);

/* ---------------------------------------------------------------- status */

/* Synchronize `stream`, then report (and clear) the library's device status word: QGEMM_OK,
 * QGEMM_ERR_TIMEOUT if a kernel gave up a bounded wait, or QGEMM_ERR_CUDA on a CUDA error or if
 * a kernel found its shared memory misaligned for its TMA copies (it then skipped its work). */
int qgemm_status(void* stream);

/* Static name of a status code. */
const char* qgemm_error_string(int code);

/* Description of the last error returned on the calling thread ("" if none). */
const char* qgemm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H */
