// Tensor-core path, dequantizing forms (Int4 / Int8 per K-block, float mode) and the shared
// host logic: K-split choice, the library's device status word, the tensor-map encoder.
#include <mutex>

#include "prefill_kernel.cuh"

namespace qg {

// Set (bitwise OR) by a kernel that gave up a bounded wait; read and cleared by qgemm_status.
__device__ unsigned int g_status_word;

EncodeTiledFn tensor_map_encoder() {
    // looked up once (thread-safe one-time initialization); nullptr if the driver lacks it
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(f);
        return EncodeTiledFn(nullptr);
    }();
    return fn;
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
unsigned int* g_status_addr[kMaxDevices] = {};
}  // namespace

unsigned int* status_word_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_addr[dev] = static_cast<unsigned int*>(p);
    }
    return g_status_addr[dev];
}

cudaError_t read_and_clear_status(int* value, cudaStream_t s) {
    unsigned int h = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&h, g_status_word, sizeof(h), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *value = (int)h;
    if (h != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero));
    }
    return e;
}

int prefill_splits(int M, int K, int N, int fmt) {
    (void)fmt;
    // Mid-sized M leaves most SMs idle (one block per 128 channels x BN rows): split K across
    // up to one wave of blocks, each split keeping at least kMinStages stages of 64. The split
    // partial sums cost splits * M * N * 4 bytes of traffic: 256-row tiles that already fill a
    // third of a wave or more stay whole (two splits measured slower at 64 and 76 tiles), smaller
    // tiles split in two from half a wave down (measured faster at 76 tiles, M = 24..128).
    constexpr int kMinStages = 8;
    const int bn = pf::pick_bn(M);
    const long long tiles = (long long)((N + pf::kBM - 1) / pf::kBM) * ((M + bn - 1) / bn);
    long long splits = kTargetSms / tiles;
    if (splits < (bn >= 256 ? 3 : 2)) return 1;
    const int by_k = (K / pf::kBK) / kMinStages;
    if (splits > by_k) splits = by_k;
    return splits > 1 ? (int)splits : 1;
}

bool prefill_supported(int M, int K, int N, int fmt, int a_dtype) {
    (void)K;
    (void)N;
    (void)fmt;
    return M > 16 && (a_dtype == DT_F16 || a_dtype == DT_BF16);
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
    pf::Params p{};
    p.M = a.M; p.K = a.K; p.N = a.N; p.block = a.block; p.nb = a.K / a.block;
    p.BN = pf::pick_bn(a.M);
    p.Bp = static_cast<const uint8_t*>(a.Bp); p.T = a.T; p.C = a.C;
    p.splits = a.splits > 1 ? a.splits : 1;
    p.status = status_word_address();
    if (!p.status) return cudaErrorInvalidValue;
    p.wait_ns = option_wait_ns();
    p.stall = option_stall();
    p.ep = p.splits > 1 ? Epilogue{} : a.ep;   // split partials: the reduction applies it
    p.rowmax = p.splits > 1 ? nullptr : a.rowmax;
    // with K-splits the kernel writes float32 partial sums [splits][M][N], reduced in fixed order
    const int kdt = p.splits > 1 ? DT_F32 : a.c_dtype;
    if (p.splits > 1) p.C = a.partial;
    const bool bf = a.a_dtype == DT_BF16;
    pf::Maps maps;
    cudaError_t e = pf::make_tmap(&maps.a, a.A, bf, a.M, a.K, p.BN);
    if (e != cudaSuccess) return e;
    p.c_tma = pf::make_out_map(&maps.c, p.C, kdt, a.M, a.N, pf::kSlabRows, p.splits) ? 1 : 0;
    if (!p.c_tma) maps.c = maps.a;             // unused
    p.r_tma = p.ep.residual && pf::make_out_map(&maps.r, const_cast<void*>(p.ep.residual), kdt, a.M, a.N, p.BN, 1) ? 1 : 0;
    if (!p.r_tma) maps.r = maps.a;             // unused
    if (prefill_codes_path(a.fmt, a.K, a.block, a.M, a.a_dtype)) {
        // Int8-Block0: raw codes on the tensor cores, s * acc + o * sum_k a in the epilogue
        e = launch_row_sums(a.M, a.K, a.A, a.a_dtype, a.rowsum, s);
        if (e != cudaSuccess) return e;
        p.rowsum_f = a.rowsum;
        e = launch_prefill_codes8(maps, p, kdt, s);   // bf16 only
    } else if (a.fmt == FMT_INT4)
        e = bf ? pf::launch_wf<pf::WF_INT4, true, pf::EPI_STORE>(maps, p, kdt, s)
               : pf::launch_wf<pf::WF_INT4, false, pf::EPI_STORE>(maps, p, kdt, s);
    else if (a.fmt == FMT_INT8)
        e = bf ? pf::launch_wf<pf::WF_INT8, true, pf::EPI_STORE>(maps, p, kdt, s)
               : pf::launch_wf<pf::WF_INT8, false, pf::EPI_STORE>(maps, p, kdt, s);
    else
        e = bf ? pf::launch_wf<pf::WF_FLOAT, true, pf::EPI_STORE>(maps, p, kdt, s)
               : pf::launch_wf<pf::WF_FLOAT, false, pf::EPI_STORE>(maps, p, kdt, s);
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_splitk_reduce(a.partial, p.splits, (size_t)a.M * a.N, a.N, a.ep, a.C, a.c_dtype, s);
}

}  // namespace qg
