// Tensor-core path for the raw-code forms: W4A8 (4-bit weight codes x 8-bit activation codes,
// exact) and Int8-Block0 with bf16 activations (8-bit codes, per-channel scale and offset in the
// epilogue). The kernel template is in prefill_kernel.cuh.
#include "prefill_kernel.cuh"

namespace qg {
namespace pf {

// ---------------------------------------------------------------- W4A8 activation codes as f16
__global__ void codes_to_f16_kernel(const int8_t* __restrict__ qa, __half* __restrict__ out, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        out[i] = __int2half_rn(qa[i]);
}

}  // namespace pf

cudaError_t launch_prefill_codes8(const pf::Maps& maps, const pf::Params& p, int kdt, cudaStream_t s) {
    return pf::launch_wf<pf::WF_CODES8, true, pf::EPI_W4A8>(maps, p, kdt, s);
}

cudaError_t launch_w4a8_gemm(const W4A8Args& a, cudaStream_t s) {
    pf::Params p{};
    const int block = a.block > 0 ? a.block : a.K;
    p.M = a.M; p.K = a.K; p.N = a.N; p.block = block; p.nb = a.K / block;
    p.BN = pf::pick_bn(a.M);
    p.Bp = static_cast<const uint8_t*>(a.Bp); p.T = a.T; p.C = a.C;
    p.a_scale = a.as; p.rowsum = a.rowsum; p.acc = a.acc; p.splits = 1;
    p.status = status_word_address();
    if (!p.status) return cudaErrorInvalidValue;
    p.ep = a.acc ? Epilogue{} : a.ep;
    pf::Maps maps;
    cudaError_t e = pf::make_tmap(&maps.a, a.qa16, false, a.M, a.K, p.BN);
    if (e != cudaSuccess) return e;
    p.c_tma = a.acc ? (pf::make_out_map(&maps.c, a.acc, -1, a.M, a.N, p.BN, 1) ? 1 : 0)
                    : (pf::make_out_map(&maps.c, a.C, a.c_dtype, a.M, a.N, p.BN, 1) ? 1 : 0);
    if (!p.c_tma) maps.c = maps.a;     // unused
    p.r_tma = p.ep.residual && pf::make_out_map(&maps.r, const_cast<void*>(p.ep.residual), a.c_dtype, a.M, a.N, p.BN, 1)
                  ? 1 : 0;
    if (!p.r_tma) maps.r = maps.a;     // unused
    if (a.acc) return pf::launch_wf<pf::WF_CODES4, false, pf::EPI_ACC>(maps, p, DT_F32, s);
    if (block != a.K) {
        // weights quantized per K-block: the block {offset, scale} vary along K, so the weights are
        // dequantized per block into f16 (as on the Int4 path) and multiplied with the activation
        // codes (exact f16 integers); the epilogue applies the row scale as only:
        // as * sum_k qa (q s + o) = as * sum_b (s_b sum qa q + o_b sum qa)
        return pf::launch_wf<pf::WF_INT4, false, pf::EPI_W4A8>(maps, p, a.c_dtype, s);
    }
    return pf::launch_wf<pf::WF_CODES4, false, pf::EPI_W4A8>(maps, p, a.c_dtype, s);
}

cudaError_t launch_codes_to_f16(const int8_t* qa, void* out, size_t n, cudaStream_t s) {
    const int threads = 256;
    const size_t want = (n + threads - 1) / threads;
    pf::codes_to_f16_kernel<<<(int)(want < 8192 ? want : 8192), threads, 0, s>>>(qa, static_cast<__half*>(out), n);
    return cudaGetLastError();
}

}  // namespace qg
