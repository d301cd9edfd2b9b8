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

// C = epilogue(as * (ws * acc + off * rowsum)) with the same float32 steps as the tensor-core
// kernel's W4A8 epilogue: fma(ws, as * acc, off * (as * rowsum)).
template <int CDT>
__global__ void w4a8_rescale_kernel(int M, int N, const int32_t* __restrict__ acc, const float* __restrict__ as,
                                    const int32_t* __restrict__ rowsum, const float* __restrict__ T, Epilogue ep,
                                    void* C) {
    const size_t count = (size_t)M * N;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count; i += (size_t)gridDim.x * blockDim.x) {
        const int m = (int)(i / (size_t)N), n = (int)(i - (size_t)m * N);
        const float a = __ldg(as + m);
        const float2 t = __ldg(reinterpret_cast<const float2*>(T + tab_index(n, 1, 0) * 2));   // {off, ws}
        const float y = fmaf(t.y, a * (float)__ldg(acc + i), t.x * (a * (float)__ldg(rowsum + m)));
        store_c<CDT>(C, i, epilogue_apply<CDT>(ep, y, i, n));
    }
}

}  // namespace pf

cudaError_t launch_w4a8_rescale(int M, int N, const int32_t* acc, const float* as, const int32_t* rowsum,
                                const float* T, const Epilogue& ep, void* C, int c_dtype, cudaStream_t s) {
    const int threads = 256;
    const size_t want = ((size_t)M * N + threads - 1) / threads;
    const int blocks = (int)(want < 8192 ? want : 8192);
    switch (c_dtype) {
        case DT_F32: pf::w4a8_rescale_kernel<DT_F32><<<blocks, threads, 0, s>>>(M, N, acc, as, rowsum, T, ep, C); break;
        case DT_F16: pf::w4a8_rescale_kernel<DT_F16><<<blocks, threads, 0, s>>>(M, N, acc, as, rowsum, T, ep, C); break;
        default: pf::w4a8_rescale_kernel<DT_BF16><<<blocks, threads, 0, s>>>(M, N, acc, as, rowsum, T, ep, C); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_prefill_codes8(const pf::Maps& maps, const pf::Params& p, int kdt, cudaStream_t s) {
    return pf::launch_wf<pf::WF_CODES8, true, pf::EPI_W4A8>(maps, p, kdt, s);
}

cudaError_t launch_w4a8_gemm(const W4A8Args& a, cudaStream_t s) {
    pf::Params p{};
    const int block = a.block > 0 ? a.block : a.K;
    p.M = a.M; p.K = a.K; p.N = a.N; p.block = block; p.nb = a.K / block;
    p.BN = pf::pick_bn(a.M);
    p.Bp = static_cast<const uint8_t*>(a.Bp); p.T = a.T; p.C = a.C;
    p.a_scale = a.as; p.rowsum = a.rowsum; p.acc = a.acc;
    p.splits = a.splits > 1 ? a.splits : 1;
    p.acc_add = a.acc_add;
    if (p.splits > 1 && !(a.acc && a.acc_add)) return cudaErrorInvalidValue;   // K-chunks add int32 sums
    p.status = status_word_address();
    if (!p.status) return cudaErrorInvalidValue;
    p.wait_ns = option_wait_ns();
    p.stall = option_stall();
    p.ep = a.acc ? Epilogue{} : a.ep;
    p.rowmax = a.acc ? nullptr : a.rowmax;
    pf::Maps maps;
    cudaError_t e = pf::make_tmap(&maps.a, a.qa16, false, a.M, a.K, p.BN);
    if (e != cudaSuccess) return e;
    p.c_tma = a.acc ? (pf::make_out_map(&maps.c, a.acc, -1, a.M, a.N, pf::kSlabRows, 1) ? 1 : 0)
                    : (pf::make_out_map(&maps.c, a.C, a.c_dtype, a.M, a.N, pf::kSlabRows, 1) ? 1 : 0);
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
