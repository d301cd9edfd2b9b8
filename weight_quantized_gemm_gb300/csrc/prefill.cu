// Tensor-core (tcgen05 / TMEM / TMA) kernels for large M and for W4A8, and the device status
// word that bounded waits report into.
#include "internal.h"

namespace qg {

// Set (bitwise OR) by a kernel that gave up a bounded wait; read and cleared by qgemm_status.
__device__ unsigned int g_status_word;

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

bool prefill_supported(int, int, int, int, int) { return false; }
cudaError_t launch_prefill(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_w4a8_gemm(const W4A8Args&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace qg
