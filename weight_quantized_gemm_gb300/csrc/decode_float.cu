// Tensor-core decode kernel instantiations for float weights (see decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace qg {

cudaError_t launch_decode_float(const DecodeArgs& a, cudaStream_t s) {
    return a.a_dtype == DT_BF16 ? dec::launch_fmt<FMT_FLOAT, true>(a, s) : dec::launch_fmt<FMT_FLOAT, false>(a, s);
}

}  // namespace qg
