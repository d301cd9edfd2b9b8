// Tensor-core decode kernel instantiations for int4 weights (see decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace qg {

cudaError_t launch_decode_int4(const DecodeArgs& a, cudaStream_t s) {
    return a.a_dtype == DT_BF16 ? dec::launch_fmt<FMT_INT4, true>(a, s) : dec::launch_fmt<FMT_INT4, false>(a, s);
}

}  // namespace qg
