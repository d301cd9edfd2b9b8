// Tensor-core decode kernel instantiations for int8 weights (see decode_kernel.cuh).
#include "decode_kernel.cuh"

namespace qg {

cudaError_t launch_decode_int8(const DecodeArgs& a, cudaStream_t s) {
    return a.a_dtype == DT_BF16 ? dec::launch_fmt<FMT_INT8, true>(a, s) : dec::launch_fmt<FMT_INT8, false>(a, s);
}

}  // namespace qg
