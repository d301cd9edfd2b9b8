// Decode kernel instantiations for int8 weights: the TMA-fed kernel (decode_stream.cuh) where the
// shape suits it, else the cp.async kernel (decode_kernel.cuh).
#include "decode_stream.cuh"

namespace qg {

cudaError_t launch_decode_int8(const DecodeArgs& a, cudaStream_t s) {
    const bool bf = a.a_dtype == DT_BF16;
    if (dstream::supported<FMT_INT8>(a))
        return bf ? dstream::launch_fmt<FMT_INT8, true>(a, s) : dstream::launch_fmt<FMT_INT8, false>(a, s);
    return bf ? dec::launch_fmt<FMT_INT8, true>(a, s) : dec::launch_fmt<FMT_INT8, false>(a, s);
}

}  // namespace qg
