// PolarQuant decode scan instantiations for 1 and 2 query heads per KV head.
#include "polar_decode.cuh"

namespace tqk {

cudaError_t launch_polar_decode_g12(const PolarDecodeParams& p, int b1, int b2, cudaStream_t s) {
    if (p.group == 1) return dispatch_polar_decode<1>(p, b1, b2, s);
    if (p.group == 2) return dispatch_polar_decode<2>(p, b1, b2, s);
    return cudaErrorInvalidValue;
}

}  // namespace tqk
