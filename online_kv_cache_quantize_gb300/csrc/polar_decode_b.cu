// PolarQuant decode scan instantiations for 4 and 8 query heads per KV head.
#include "polar_decode.cuh"

namespace tqk {

cudaError_t launch_polar_decode_g48(const PolarDecodeParams& p, int b1, int b2, cudaStream_t s) {
    if (p.group == 4) return dispatch_polar_decode<4>(p, b1, b2, s);
    if (p.group == 8) return dispatch_polar_decode<8>(p, b1, b2, s);
    return cudaErrorInvalidValue;
}

}  // namespace tqk
