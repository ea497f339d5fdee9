// Tensor-core decode scan instantiations for 1 query head(s) per KV head.
#include "decode_mma.cuh"

namespace tqk {

cudaError_t launch_decode_mma_g1(const DecodeParams& p, int kbits, int vbits, bool two, cudaStream_t s) {
    return dispatch_decode_mma<1>(p, kbits, vbits, two, s);
}

}  // namespace tqk
