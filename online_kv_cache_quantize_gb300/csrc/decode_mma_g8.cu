// Tensor-core decode scan instantiations for 8 query head(s) per KV head.
#include "decode_mma.cuh"

namespace tqk {

cudaError_t launch_decode_mma_g8(const DecodeParams& p, int kbits, int vbits, bool two, cudaStream_t s) {
    return dispatch_decode_mma<8>(p, kbits, vbits, two, s);
}

}  // namespace tqk
