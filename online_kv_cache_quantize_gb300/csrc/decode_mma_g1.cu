// Tensor-core decode scan instantiations for 1 query head(s) per KV head.
#include "decode_mma.cuh"

namespace tqk {

template <int KB, int VB>
static cudaError_t go(const DecodeParams& p, cudaStream_t s) {
    return launch_decode_mma_t<KB, VB, 1>(p, s);
}

template <int KB>
static cudaError_t go_k(const DecodeParams& p, int vbits, cudaStream_t s) {
    switch (vbits) {
        case 1: return go<KB, 1>(p, s);
        case 2: return go<KB, 2>(p, s);
        case 3: return go<KB, 3>(p, s);
        case 4: return go<KB, 4>(p, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_mma_g1(const DecodeParams& p, int kbits, int vbits, cudaStream_t s) {
    switch (kbits) {
        case 1: return go_k<1>(p, vbits, s);
        case 2: return go_k<2>(p, vbits, s);
        case 3: return go_k<3>(p, vbits, s);
        case 4: return go_k<4>(p, vbits, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tqk
