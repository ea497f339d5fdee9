// Tensor-core quantize-on-append instantiations (d = m = 128).
#include "quantize_mma.cuh"

namespace tqk {

template <typename XT, int CB, bool PROD, bool RHT>
static cudaError_t go(const QuantParams& p, cudaStream_t s) {
    return launch_quantize_mma_t<XT, CB, PROD, RHT>(p, s);
}

template <typename XT, bool PROD, bool RHT>
static cudaError_t go_cb(const QuantParams& p, int cb, cudaStream_t s) {
    switch (cb) {
        case 1: return go<XT, 1, PROD, RHT>(p, s);
        case 2: return go<XT, 2, PROD, RHT>(p, s);
        case 3: return go<XT, 3, PROD, RHT>(p, s);
        case 4: return go<XT, 4, PROD, RHT>(p, s);
    }
    return cudaErrorInvalidValue;
}

template <typename XT>
static cudaError_t go_x(const QuantParams& p, int rht, int prod, int cb, cudaStream_t s) {
    if (rht) return prod ? go_cb<XT, true, true>(p, cb, s) : go_cb<XT, false, true>(p, cb, s);
    return prod ? go_cb<XT, true, false>(p, cb, s) : go_cb<XT, false, false>(p, cb, s);
}

cudaError_t launch_quantize_mma(const QuantParams& p, int dtype, int rht, int prod, int cb, cudaStream_t s) {
    return dtype == 0 ? go_x<float>(p, rht, prod, cb, s) : go_x<__nv_bfloat16>(p, rht, prod, cb, s);
}

}  // namespace tqk
