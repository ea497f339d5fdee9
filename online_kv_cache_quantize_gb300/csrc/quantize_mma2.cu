// Tensor-core quantize-on-append instantiations for fractional-rate caches
// (d = m = 128): coordinates with i % 16 < 8 at CB code bits, the rest at
// CB - 1, each group with its own codebook.
#include "quantize_mma.cuh"

namespace tqk {

template <typename XT, bool PROD, bool RHT>
static cudaError_t go_cb2(const QuantParams& p, int cb, cudaStream_t s) {
    switch (cb) {
        case 2: return launch_quantize_mma_t<XT, 2, PROD, RHT, 1>(p, s);
        case 3: return launch_quantize_mma_t<XT, 3, PROD, RHT, 2>(p, s);
        case 4: return launch_quantize_mma_t<XT, 4, PROD, RHT, 3>(p, s);
    }
    return cudaErrorInvalidValue;
}

template <typename XT>
static cudaError_t go_x2(const QuantParams& p, int rht, int prod, int cb, cudaStream_t s) {
    if (rht) return prod ? go_cb2<XT, true, true>(p, cb, s) : go_cb2<XT, false, true>(p, cb, s);
    return prod ? go_cb2<XT, true, false>(p, cb, s) : go_cb2<XT, false, false>(p, cb, s);
}

cudaError_t launch_quantize_mma2(const QuantParams& p, int dtype, int rht, int prod, int cb, cudaStream_t s) {
    if (p.code_bits2 != cb - 1) return cudaErrorInvalidValue;
    return dtype == 0 ? go_x2<float>(p, rht, prod, cb, s) : go_x2<__nv_bfloat16>(p, rht, prod, cb, s);
}

}  // namespace tqk
