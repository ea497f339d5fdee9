// The tcgen05 quantize kernel (quantize_umma.cuh) for fractional-rate caches:
// two channel groups, the second one code bit narrower.
#include "quantize_umma.cuh"

namespace tqk {

cudaError_t launch_quantize_umma2(const QuantUmmaParams& P, int rht, int prod, int code_bits, cudaStream_t s) {
    constexpr int NP = kQuParts;
#define TQ_QU2(CBV, PR)                                                                          \
    if (code_bits == CBV && (prod != 0) == PR)                                                   \
        return rht ? go_qu<CBV, CBV - 1, PR, true, NP>(P, s) : go_qu<CBV, CBV - 1, PR, false, NP>(P, s);
    TQ_QU2(2, false)
    TQ_QU2(3, false)
    TQ_QU2(4, false)
    TQ_QU2(2, true)
    TQ_QU2(3, true)
#undef TQ_QU2
    return cudaErrorNotSupported;
}

}  // namespace tqk
