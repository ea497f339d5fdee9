// The tcgen05 quantize kernel (quantize_umma.cuh) for one code width.
#include "quantize_umma.cuh"

namespace tqk {

bool quantize_umma_supported(const QuantParams& p, int dtype, int code_bits) {
    if (!qu_shape_ok(p, dtype) || code_bits < 1) return false;
    if (p.code_bits2 == 0) return code_bits <= (p.m == 128 ? 3 : 4);
    // fractional-rate caches: the second group one bit narrower; keys (PROD)
    // 2/1 and 3/2 code bits, values 2/1, 3/2, 4/3
    return p.code_bits2 == code_bits - 1 && code_bits >= 2 && code_bits <= (p.m == 128 ? 3 : 4);
}

cudaError_t launch_quantize_umma2(const QuantUmmaParams& P, int rht, int prod, int code_bits, cudaStream_t s);

cudaError_t launch_quantize_umma(const QuantParams& p, const void* w_umma, const void* s_umma, int rht, int prod,
                                 int code_bits, cudaStream_t s) {
    if (p.n <= 0) return cudaSuccess;
    QuantUmmaParams P;
    cudaError_t e = qu_params(p, w_umma, s_umma, &P);
    if (e != cudaSuccess) return e;
    if (p.code_bits2 != 0) return launch_quantize_umma2(P, rht, prod, code_bits, s);
    constexpr int NP = kQuParts;
    // keys (PROD) have 1..3 code bits (2..4 bits with the sign bit), values 1..4
#define TQ_QU_MSE(CBV) \
    if (code_bits == CBV && !prod)                                                                         \
        return rht ? go_qu<CBV, CBV, false, true, NP>(P, s) : go_qu<CBV, CBV, false, false, NP>(P, s);
#define TQ_QU_PROD(CBV) \
    if (code_bits == CBV && prod) return rht ? go_qu<CBV, CBV, true, true, NP>(P, s) : go_qu<CBV, CBV, true, false, NP>(P, s);
    TQ_QU_MSE(1)
    TQ_QU_MSE(2)
    TQ_QU_MSE(3)
    TQ_QU_MSE(4)
    TQ_QU_PROD(1)
    TQ_QU_PROD(2)
    TQ_QU_PROD(3)
#undef TQ_QU_MSE
#undef TQ_QU_PROD
    return cudaErrorNotSupported;
}

}  // namespace tqk
