// tcgen05 chunked-prefill instantiations (prefill_umma.cuh): keys at 1 or 2
// code bits (PROD 2 / 3 bits, or the 3 / 2 fractional rate) with values at
// 1..4 bits; 1-bit keys here, 2-bit keys in prefill_umma2.cu.
#include "prefill_umma.cuh"

namespace tqk {

cudaError_t launch_prefill_umma_k2(const PrefillParams& p, int vbits, bool two, cudaStream_t s);

bool prefill_umma_supported(int kbits, int vbits, bool two) {
    if (two) return kbits == 2 && vbits >= 2 && vbits <= 4;
    return (kbits == 1 || kbits == 2) && vbits >= 1 && vbits <= 4;
}

cudaError_t launch_prefill_umma(const PrefillParams& p, int kbits, int vbits, bool two, cudaStream_t s) {
    if (p.chunk <= 0 || p.batch <= 0 || p.n_splits <= 0) return cudaSuccess;
    if (!prefill_umma_supported(kbits, vbits, two)) return cudaErrorInvalidValue;
    if (kbits == 2) return launch_prefill_umma_k2(p, vbits, two, s);
    switch (vbits) {
        case 1: return launch_prefill_umma_t<1, 1, 1, 1>(p, s);
        case 2: return launch_prefill_umma_t<1, 2, 1, 2>(p, s);
        case 3: return launch_prefill_umma_t<1, 3, 1, 3>(p, s);
        case 4: return launch_prefill_umma_t<1, 4, 1, 4>(p, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tqk
