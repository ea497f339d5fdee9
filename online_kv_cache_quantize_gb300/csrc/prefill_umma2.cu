// tcgen05 chunked-prefill instantiations with 2-bit keys (prefill_umma.cuh):
// single-width values at 1..4 bits, and the fractional-rate caches (keys 2/1,
// values 2/1, 3/2, 4/3 code bits).
#include "prefill_umma.cuh"

namespace tqk {

cudaError_t launch_prefill_umma_k2(const PrefillParams& p, int vbits, bool two, cudaStream_t s) {
    if (!two) {
        switch (vbits) {
            case 1: return launch_prefill_umma_t<2, 1, 2, 1>(p, s);
            case 2: return launch_prefill_umma_t<2, 2, 2, 2>(p, s);
            case 3: return launch_prefill_umma_t<2, 3, 2, 3>(p, s);
            case 4: return launch_prefill_umma_t<2, 4, 2, 4>(p, s);
        }
    } else {
        switch (vbits) {
            case 2: return launch_prefill_umma_t<2, 2, 1, 1>(p, s);
            case 3: return launch_prefill_umma_t<2, 3, 1, 2>(p, s);
            case 4: return launch_prefill_umma_t<2, 4, 1, 3>(p, s);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace tqk
