// Tensor-core chunked-prefill instantiations: every single-width (KB, VB) in
// 1..4, and fractional-rate caches with keys and values both in two groups
// (KB2 = KB - 1, VB2 = VB - 1).
#include "prefill_mma.cuh"

namespace tqk {

template <int KB, int KB2>
static cudaError_t prefill_v(const PrefillParams& p, int vb, cudaStream_t s) {
    constexpr bool two = KB2 != KB;
    switch (vb) {
        case 1:
            if constexpr (!two) return launch_prefill_mma_t<KB, 1>(p, s);
            break;
        case 2: return launch_prefill_mma_t<KB, 2, KB2, two ? 1 : 2>(p, s);
        case 3: return launch_prefill_mma_t<KB, 3, KB2, two ? 2 : 3>(p, s);
        case 4: return launch_prefill_mma_t<KB, 4, KB2, two ? 3 : 4>(p, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_mma(const PrefillParams& p, int kbits, int vbits, bool two, cudaStream_t s) {
    if (p.chunk <= 0 || p.batch <= 0 || p.n_splits <= 0) return cudaSuccess;
    if (!two) {
        switch (kbits) {
            case 1: return prefill_v<1, 1>(p, vbits, s);
            case 2: return prefill_v<2, 2>(p, vbits, s);
            case 3: return prefill_v<3, 3>(p, vbits, s);
            case 4: return prefill_v<4, 4>(p, vbits, s);
        }
    } else {
        switch (kbits) {
            case 2: return prefill_v<2, 1>(p, vbits, s);
            case 3: return prefill_v<3, 2>(p, vbits, s);
            case 4: return prefill_v<4, 3>(p, vbits, s);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace tqk
