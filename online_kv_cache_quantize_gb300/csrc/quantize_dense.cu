// Quantize-on-append, dense QR rotation instantiations.
#include "quantize.cuh"

namespace tqk {

cudaError_t launch_quantize_dense(const QuantParams& p, int dtype, int vpl, int prod, int cb, cudaStream_t s) {
    if (dtype == 0) {
        switch (vpl) {
            case 2: return launch_quantize_t<float, 2, false>(p, prod, cb, s);
            case 4: return launch_quantize_t<float, 4, false>(p, prod, cb, s);
            case 7: return launch_quantize_t<float, 7, false>(p, prod, cb, s);
            case 8: return launch_quantize_t<float, 8, false>(p, prod, cb, s);
        }
    } else {
        switch (vpl) {
            case 2: return launch_quantize_t<__nv_bfloat16, 2, false>(p, prod, cb, s);
            case 4: return launch_quantize_t<__nv_bfloat16, 4, false>(p, prod, cb, s);
            case 7: return launch_quantize_t<__nv_bfloat16, 7, false>(p, prod, cb, s);
            case 8: return launch_quantize_t<__nv_bfloat16, 8, false>(p, prod, cb, s);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace tqk
