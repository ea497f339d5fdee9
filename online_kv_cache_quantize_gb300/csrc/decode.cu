// Decode attention launches: query preparation, split-K scan dispatch, merge.
#include "decode.cuh"

namespace tqk {

cudaError_t launch_query_prep(const PrepParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    dim3 grid((unsigned)p.rows), block(kPrepWarps * 32);
    if (p.d <= 64) query_prep_kernel<2><<<grid, block, 0, s>>>(p);
    else if (p.d <= 128) query_prep_kernel<4><<<grid, block, 0, s>>>(p);
    else if (p.d <= 224) query_prep_kernel<7><<<grid, block, 0, s>>>(p);
    else query_prep_kernel<8><<<grid, block, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode_mma_g1(const DecodeParams& p, int kbits, int vbits, cudaStream_t s);
cudaError_t launch_decode_mma_g2(const DecodeParams& p, int kbits, int vbits, cudaStream_t s);
cudaError_t launch_decode_mma_g4(const DecodeParams& p, int kbits, int vbits, cudaStream_t s);
cudaError_t launch_decode_mma_g8(const DecodeParams& p, int kbits, int vbits, cudaStream_t s);

cudaError_t launch_decode_mma(const DecodeParams& p, int kbits, int vbits, cudaStream_t s) {
    switch (p.group) {
        case 1: return launch_decode_mma_g1(p, kbits, vbits, s);
        case 2: return launch_decode_mma_g2(p, kbits, vbits, s);
        case 4: return launch_decode_mma_g4(p, kbits, vbits, s);
        case 8: return launch_decode_mma_g8(p, kbits, vbits, s);
    }
    return cudaErrorInvalidValue;
}

// Programmatic dependent launch: the merge's CTAs may be scheduled while the
// scan's last CTAs still run (the scan signals launch_dependents once its
// tiles are done); the merge waits for the scan grid to complete before it
// reads a partial (griddepcontrol.wait).
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.rows);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace tqk
