// Decode attention launches: query preparation (fused with the decode
// step's appends), split-K scan dispatch, merge.
#include "append.cuh"
#include "decode.cuh"

namespace tqk {

// The decode step's work before its scan in one launch: query prep rows
// (decode.cuh) and the appended key and value vectors (append.cuh).
__global__ void __launch_bounds__(kPrepWarps * 32) step_prep_kernel(const __grid_constant__ StepPrepParams p) {
    // the scan that follows on the stream may be scheduled now: it waits for
    // this grid to complete before it reads anything written here
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    __shared__ AppendSmem s;
    int64_t b = blockIdx.x;
    if (b < p.pp.rows) {
        prep_row<4>(p.pp, b);
        return;
    }
    b -= p.pp.rows;
    if (threadIdx.x >= kAppendThreads) return;
    if (b < p.k.n) {
        append_vector(p.k, p.k_dtype, p.k_cb, true, p.k_rht != 0, b, s);
        return;
    }
    b -= p.k.n;
    if (b < p.v.n) append_vector(p.v, p.v_dtype, p.v_cb, false, p.v_rht != 0, b, s);
}

cudaError_t launch_step_prep(const StepPrepParams& p, cudaStream_t s) {
    const int64_t ctas = p.pp.rows + p.k.n + p.v.n;
    if (ctas <= 0) return cudaSuccess;
    if (ctas > 0x7fffffff || (p.pp.rows > 0 && p.pp.d != 128) || (p.k.n > 0 && (p.k.d != 128 || p.k.m != 128)) ||
        (p.v.n > 0 && p.v.d != 128))
        return cudaErrorInvalidValue;
    step_prep_kernel<<<(unsigned)ctas, kPrepWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

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
