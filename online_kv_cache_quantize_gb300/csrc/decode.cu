// Decode attention launches: query preparation, split-K scan, merge.
#include "decode.cuh"

namespace tqk {

cudaError_t launch_query_prep(const PrepParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    dim3 grid((unsigned)((p.rows + 7) / 8)), block(256);
    if (p.d <= 64) query_prep_kernel<2><<<grid, block, 0, s>>>(p);
    else if (p.d <= 128) query_prep_kernel<4><<<grid, block, 0, s>>>(p);
    else if (p.d <= 224) query_prep_kernel<7><<<grid, block, 0, s>>>(p);
    else query_prep_kernel<8><<<grid, block, 0, s>>>(p);
    return cudaGetLastError();
}

template <int KB, int VB>
static cudaError_t launch_decode_kv(const DecodeParams& p, dim3 grid, cudaStream_t s) {
    dim3 block(kDecWarps * 32);
    switch (p.group) {
        case 1: decode_kernel<KB, VB, 1><<<grid, block, 0, s>>>(p); break;
        case 2: decode_kernel<KB, VB, 2><<<grid, block, 0, s>>>(p); break;
        case 4: decode_kernel<KB, VB, 4><<<grid, block, 0, s>>>(p); break;
        case 8: decode_kernel<KB, VB, 8><<<grid, block, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int KB>
static cudaError_t launch_decode_k(const DecodeParams& p, int vbits, dim3 grid, cudaStream_t s) {
    switch (vbits) {
        case 1: return launch_decode_kv<KB, 1>(p, grid, s);
        case 2: return launch_decode_kv<KB, 2>(p, grid, s);
        case 3: return launch_decode_kv<KB, 3>(p, grid, s);
        case 4: return launch_decode_kv<KB, 4>(p, grid, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const DecodeParams& p, int kbits, int vbits, cudaStream_t s) {
    dim3 grid(p.n_splits, p.hkv, p.batch);
    switch (kbits) {
        case 1: return launch_decode_k<1>(p, vbits, grid, s);
        case 2: return launch_decode_k<2>(p, vbits, grid, s);
        case 3: return launch_decode_k<3>(p, vbits, grid, s);
        case 4: return launch_decode_k<4>(p, vbits, grid, s);
    }
    return cudaErrorInvalidValue;
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

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    combine_kernel<<<p.rows, p.d, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tqk
