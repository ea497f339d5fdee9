// Top-k search launches.
#include "topk.cuh"

namespace tqk {

template <int VPL, int CB>
static cudaError_t launch_topk_vc(const TopkParams& p, int prod, cudaStream_t s) {
    dim3 grid(p.n_chunks, (p.nq + kTopkQ - 1) / kTopkQ), block(kTopkWarps * 32);
    if (prod) topk_scan_kernel<VPL, CB, true><<<grid, block, 0, s>>>(p);
    else topk_scan_kernel<VPL, CB, false><<<grid, block, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    topk_merge_kernel<<<(p.nq + 7) / 8, 256, 0, s>>>(p);
    return cudaGetLastError();
}

template <int VPL>
static cudaError_t launch_topk_v(const TopkParams& p, int cb, int prod, cudaStream_t s) {
    switch (cb) {
        case 1: return launch_topk_vc<VPL, 1>(p, prod, s);
        case 2: return launch_topk_vc<VPL, 2>(p, prod, s);
        case 3: return launch_topk_vc<VPL, 3>(p, prod, s);
        case 4: return launch_topk_vc<VPL, 4>(p, prod, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_topk(const TopkParams& p, int cb, int prod, cudaStream_t s) {
    if (p.d <= 64) return launch_topk_v<2>(p, cb, prod, s);
    if (p.d <= 128) return launch_topk_v<4>(p, cb, prod, s);
    if (p.d <= 224) return launch_topk_v<7>(p, cb, prod, s);
    return launch_topk_v<8>(p, cb, prod, s);
}

}  // namespace tqk
