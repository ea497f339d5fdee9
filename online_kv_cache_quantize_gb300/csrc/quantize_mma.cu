// Tensor-core quantize-on-append instantiations (d = m = 128).
#include "quantize_mma.cuh"

namespace tqk {

template <typename XT, int CB, bool PROD, bool RHT>
static cudaError_t go(const QuantParams& p, cudaStream_t s) {
    if (p.n <= 0) return cudaSuccess;
    auto kern = quantize_mma_kernel<XT, CB, PROD, RHT>;
    constexpr int NW = qm_warps<XT, RHT>();
    constexpr size_t smem = quantize_mma_smem<XT, CB, PROD, RHT>();
    static_assert(smem + kMaxLevels * sizeof(float) <= kQmSmemLimit, "shared memory above the per-CTA limit");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t tiles = (p.n + 15) / 16;
    int64_t blocks = (tiles + NW - 1) / NW;
    if (blocks > (int64_t)sms * per_sm) blocks = (int64_t)sms * per_sm;
    kern<<<(unsigned)blocks, NW * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename XT, bool PROD, bool RHT>
static cudaError_t go_cb(const QuantParams& p, int cb, cudaStream_t s) {
    switch (cb) {
        case 1: return go<XT, 1, PROD, RHT>(p, s);
        case 2: return go<XT, 2, PROD, RHT>(p, s);
        case 3: return go<XT, 3, PROD, RHT>(p, s);
        case 4: return go<XT, 4, PROD, RHT>(p, s);
    }
    return cudaErrorInvalidValue;
}

template <typename XT>
static cudaError_t go_x(const QuantParams& p, int rht, int prod, int cb, cudaStream_t s) {
    if (rht) return prod ? go_cb<XT, true, true>(p, cb, s) : go_cb<XT, false, true>(p, cb, s);
    return prod ? go_cb<XT, true, false>(p, cb, s) : go_cb<XT, false, false>(p, cb, s);
}

cudaError_t launch_quantize_mma(const QuantParams& p, int dtype, int rht, int prod, int cb, cudaStream_t s) {
    return dtype == 0 ? go_x<float>(p, rht, prod, cb, s) : go_x<__nv_bfloat16>(p, rht, prod, cb, s);
}

}  // namespace tqk
