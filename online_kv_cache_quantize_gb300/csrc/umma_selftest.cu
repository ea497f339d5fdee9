// Self-test of the tcgen05 building blocks: one CTA computes D = A B^T with
// A [128 x K] and B [N x K] fp16 (K contiguous in global memory), D fp32
// [128 x N], through shared-memory core-matrix tiles, tcgen05.mma into TMEM
// and tcgen05.ld back. Used by the tests to pin the descriptor encodings
// against a CPU matmul before any kernel relies on them.
#include "pipeline.cuh"
#include "tcgen05.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kUmmaTestMaxK = 128;

// A_TMEM: A is written into TMEM with tcgen05.st (row r in lane r, column
// 128 + k / 2 holding elements k, k + 1) and the MMA reads it from there.
template <bool A_TMEM>
__global__ void __launch_bounds__(128) umma_selftest_kernel(const __half* __restrict__ A, const __half* __restrict__ B,
                                                            float* __restrict__ D, int N, int K, uint32_t* err) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_tmem;
    unsigned char* sa = smem;                       // [128 x K]
    unsigned char* sb = smem + 128 * K * 2;         // [N x K], room for 128 rows
    const int tid = threadIdx.x, warp = tid >> 5;

    // operands into the core-matrix layout, two fp16 (one 32-bit word) at a time
    if (!A_TMEM)
        for (int e = tid; e < 128 * K / 2; e += blockDim.x) {
            const int r = (2 * e) / K, k = (2 * e) % K;
            *reinterpret_cast<uint32_t*>(sa + umma_off(r, k, K)) = *reinterpret_cast<const uint32_t*>(A + (size_t)r * K + k);
        }
    for (int e = tid; e < N * K / 2; e += blockDim.x) {
        const int r = (2 * e) / K, k = (2 * e) % K;
        *reinterpret_cast<uint32_t*>(sb + umma_off(r, k, K)) = *reinterpret_cast<const uint32_t*>(B + (size_t)r * K + k);
    }
    const uint32_t bar_a = (uint32_t)__cvta_generic_to_shared(&bar);
    if (tid == 0) {
        mbar_init(bar_a, 1);
        mbar_init_fence();
    }
    fence_proxy_async_smem();  // generic-proxy tile writes before the tensor core reads them
    // 256 columns, twice the largest n: a single test CTA can afford the margin
    const uint32_t ncols = 256;
    if (warp == 0) {
        tmem_alloc((uint32_t)__cvta_generic_to_shared(&s_tmem), ncols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;
    if (A_TMEM) {
        // thread t of warp w: row 32 w + t into its lane, 8 columns per store
        const int row = 32 * warp + (tid & 31);
        for (int c0 = 0; c0 < K / 2; c0 += 8) {
            uint32_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = *reinterpret_cast<const uint32_t*>(A + (size_t)row * K + 2 * (c0 + j));
            tmem_st8(tmem + ((uint32_t)(32 * warp) << 16) + 128u + (uint32_t)c0, v);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
    }

    if (tid == 0) {
        const uint32_t a0 = (uint32_t)__cvta_generic_to_shared(sa), b0 = (uint32_t)__cvta_generic_to_shared(sb);
        const uint32_t idesc = umma_idesc_f16(128, N);
        for (int s = 0; s < K / 16; ++s) {
            if (A_TMEM)
                umma_f16_ta(tmem, tmem + 128u + 8u * s, umma_desc(b0 + 256 * s, 128, K * 16), idesc, s > 0);
            else
                umma_f16(tmem, umma_desc(a0 + 256 * s, 128, K * 16), umma_desc(b0 + 256 * s, 128, K * 16), idesc, s > 0);
        }
        umma_commit(bar_a);
    }
    __syncwarp();
    const bool done = mbar_wait_bounded(bar_a, 0, kWaitLimitNs, err, kErrSelfTestWait);
    tc_fence_after_sync();
    if (__all_sync(TQ_FULL_MASK, done)) {
        const int row = 32 * warp + (tid & 31);
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) D[(size_t)row * N + c0 + j] = v[j];
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, ncols);
}

cudaError_t launch_umma_selftest(const void* a, const void* b, float* d, int n, int k, int a_tmem, uint32_t* err,
                                 cudaStream_t s) {
    if ((n != 16 && n != 32 && n != 64 && n != 128) || k < 16 || k > kUmmaTestMaxK || k % 16)
        return cudaErrorInvalidValue;
    // B gets room for 128 rows whatever n is, so that every address an MMA
    // could form from these descriptors stays inside the allocation
    const size_t smem = (size_t)(128 + 128) * k * 2;
    auto kern = a_tmem ? umma_selftest_kernel<true> : umma_selftest_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<1, 128, smem, s>>>(static_cast<const __half*>(a), static_cast<const __half*>(b), d, n, k, err);
    return cudaGetLastError();
}

}  // namespace tqk
