// The library's device error word and the self-test of the bounded wait.
#include <mutex>

#include "pipeline.cuh"
#include "tq_launch.h"

// In host code this name is only a stand-in for the device word: its device
// address comes from cudaGetSymbolAddress, once per device.
static __device__ uint32_t g_tq_device_errors;

namespace tqk {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_err_mutex;
uint32_t* g_err_addr[kMaxDevices] = {};
}  // namespace

cudaError_t device_error_word(uint32_t** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_err_mutex);
    if (!g_err_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_tq_device_errors);
        if (e != cudaSuccess) return e;
        g_err_addr[dev] = static_cast<uint32_t*>(p);
    }
    *out = g_err_addr[dev];
    return cudaSuccess;
}

// One warp waits on a freshly initialised mbarrier that nothing arrives on:
// every lane's bounded wait runs out and sets kErrSelfTestWait.
__global__ void wait_selftest_kernel(uint32_t* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(&bar);
    if (threadIdx.x == 0) {
        mbar_init(a, 1);
        mbar_init_fence();
    }
    __syncwarp();
    mbar_wait_bounded(a, 0, limit_ns, err, kErrSelfTestWait);
}

cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace tqk
