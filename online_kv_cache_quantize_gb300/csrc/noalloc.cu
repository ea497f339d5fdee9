// Decode attention for callers that must not allocate device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocator) at
// the point where they run decode: an engine plugin whose host owns every
// byte of device memory, work enqueued while a CUDA graph is being captured,
// or a runtime that forbids allocation after start-up. tq_attn_decode needs
// a caller-provided workspace; tq_attn_decode_static instead uses a scratch
// array compiled into the library, so the caller passes only its inputs and
// outputs. The array is held by every device that loads the library until
// the process exits.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "tq_internal.h"

// File-scope scratch. In host code this name is only a host-side stand-in for
// the device array: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_tq_decode_scratch[TQ_STATIC_DECODE_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" tq_status tq_attn_decode_static(const tq_decode_args* a, tq_stream stream) {
    if (!a) return tq::fail(TQ_ERR_INVALID_ARG, "tq_attn_decode_static: args are NULL");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tq::fail(TQ_ERR_CUDA, std::string("tq_attn_decode_static: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return tq::fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode_static: device ordinal >= 64");
    void* ptr = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mutex);
        if (!g_scratch_addr[dev]) {
            // once per device, with that device current
            e = cudaGetSymbolAddress(&ptr, g_tq_decode_scratch);
            if (e != cudaSuccess)
                return tq::fail(TQ_ERR_CUDA, std::string("tq_attn_decode_static: cudaGetSymbolAddress: ") +
                                                 cudaGetErrorString(e));
            g_scratch_addr[dev] = ptr;
        }
        ptr = g_scratch_addr[dev];
    }
    // tq_attn_decode checks every argument first and the scratch size last,
    // so an invalid call gets the same status here as there; only the
    // message of a too-small scratch is made specific to the static array.
    // Every scratch byte the decode reads is written earlier in the same
    // call, so nothing needs clearing between calls.
    const tq_status s = tq_attn_decode(a, ptr, (size_t)TQ_STATIC_DECODE_SCRATCH_BYTES, stream);
    if (s == TQ_ERR_WORKSPACE)
        return tq::fail(TQ_ERR_WORKSPACE, "tq_attn_decode_static: these arguments need " +
                                              std::to_string(tq_attn_decode_workspace(a)) +
                                              " bytes of scratch; the static array holds " +
                                              std::to_string((size_t)TQ_STATIC_DECODE_SCRATCH_BYTES) +
                                              " (use tq_attn_decode with a workspace)");
    return s;
}
