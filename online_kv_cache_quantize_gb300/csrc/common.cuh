// Device helpers shared by the libtq kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define TQ_FULL_MASK 0xffffffffu

namespace tqk {

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(TQ_FULL_MASK, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(TQ_FULL_MASK, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(TQ_FULL_MASK, v, o));
    return v;
}

// float -> fp16 bits, round to nearest even, saturated at 65504 (the packed
// cache never stores an infinity).
__device__ __forceinline__ uint16_t f16_bits_sat(float v) {
    v = fminf(fmaxf(v, -65504.0f), 65504.0f);
    return __half_as_ushort(__float2half_rn(v));
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// fp16 bits of v (lo = 0) or of v - fp16(v) (lo = 1): the hi/lo split that
// carries an fp32 operand into fp16 tensor-core products
__device__ __forceinline__ uint32_t half_split(float v, int lo) {
    __half h = __float2half_rn(v);
    if (lo) h = __float2half_rn(v - __half2float(h));
    return (uint32_t)__half_as_ushort(h);
}

// Bits [off, off + nbits) of a little-endian bit stream held in 32-bit words,
// nbits <= 32, reading at most words[off/32] and words[off/32 + 1].
__device__ __forceinline__ uint32_t stream_bits(const uint32_t* words, int off, int nbits, int nwords) {
    int w = off >> 5, sh = off & 31;
    uint32_t lo = words[w];
    uint32_t hi = (w + 1 < nwords) ? words[w + 1] : 0u;
    uint32_t v = __funnelshift_r(lo, hi, sh);
    return nbits >= 32 ? v : (v & ((1u << nbits) - 1u));
}

}  // namespace tqk
