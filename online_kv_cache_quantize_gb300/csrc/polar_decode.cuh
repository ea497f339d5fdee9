// Split-K decode scan over PolarQuant keys and MSE values (d = 128): the
// comparison variant of the DeepSignal TurboQuant article ("PolarQuant") and
// the A2A TurboQuant explainer ("Stage 1" PolarQuant bullets), scored from the
// stored angle codes with the query rotated once:
//   l_t = n_t <q', y_hat_t>,  y_hat_t the inverse recursion of the centroid
//   angles (level 7 down to the coordinate pairs);
//   p = softmax(scale * l),  a = sum_t p_t nV_t cV[idxV_t]  (rotated domain).
// The merge of the splits and the un-rotation o = Pi^T a are the TurboQuant
// decode's (combine_kernel).
//
// The dot product is evaluated bottom-up over the recursion tree without
// forming y_hat: a level-1 pair contributes q'_2i cos c + q'_2i+1 sin c, a
// table of every pair and code per query head built once per CTA, and a
// node of level l combines its children as cos(c_l) left + sin(c_l) right.
// One thread per token for the keys (its codes in registers, offsets known
// at compile time); one warp per token for the values (lane l owns
// coordinates 4l .. 4l+3, two codes per table lookup). Tokens go in chunks
// of 128; the running softmax maximum is CTA-wide, so the four warps' value
// sums share it and add up at the end.
#pragma once

#include "common.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kPdThreads = 128;  // tokens per chunk, one per thread in the key phase

// 2^x with the hardware approximation (softmax weights only, never logits)
__device__ __forceinline__ float pd_ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
    return r;
}

// bits [off, off + n) of the little-endian words w (off, n folded at compile time)
__device__ __forceinline__ uint32_t pd_bits(const uint32_t* w, int off, int n) {
    const int W = off >> 5, S = off & 31;
    const uint32_t v = (S + n <= 32) ? (w[W] >> S) : __funnelshift_r(w[W], w[W + 1], S);
    return v & ((1u << n) - 1u);
}

template <int B1, int B2>
struct PolarRow {
    static constexpr int kBits = 64 * B1 + 63 * B2;
    static constexpr int kBytes = ((kBits + 7) / 8 + 15) / 16 * 16;
    static constexpr int kWords = kBytes / 4;
    // first stream bit of level l >= 2: the 64 level-1 angles, then 64 - 2^(8-l) angles of levels 2 .. l-1
    static constexpr int off(int l) { return 64 * B1 + B2 * (64 - (1 << (8 - l))); }
};

template <int B1, int B2, int G>
size_t polar_decode_smem() {
    return (size_t)G * 64 * (1 << B1) * sizeof(float);  // the level-1 pair tables
}

template <int B1, int B2, int G>
__global__ void __launch_bounds__(kPdThreads) polar_decode_kernel(const __grid_constant__ PolarDecodeParams p) {
    using R = PolarRow<B1, B2>;
    constexpr int L1 = 1 << B1, L2 = 1 << B2;
    extern __shared__ __align__(16) float s_lut[];                    // [G][64][L1]
    __shared__ float2 s_cs[kPolarLevels - 1][L2];                     // (cos, sin) of levels 2 .. 7
    __shared__ __align__(16) float2 s_vpair[256];                     // value codes in pairs
    __shared__ __align__(16) float s_w[kPdThreads][G];                // p_t nV_t of the chunk
    __shared__ __align__(16) uint32_t s_vc[kPdThreads * 16];          // the chunk's value codes (<= 64 B a token)
    __shared__ float s_red[4][G];
    __shared__ float s_acc[4][G][128];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;
    const int VB = p.vbits;
    const int vwords = p.vcode_stride >> 2;

    // tables that do not depend on the query (before the wait on the prep)
    for (int i = tid; i < (kPolarLevels - 1) * L2; i += kPdThreads)
        s_cs[i / L2][i % L2] = make_float2(p.ccos[i / L2][i % L2], p.csin[i / L2][i % L2]);
    for (int i = tid; i < (1 << (2 * VB)); i += kPdThreads)
        s_vpair[i] = make_float2(p.vc[i & ((1 << VB) - 1)], p.vc[i >> VB]);

    int rows[G];
#pragma unroll
    for (int g = 0; g < G; ++g) rows[g] = b * p.hq + (p.use_table ? (int)p.head_table[kv * G + g] : kv * G + g);

    // the query prep (the launch before this one) has written q'
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    for (int i = tid; i < G * 64 * L1; i += kPdThreads) {
        const int g = i / (64 * L1), pi = (i / L1) % 64, k = i % L1;
        const float* q = p.qprime + (int64_t)rows[g] * 128;
        s_lut[i] = fmaf(q[2 * pi], p.c1cos[k], q[2 * pi + 1] * p.c1sin[k]);
    }
    __syncthreads();

    const int L = p.seq_lens[b];
    const int64_t t_begin = (int64_t)split * p.chunk;
    const int64_t t_end = min((int64_t)L, t_begin + p.chunk);
    const int64_t rowbase = ((int64_t)b * p.hkv + kv) * p.capacity;

    float M[G], Z[G], acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        M[g] = -INFINITY;
        Z[g] = 0.0f;
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[g][r] = 0.0f;
    }

    for (int64_t c0 = t_begin; c0 < t_end; c0 += kPdThreads) {
        const int nt = (int)min((int64_t)kPdThreads, t_end - c0);
        // stage the chunk's value codes (contiguous rows of the cache)
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.vcodes + (rowbase + c0) * p.vcode_stride);
            uint4* dst = reinterpret_cast<uint4*>(s_vc);
            const int n16 = nt * (p.vcode_stride >> 4);
            for (int i = tid; i < n16; i += kPdThreads) dst[i] = src[i];
        }
        // ---- keys: thread = token ----
        float s[G];
        const bool valid = tid < nt;
#pragma unroll
        for (int g = 0; g < G; ++g) s[g] = -INFINITY;
        if (valid) {
            const int64_t slot = rowbase + c0 + tid;
            uint32_t kw[R::kWords];
            const uint4* kr = reinterpret_cast<const uint4*>(p.kcodes + slot * p.kcode_stride);
#pragma unroll
            for (int i = 0; i < R::kWords / 4; ++i) {
                const uint4 t = kr[i];
                kw[4 * i] = t.x;
                kw[4 * i + 1] = t.y;
                kw[4 * i + 2] = t.z;
                kw[4 * i + 3] = t.w;
            }
            float v4[8][G];
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
                float v2[4][G];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int i0 = 8 * j4 + 2 * q;
                    const uint32_t ka = pd_bits(kw, B1 * i0, B1), kb = pd_bits(kw, B1 * (i0 + 1), B1);
                    const float2 cs = s_cs[0][pd_bits(kw, R::off(2) + B2 * (4 * j4 + q), B2)];
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        v2[q][g] = fmaf(cs.x, s_lut[(g * 64 + i0) * L1 + ka], cs.y * s_lut[(g * 64 + i0 + 1) * L1 + kb]);
                }
                float v3[2][G];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float2 cs = s_cs[1][pd_bits(kw, R::off(3) + B2 * (2 * j4 + r), B2)];
#pragma unroll
                    for (int g = 0; g < G; ++g) v3[r][g] = fmaf(cs.x, v2[2 * r][g], cs.y * v2[2 * r + 1][g]);
                }
                const float2 cs = s_cs[2][pd_bits(kw, R::off(4) + B2 * j4, B2)];
#pragma unroll
                for (int g = 0; g < G; ++g) v4[j4][g] = fmaf(cs.x, v3[0][g], cs.y * v3[1][g]);
            }
#pragma unroll
            for (int j5 = 0; j5 < 4; ++j5) {
                const float2 cs = s_cs[3][pd_bits(kw, R::off(5) + B2 * j5, B2)];
#pragma unroll
                for (int g = 0; g < G; ++g) v4[j5][g] = fmaf(cs.x, v4[2 * j5][g], cs.y * v4[2 * j5 + 1][g]);
            }
#pragma unroll
            for (int j6 = 0; j6 < 2; ++j6) {
                const float2 cs = s_cs[4][pd_bits(kw, R::off(6) + B2 * j6, B2)];
#pragma unroll
                for (int g = 0; g < G; ++g) v4[j6][g] = fmaf(cs.x, v4[2 * j6][g], cs.y * v4[2 * j6 + 1][g]);
            }
            const float2 cs = s_cs[5][pd_bits(kw, R::off(7), B2)];
            const float kn = f16_bits_to_f32(p.knorm[slot]);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float l = kn * fmaf(cs.x, v4[0][g], cs.y * v4[1][g]);
                if (p.logits) p.logits[(int64_t)rows[g] * p.max_seq_len + c0 + tid] = l;
                s[g] = l * p.scale_log2;
            }
        }
        // ---- softmax: CTA-wide chunk maximum, weights, sums ----
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float m = warp_max(s[g]);
            if (lane == 0) s_red[warp][g] = m;
        }
        __syncthreads();
        float scale[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float mc = fmaxf(fmaxf(s_red[0][g], s_red[1][g]), fmaxf(s_red[2][g], s_red[3][g]));
            const float mn = fmaxf(M[g], mc);
            scale[g] = (M[g] == -INFINITY) ? 0.0f : pd_ex2(M[g] - mn);
            M[g] = mn;
        }
        __syncthreads();  // s_red reused below
        const float vn = valid ? f16_bits_to_f32(p.vnorm[rowbase + c0 + tid]) : 0.0f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float w = valid && M[g] != -INFINITY ? pd_ex2(s[g] - M[g]) : 0.0f;
            s_w[tid][g] = w * vn;
            const float z = warp_sum(w);
            if (lane == 0) s_red[warp][g] = z;
        }
        __syncthreads();
#pragma unroll
        for (int g = 0; g < G; ++g) {
            Z[g] = Z[g] * scale[g] + ((s_red[0][g] + s_red[1][g]) + (s_red[2][g] + s_red[3][g]));
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[g][r] *= scale[g];
        }
        // ---- values: warp = token, lane = 4 coordinates ----
        const int off = 4 * VB * lane, wi = off >> 5, sh = off & 31;
        const int pm = (1 << (2 * VB)) - 1;
        for (int t = warp; t < nt; t += 4) {
            const uint32_t* row = s_vc + t * vwords;
            const uint32_t hi = wi + 1 < vwords ? row[wi + 1] : 0u;
            const uint32_t bits = __funnelshift_r(row[wi], hi, sh);
            const float2 c01 = s_vpair[bits & pm];
            const float2 c23 = s_vpair[(bits >> (2 * VB)) & pm];
            float w[G];
            if constexpr (G % 4 == 0) {
#pragma unroll
                for (int g = 0; g < G; g += 4) {
                    const float4 t4 = *reinterpret_cast<const float4*>(&s_w[t][g]);
                    w[g] = t4.x;
                    w[g + 1] = t4.y;
                    w[g + 2] = t4.z;
                    w[g + 3] = t4.w;
                }
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) w[g] = s_w[t][g];
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                acc[g][0] = fmaf(w[g], c01.x, acc[g][0]);
                acc[g][1] = fmaf(w[g], c01.y, acc[g][1]);
                acc[g][2] = fmaf(w[g], c23.x, acc[g][2]);
                acc[g][3] = fmaf(w[g], c23.y, acc[g][3]);
            }
        }
        __syncthreads();  // s_w, s_vc and s_red are refilled by the next chunk
    }

    // ---- the four warps' sums (they share M) -> this split's partial ----
#pragma unroll
    for (int g = 0; g < G; ++g)
        *reinterpret_cast<float4*>(&s_acc[warp][g][4 * lane]) = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float* out = p.partial + ((int64_t)rows[g] * p.n_splits + split) * (128 + kPartPad);
        out[tid] = (s_acc[0][g][tid] + s_acc[1][g][tid]) + (s_acc[2][g][tid] + s_acc[3][g][tid]);
        if (tid == 0) {
            out[128] = M[g];
            out[129] = Z[g];
        }
    }
}

template <int B1, int B2, int G>
cudaError_t launch_polar_decode_t(const PolarDecodeParams& p, cudaStream_t s) {
    const size_t smem = polar_decode_smem<B1, B2, G>();
    auto kern = polar_decode_kernel<B1, B2, G>;
    // the static tables plus the pair tables can pass the default 48 KB
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.n_splits, (unsigned)p.hkv, (unsigned)p.batch);
    cfg.blockDim = dim3(kPdThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// every supported (bits1, bits2) for one group size
template <int G>
cudaError_t dispatch_polar_decode(const PolarDecodeParams& p, int b1, int b2, cudaStream_t s) {
    if (b1 == 2 && b2 == 2) return launch_polar_decode_t<2, 2, G>(p, s);
    if (b1 == 3 && b2 == 2) return launch_polar_decode_t<3, 2, G>(p, s);
    if (b1 == 4 && b2 == 2) return launch_polar_decode_t<4, 2, G>(p, s);
    if (b1 == 4 && b2 == 3) return launch_polar_decode_t<4, 3, G>(p, s);
    if (b1 == 3 && b2 == 3) return launch_polar_decode_t<3, 3, G>(p, s);
    if (b1 == 4 && b2 == 4) return launch_polar_decode_t<4, 4, G>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace tqk
