// Quantize-on-append kernel: norm, rotation, Lloyd-Max bucketize, bit-pack
// and (keys) the residual QJL sign sketch, one warp per vector.
//
// Follows: A2A TurboQuant explainer, "Stage 1: random rotation + PolarQuant"
// (normalise, rotate, Lloyd-Max per coordinate) and "Stage 2: QJL residual
// correction" (one sign bit per projected residual coordinate); Qiita
// TurboQuant article, "Rotate, then quantize" and "One more stage so
// attention does not break".
//
// Precision: y = Pi x / ||x|| is computed in fp32. Any coordinate whose fp32
// value lies within `guard` of a codebook boundary is recomputed in fp64
// (one warp-wide fp64 dot product) and its code decided from the fp64 value,
// so codes agree with an fp64 evaluation except in a window of a few fp64
// ulps around each boundary. The fp16 norm is likewise recomputed in fp64
// when the fp32 value sits near an fp16 rounding midpoint.
#pragma once

#include "common.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kQuantWarps = 8;

template <typename XT, int VPL, int CB, bool PROD, bool RHT>
__global__ void __launch_bounds__(kQuantWarps * 32) quantize_kernel(const __grid_constant__ QuantParams p) {
    constexpr int DMAX = 32 * VPL;
    constexpr int L = 1 << CB;
    __shared__ float s_buf[kQuantWarps][DMAX];
    __shared__ __align__(16) uint32_t s_cw[kQuantWarps][36];
    __shared__ __align__(16) uint32_t s_sw[kQuantWarps][12];
    __shared__ float s_cent[kMaxLevels];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x < kMaxLevels) s_cent[threadIdx.x] = p.cb.c[threadIdx.x];
    __syncthreads();

    const int d = p.d;
    float sg[VPL];
    if constexpr (RHT) {
#pragma unroll
        for (int r = 0; r < VPL; ++r) sg[r] = p.sgn[VPL * lane + r];
    }

    const int64_t step = (int64_t)gridDim.x * kQuantWarps;
    for (int64_t v = (int64_t)blockIdx.x * kQuantWarps + warp; v < p.n; v += step) {
        int64_t slot;
        if (p.dst_slot) {
            slot = p.dst_slot[v];
        } else if (p.append_pos) {
            int32_t pos = p.append_pos[v / p.heads];
            slot = (pos >= 0 && pos < p.capacity) ? v * p.capacity + pos : -1;
        } else {
            slot = p.slot0 + v;
        }
        if (slot < 0 || slot >= p.total_slots) continue;  // warp-uniform skip

        // ---- load x (lane owns coordinates VPL*lane .. VPL*lane+VPL-1) ----
        const XT* xr = reinterpret_cast<const XT*>(p.x) + v * p.x_stride;
        float x[VPL];
#pragma unroll
        for (int r = 0; r < VPL; ++r) {
            int e = VPL * lane + r;
            x[r] = (e < d) ? to_f32(xr[e]) : 0.0f;
        }

        // ---- norm ----
        float ss = 0.0f;
#pragma unroll
        for (int r = 0; r < VPL; ++r) ss = fmaf(x[r], x[r], ss);
        ss = warp_sum(ss);
        float n32 = sqrtf(ss);
        if (!(ss > 1.0e-30f && ss < 1.0e30f)) {
            // squares may have under/overflowed: rescale by the largest |x_i|
            float amax = 0.0f;
#pragma unroll
            for (int r = 0; r < VPL; ++r) amax = fmaxf(amax, fabsf(x[r]));
            amax = warp_max(amax);
            float s2 = 0.0f;
            if (amax > 0.0f) {
                const float ia = 1.0f / amax;
#pragma unroll
                for (int r = 0; r < VPL; ++r) s2 = fmaf(x[r] * ia, x[r] * ia, s2);
            }
            s2 = warp_sum(s2);
            n32 = amax * sqrtf(s2);
        }
        const float inv_n = n32 > 0.0f ? 1.0f / n32 : 0.0f;

        // ---- rotation: y = Pi x / n ----
        float y[VPL];
        if constexpr (RHT) {
#pragma unroll
            for (int r = 0; r < VPL; ++r) y[r] = x[r] * sg[r];
            // in-register butterflies (strides 1 .. VPL/2)
#pragma unroll
            for (int h = 1; h < VPL; h <<= 1) {
#pragma unroll
                for (int r = 0; r < VPL; ++r) {
                    if ((r & h) == 0) {
                        float a = y[r], b = y[r + h];
                        y[r] = a + b;
                        y[r + h] = a - b;
                    }
                }
            }
            // cross-lane butterflies (strides VPL .. 16*VPL)
#pragma unroll
            for (int hb = 1; hb < 32; hb <<= 1) {
                const bool upper = (lane & hb) != 0;
#pragma unroll
                for (int r = 0; r < VPL; ++r) {
                    float o = __shfl_xor_sync(TQ_FULL_MASK, y[r], hb);
                    y[r] = upper ? (o - y[r]) : (y[r] + o);
                }
            }
            const float sc = p.inv_sqrt_d * inv_n;
#pragma unroll
            for (int r = 0; r < VPL; ++r) y[r] *= sc;
        } else {
#pragma unroll
            for (int r = 0; r < VPL; ++r) {
                int e = VPL * lane + r;
                if (e < d) s_buf[warp][e] = x[r];
            }
            __syncwarp();
            float acc[VPL];
#pragma unroll
            for (int r = 0; r < VPL; ++r) acc[r] = 0.0f;
            for (int j = 0; j < d; ++j) {
                const float xj = s_buf[warp][j];
                const float* row = p.pit32 + (size_t)j * d;
#pragma unroll
                for (int r = 0; r < VPL; ++r) {
                    int e = VPL * lane + r;
                    if (e < d) acc[r] = fmaf(__ldg(row + e), xj, acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < VPL; ++r) y[r] = acc[r] * inv_n;
            __syncwarp();
        }

        // ---- bucketize with guard band ----
        int idx[VPL];
        uint32_t flags = 0;
#pragma unroll
        for (int r = 0; r < VPL; ++r) {
            int k = 0;
            float dmin = 3.0e38f;
#pragma unroll
            for (int j = 0; j < L - 1; ++j) {
                k += (y[r] >= p.cb.t[j]) ? 1 : 0;
                dmin = fminf(dmin, fabsf(y[r] - p.cb.t[j]));
            }
            idx[r] = k;
            int e = VPL * lane + r;
            if (e < d && !(dmin >= p.guard)) flags |= 1u << r;
        }

        // fp16 norm: near a rounding midpoint, decide from the fp64 norm
        uint16_t n16 = f16_bits_sat(n32);
        bool norm_close = false;
        if (n32 > 0.0f && n32 < 65504.0f) {
            float dn = __half2float(__float2half_rd(n32));
            float up = __half2float(__float2half_ru(n32));
            float mid = 0.5f * (dn + up);
            norm_close = dn != up && fabsf(n32 - mid) <= 1.0e-6f * n32;
        }

        if (__any_sync(TQ_FULL_MASK, flags != 0 || norm_close)) {
            double ss64 = 0.0;
#pragma unroll
            for (int r = 0; r < VPL; ++r) ss64 = fma((double)x[r], (double)x[r], ss64);
            ss64 = warp_sum(ss64);
            const double n64 = sqrt(ss64);
            if (norm_close) n16 = __half_as_ushort(__double2half(fmin(n64, 65504.0)));
            while (true) {
                unsigned bal = __ballot_sync(TQ_FULL_MASK, flags != 0);
                if (!bal) break;
                const int src = __ffs(bal) - 1;
                const int rsrc = __shfl_sync(TQ_FULL_MASK, __ffs(flags) - 1, src);
                const int i = VPL * src + rsrc;
                double part = 0.0;
                if constexpr (RHT) {
#pragma unroll
                    for (int r = 0; r < VPL; ++r) {
                        int e = VPL * lane + r;
                        double t = (double)sg[r] * (double)x[r];
                        part += (__popc(i & e) & 1) ? -t : t;
                    }
                } else {
                    const double* row = p.pi64 + (size_t)i * d;
#pragma unroll
                    for (int r = 0; r < VPL; ++r) {
                        int e = VPL * lane + r;
                        if (e < d) part = fma(row[e], (double)x[r], part);
                    }
                }
                part = warp_sum(part);
                double y64 = 0.0;
                if (n64 > 0.0) y64 = RHT ? part / (sqrt((double)d) * n64) : part / n64;
                if (lane == src) {
#pragma unroll
                    for (int r = 0; r < VPL; ++r) {
                        if (r == rsrc) {
                            int k = 0;
#pragma unroll
                            for (int j = 0; j < L - 1; ++j) k += (y64 >= p.cb.t64[j]) ? 1 : 0;
                            idx[r] = k;
                            y[r] = (float)y64;
                        }
                    }
                    flags &= ~(1u << rsrc);
                }
            }
        }

        // ---- zero the per-warp word buffers ----
        const int cwords = p.code_stride >> 2;
        for (int w = lane; w < cwords; w += 32) s_cw[warp][w] = 0u;
        if constexpr (PROD) {
            const int swords = p.sign_stride >> 2;
            for (int w = lane; w < swords; w += 32) s_sw[warp][w] = 0u;
        }
        __syncwarp();

        // ---- pack codes: lane's CB*VPL bits at stream offset CB*VPL*lane ----
        if (VPL * lane < d) {
            uint32_t chunk = 0;
#pragma unroll
            for (int r = 0; r < VPL; ++r)
                if (VPL * lane + r < d) chunk |= (uint32_t)idx[r] << (CB * r);
            const int off = CB * VPL * lane;
            const int w = off >> 5, sh = off & 31;
            atomicOr(&s_cw[warp][w], chunk << sh);
            if (sh + CB * VPL > 32) atomicOr(&s_cw[warp][w + 1], chunk >> (32 - sh));
        }

        float gamma = 0.0f;
        if constexpr (PROD) {
            // residual r = y - c[idx], gamma = ||r||, z_j = [(S r)_j >= 0]
            float g2 = 0.0f;
#pragma unroll
            for (int r = 0; r < VPL; ++r) {
                int e = VPL * lane + r;
                float rr = (e < d) ? y[r] - s_cent[idx[r]] : 0.0f;
                g2 = fmaf(rr, rr, g2);
                if (e < d) s_buf[warp][e] = rr;
            }
            g2 = warp_sum(g2);
            gamma = sqrtf(g2);
            __syncwarp();
            const int m = p.m;
            const int mpl = (m + 31) >> 5;
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
            for (int i = 0; i < d; ++i) {
                const float ri = s_buf[warp][i];
                const float* row = p.st32 + (size_t)i * m;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    int j = mpl * lane + r;
                    if (r < mpl && j < m) acc[r] = fmaf(__ldg(row + j), ri, acc[r]);
                }
            }
            uint32_t sbits = 0;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                int j = mpl * lane + r;
                if (r < mpl && j < m && acc[r] >= 0.0f) sbits |= 1u << r;
            }
            if (mpl * lane < m) {
                const int off = mpl * lane;
                const int w = off >> 5, sh = off & 31;
                atomicOr(&s_sw[warp][w], sbits << sh);
                if (sh + mpl > 32) atomicOr(&s_sw[warp][w + 1], sbits >> (32 - sh));
            }
        }
        __syncwarp();

        // ---- stores ----
        {
            uint4* dst = reinterpret_cast<uint4*>(p.codes + slot * (int64_t)p.code_stride);
            const uint4* src = reinterpret_cast<const uint4*>(&s_cw[warp][0]);
            for (int q = lane; q < (p.code_stride >> 4); q += 32) dst[q] = src[q];
        }
        if constexpr (PROD) {
            uint4* dst = reinterpret_cast<uint4*>(p.signs + slot * (int64_t)p.sign_stride);
            const uint4* src = reinterpret_cast<const uint4*>(&s_sw[warp][0]);
            for (int q = lane; q < (p.sign_stride >> 4); q += 32) dst[q] = src[q];
        }
        if (lane == 0) {
            p.norm[slot] = n16;
            if constexpr (PROD) p.rnorm[slot] = f16_bits_sat(gamma);
        }
        __syncwarp();
    }
}

template <typename XT, int VPL, bool RHT>
cudaError_t launch_quantize_t(const QuantParams& p, int prod, int cb, cudaStream_t s) {
    if (p.n <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (p.n + kQuantWarps - 1) / kQuantWarps;
    int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    dim3 grid((unsigned)blocks), block(kQuantWarps * 32);
#define TQ_QLAUNCH(CBV, PRODV) \
    quantize_kernel<XT, VPL, CBV, PRODV, RHT><<<grid, block, 0, s>>>(p)
    switch (cb * 2 + prod) {
        case 2: TQ_QLAUNCH(1, false); break;
        case 3: TQ_QLAUNCH(1, true); break;
        case 4: TQ_QLAUNCH(2, false); break;
        case 5: TQ_QLAUNCH(2, true); break;
        case 6: TQ_QLAUNCH(3, false); break;
        case 7: TQ_QLAUNCH(3, true); break;
        case 8: TQ_QLAUNCH(4, false); break;
        case 9: TQ_QLAUNCH(4, true); break;
        default: return cudaErrorInvalidValue;
    }
#undef TQ_QLAUNCH
    return cudaGetLastError();
}

}  // namespace tqk
