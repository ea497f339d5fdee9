// PolarQuant key quantization (the comparison variant), d = 128, one warp per
// vector.
//
// Follows the DeepSignal TurboQuant article ("PolarQuant": the vector taken
// from Cartesian to polar coordinates pair by pair, recursively; angles kept
// at more bits than the radius) and the A2A TurboQuant explainer ("Stage 1":
// normalise, rotate, recursive pairing, a Lloyd-Max quantizer of each
// angle's known law, no per-block normalisation constants):
//   n = ||x||, y = Pi x / n;
//   level 1: psi_1,i = atan2(y_2i+1, y_2i) in (-pi, pi], rho_1,i = hypot;
//   level l >= 2: the same on the radii of level l - 1 (psi in [0, pi/2]);
//   code of an angle = #{j : t_j <= psi} in its level's codebook.
//
// Lane l owns coordinates 4l .. 4l+3: its two level-1 pairs, the level-2
// node l, and (level l >= 3) node lane >> (l - 2) with the partner radius
// from a shuffle. Decisions in fp32 without the angle: for a boundary t of
// the pair (a, b), psi >= t exactly when b cos t - a sin t >= 0 (the cross
// product is rho sin(psi - t)); level 1 first places psi by atan2f on the
// uniform grid, then checks the two boundaries around it. A cross product
// within `guard` of zero (or a pair next to the cut at +-pi) sends the whole
// vector to an fp64 recomputation (rotation, atan2, hypot, comparisons with
// the fp64 boundaries), so every code is the one an fp64 evaluation gives.
#include "common.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kPqWarps = 8;
constexpr float kPi = 3.14159265358979323846f;

// fp64 butterflies of y (4 coordinates per lane): strides 1, 2 in the lane,
// 4 .. 64 across lanes
__device__ __forceinline__ void fwht128_f64(double (&y)[4], int lane) {
    double t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
    y[0] = t0 + t2;
    y[2] = t0 - t2;
    y[1] = t1 + t3;
    y[3] = t1 - t3;
#pragma unroll
    for (int hb = 1; hb < 32; hb <<= 1) {
        const bool upper = (lane & hb) != 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const double o = __shfl_xor_sync(TQ_FULL_MASK, y[r], hb);
            y[r] = upper ? (o - y[r]) : (y[r] + o);
        }
    }
}

template <typename XT, bool RHT>
__global__ void __launch_bounds__(kPqWarps * 32) polar_quantize_kernel(const __grid_constant__ PolarQuantParams P) {
    const QuantParams& p = P.q;
    __shared__ __align__(16) uint32_t s_w[kPqWarps][16];
    __shared__ float s_x[kPqWarps][128];
    __shared__ float s_tc[kPolarLevels][16], s_ts[kPolarLevels][16];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kPolarLevels * 15; i += blockDim.x) {
        s_tc[i / 15][i % 15] = P.cb.tc[i / 15][i % 15];
        s_ts[i / 15][i % 15] = P.cb.ts[i / 15][i % 15];
    }
    __syncthreads();
    const int B1 = P.bits1, B2 = P.bits2;
    const int L1 = 1 << B1, NB2 = (1 << B2) - 1;
    const float g = P.guard;
    float sg[4];
    if constexpr (RHT) {
#pragma unroll
        for (int r = 0; r < 4; ++r) sg[r] = p.sgn[4 * lane + r];
    }
    const int nwords = p.code_stride >> 2;

    const int64_t step = (int64_t)gridDim.x * kPqWarps;
    for (int64_t v = (int64_t)blockIdx.x * kPqWarps + warp; v < p.n; v += step) {
        int64_t slot;
        if (p.dst_slot) {
            slot = p.dst_slot[v];
        } else if (p.append_pos) {
            const int32_t pos = p.append_pos[v / p.heads];
            slot = (pos >= 0 && pos < p.capacity) ? v * p.capacity + pos : -1;
        } else {
            slot = p.slot0 + v;
        }
        if (slot < 0 || slot >= p.total_slots) continue;  // warp-uniform skip

        const XT* xr = reinterpret_cast<const XT*>(p.x) + v * p.x_stride;
        float x[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) x[r] = to_f32(xr[4 * lane + r]);

        // ---- norm (fp32; squares that under/overflow are rescaled) ----
        float ss = 0.0f;
#pragma unroll
        for (int r = 0; r < 4; ++r) ss = fmaf(x[r], x[r], ss);
        ss = warp_sum(ss);
        float n32 = sqrtf(ss);
        if (!(ss > 1.0e-30f && ss < 1.0e30f)) {
            float amax = 0.0f;
#pragma unroll
            for (int r = 0; r < 4; ++r) amax = fmaxf(amax, fabsf(x[r]));
            amax = warp_max(amax);
            float s2 = 0.0f;
            if (amax > 0.0f) {
                const float ia = 1.0f / amax;
#pragma unroll
                for (int r = 0; r < 4; ++r) s2 = fmaf(x[r] * ia, x[r] * ia, s2);
            }
            n32 = amax * sqrtf(warp_sum(s2));
        }
        const float inv_n = n32 > 0.0f ? 1.0f / n32 : 0.0f;

        // ---- rotation: y = Pi x / n (fp32) ----
        float y[4];
        if constexpr (RHT) {
#pragma unroll
            for (int r = 0; r < 4; ++r) y[r] = x[r] * sg[r];
            float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
            y[0] = t0 + t2;
            y[2] = t0 - t2;
            y[1] = t1 + t3;
            y[3] = t1 - t3;
#pragma unroll
            for (int hb = 1; hb < 32; hb <<= 1) {
                const bool upper = (lane & hb) != 0;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float o = __shfl_xor_sync(TQ_FULL_MASK, y[r], hb);
                    y[r] = upper ? (o - y[r]) : (y[r] + o);
                }
            }
            const float sc = p.inv_sqrt_d * inv_n;
#pragma unroll
            for (int r = 0; r < 4; ++r) y[r] *= sc;
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r) s_x[warp][4 * lane + r] = x[r];
            __syncwarp();
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 8
            for (int j = 0; j < 128; ++j) {
                const float xj = s_x[warp][j];
                const float4 pt = __ldg(reinterpret_cast<const float4*>(p.pit32 + (size_t)j * 128) + lane);
                acc[0] = fmaf(pt.x, xj, acc[0]);
                acc[1] = fmaf(pt.y, xj, acc[1]);
                acc[2] = fmaf(pt.z, xj, acc[2]);
                acc[3] = fmaf(pt.w, xj, acc[3]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) y[r] = acc[r] * inv_n;
            __syncwarp();
        }

        // ---- the polar recursion in fp32 with guarded decisions ----
        bool flag = false;
        int c1[2];
        float rho[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float a = y[2 * q], b = y[2 * q + 1];
            const float psi = atan2f(b, a);
            int k = (int)floorf((psi + kPi) * P.inv_w1);
            k = k < 0 ? 0 : (k > L1 - 1 ? L1 - 1 : k);
            if (k >= 1) {  // psi >= t_k (boundary k - 1 of the list)
                const float sl = fmaf(b, s_tc[0][k - 1], -a * s_ts[0][k - 1]);
                flag |= !(sl >= g);
            }
            if (k <= L1 - 2) {  // psi < t_(k+1)
                const float sh = fmaf(b, s_tc[0][k], -a * s_ts[0][k]);
                flag |= !(sh <= -g);
            }
            flag |= a < g && fabsf(b) < g;  // next to the cut at +-pi (or the origin)
            c1[q] = k;
            rho[q] = hypotf(a, b);
        }
        // level 2: node `lane` from the lane's two level-1 radii
        int cl[kPolarLevels];  // codes of levels 2 .. 7 at index 1 .. 6
        float r_cur;
        {
            const float a = rho[0], b = rho[1];
            int k = 0;
            for (int j = 0; j < NB2; ++j) {
                const float sj = fmaf(b, s_tc[1][j], -a * s_ts[1][j]);
                k += sj >= 0.0f ? 1 : 0;
                flag |= !(fabsf(sj) >= g);
            }
            cl[1] = k;
            r_cur = hypotf(a, b);
        }
#pragma unroll
        for (int lev = 3; lev <= kPolarLevels; ++lev) {
            const int sh = lev - 3;
            const float o = __shfl_xor_sync(TQ_FULL_MASK, r_cur, 1 << sh);
            const bool left = ((lane >> sh) & 1) == 0;
            const float a = left ? r_cur : o, b = left ? o : r_cur;
            int k = 0;
            for (int j = 0; j < NB2; ++j) {
                const float sj = fmaf(b, s_tc[lev - 1][j], -a * s_ts[lev - 1][j]);
                k += sj >= 0.0f ? 1 : 0;
                flag |= !(fabsf(sj) >= g);
            }
            cl[lev - 1] = k;
            r_cur = hypotf(a, b);
        }

        // fp16 norm: near a rounding midpoint, decide from the fp64 norm
        uint16_t n16 = f16_bits_sat(n32);
        bool norm_close = false;
        if (n32 > 0.0f && n32 < 65504.0f) {
            const float dn = __half2float(__float2half_rd(n32));
            const float up = __half2float(__float2half_ru(n32));
            norm_close = dn != up && fabsf(n32 - 0.5f * (dn + up)) <= 1.0e-6f * n32;
        }

        // ---- rare: the whole vector in fp64 ----
        if (__any_sync(TQ_FULL_MASK, flag || norm_close)) {
            double ss64 = 0.0;
#pragma unroll
            for (int r = 0; r < 4; ++r) ss64 = fma((double)x[r], (double)x[r], ss64);
            const double n64 = sqrt(warp_sum(ss64));
            if (norm_close) n16 = __half_as_ushort(__double2half(fmin(n64, 65504.0)));
            if (__any_sync(TQ_FULL_MASK, flag)) {
                double y64[4];
                if constexpr (RHT) {
#pragma unroll
                    for (int r = 0; r < 4; ++r) y64[r] = (double)(x[r] * sg[r]);  // +-x: exact
                    fwht128_f64(y64, lane);
#pragma unroll
                    for (int r = 0; r < 4; ++r) y64[r] = n64 > 0.0 ? y64[r] / (sqrt(128.0) * n64) : 0.0;
                } else {
                    // s_x still holds x (the dense path staged it)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const double* row = p.pi64 + (size_t)(4 * lane + r) * 128;
                        double acc = 0.0;
                        for (int j = 0; j < 128; ++j) acc = fma(row[j], (double)s_x[warp][j], acc);
                        y64[r] = n64 > 0.0 ? acc / n64 : 0.0;
                    }
                }
                double rr[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const double a = y64[2 * q], b = y64[2 * q + 1];
                    const double psi = atan2(b, a);
                    int k = 0;
                    for (int j = 0; j < L1 - 1; ++j) k += P.cb.t64[0][j] <= psi ? 1 : 0;
                    c1[q] = k;
                    rr[q] = hypot(a, b);
                }
                double r64;
                {
                    const double psi = atan2(rr[1], rr[0]);
                    int k = 0;
                    for (int j = 0; j < NB2; ++j) k += P.cb.t64[1][j] <= psi ? 1 : 0;
                    cl[1] = k;
                    r64 = hypot(rr[0], rr[1]);
                }
#pragma unroll
                for (int lev = 3; lev <= kPolarLevels; ++lev) {
                    const int sh = lev - 3;
                    const double o = __shfl_xor_sync(TQ_FULL_MASK, r64, 1 << sh);
                    const bool left = ((lane >> sh) & 1) == 0;
                    const double a = left ? r64 : o, b = left ? o : r64;
                    const double psi = atan2(b, a);
                    int k = 0;
                    for (int j = 0; j < NB2; ++j) k += P.cb.t64[lev - 1][j] <= psi ? 1 : 0;
                    cl[lev - 1] = k;
                    r64 = hypot(a, b);
                }
            }
        }
        if constexpr (!RHT) __syncwarp();  // s_x reads done before the next vector stages

        // ---- pack: one LSB-first stream, level 1 first ----
        for (int w = lane; w < nwords; w += 32) s_w[warp][w] = 0u;
        __syncwarp();
        auto put = [&](int off, uint32_t code, int width) {
            const int w = off >> 5, sh = off & 31;
            atomicOr(&s_w[warp][w], code << sh);
            if (sh + width > 32) atomicOr(&s_w[warp][w + 1], code >> (32 - sh));
        };
        put(B1 * 2 * lane, (uint32_t)c1[0] | ((uint32_t)c1[1] << B1), 2 * B1);
        put(64 * B1 + B2 * lane, (uint32_t)cl[1], B2);
#pragma unroll
        for (int lev = 3; lev <= kPolarLevels; ++lev) {
            // level lev: node j = lane >> (lev - 2), held by the lanes with
            // lane % 2^(lev-2) == 0; the levels before it hold 64 - 2^(8-lev) angles
            if ((lane & ((1 << (lev - 2)) - 1)) == 0)
                put(64 * B1 + B2 * (64 - (1 << (8 - lev)) + (lane >> (lev - 2))), (uint32_t)cl[lev - 1], B2);
        }
        __syncwarp();
        {
            uint4* dst = reinterpret_cast<uint4*>(p.codes + slot * (int64_t)p.code_stride);
            const uint4* src = reinterpret_cast<const uint4*>(&s_w[warp][0]);
            for (int q = lane; q < (p.code_stride >> 4); q += 32) dst[q] = src[q];
        }
        if (lane == 0) p.norm[slot] = n16;
        __syncwarp();
    }
}

cudaError_t launch_polar_quantize(const PolarQuantParams& p, int dtype, int rht, cudaStream_t s) {
    if (p.q.n <= 0) return cudaSuccess;
    if (p.q.d != 128 || p.q.code_stride > 64 || (p.q.code_stride & 15)) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (p.q.n + kPqWarps - 1) / kPqWarps;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    const dim3 grid((unsigned)blocks), block(kPqWarps * 32);
    if (dtype == 1) {
        if (rht) polar_quantize_kernel<__nv_bfloat16, true><<<grid, block, 0, s>>>(p);
        else polar_quantize_kernel<__nv_bfloat16, false><<<grid, block, 0, s>>>(p);
    } else {
        if (rht) polar_quantize_kernel<float, true><<<grid, block, 0, s>>>(p);
        else polar_quantize_kernel<float, false><<<grid, block, 0, s>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_polar_decode_g12(const PolarDecodeParams& p, int b1, int b2, cudaStream_t s);
cudaError_t launch_polar_decode_g48(const PolarDecodeParams& p, int b1, int b2, cudaStream_t s);

bool polar_decode_supported(int b1, int b2) {
    return (b2 == 2 && b1 >= 2 && b1 <= 4) || (b1 == 4 && b2 == 3) || (b1 == 3 && b2 == 3) || (b1 == 4 && b2 == 4);
}

cudaError_t launch_polar_decode(const PolarDecodeParams& p, int b1, int b2, cudaStream_t s) {
    if (!polar_decode_supported(b1, b2)) return cudaErrorInvalidValue;
    return p.group <= 2 ? launch_polar_decode_g12(p, b1, b2, s) : launch_polar_decode_g48(p, b1, b2, s);
}

}  // namespace tqk
