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
// product is rho sin(psi - t)): level 1 takes the half plane from the sign of
// the second component, then locates psi inside it; the other levels count
// their boundaries from the squared radii (no square roots). A cross product
// within `guard` of zero (or a pair next to the cut at +-pi) sends the whole
// vector to an fp64 recomputation (rotation, the same cross products against
// the fp64 boundaries' cosines and sines, radii by fp64 square roots), so
// every code is the one an fp64 evaluation gives.
#include "common.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kPqWarps = 8;

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

// psi >= t_j for the pair (a, b) and the boundary t_j = (tc, ts), when
// |psi - t_j| < pi: the sign of the cross product rho sin(psi - t_j)
template <typename F>
__device__ __forceinline__ F cross(F a, F b, F tc, F ts) { return fma(b, tc, -a * ts); }

// The level-1 code of (a, b) (cells of 2 pi / L1 from -pi; boundary j at
// index j - 1 of tc / ts): the half plane from the sign of b (boundary
// L1 / 2 is 0, the cut is +-pi), then bisection by cross products inside it,
// whose boundaries all lie within pi of psi. Flags the pair when b or either
// edge of the chosen cell is within g of zero.
__device__ __forceinline__ float xcross(float a, float b, float2 t) { return fmaf(b, t.x, -a * t.y); }

// t[j - 1] = (cos t_j, sin t_j). With L1 a compile-time constant (the
// default widths) the bisection unrolls completely.
__device__ __forceinline__ int level1_code(float a, float b, int L1, const float2* t, float g, bool& flag) {
    int lo = b >= 0.0f ? L1 / 2 : 0;
#pragma unroll
    for (int step = L1 / 4; step >= 1; step >>= 1) {
        const int j = lo + step;
        if (xcross(a, b, t[j - 1]) >= 0.0f) lo = j;
    }
    flag |= !(fabsf(b) >= g);
    if (lo >= 1) flag |= !(xcross(a, b, t[lo - 1]) >= g);
    if (lo + 1 <= L1 - 1) flag |= !(xcross(a, b, t[lo]) <= -g);
    return lo;
}

// Branch-free level 1 for a compile-time width: the lower half plane is the
// upper one turned by pi (t_j - pi = t_(j + L1/2) and (a, b) -> (-a, -b)
// negates every cross product), so after the turn the code is L1/2 (upper
// half) or 0 plus the count of the upper half's L1/2 - 1 boundaries below psi
// (t = the table from boundary L1/2 + 1 on). Every cross product takes part
// in the guard (a far boundary is only close to zero when the radius is).
template <int L1>
__device__ __forceinline__ int level1_code_lin(float a, float b, const float2* t, float g, bool& flag) {
    const bool up = b >= 0.0f;
    const float aa = up ? a : -a, bb = up ? b : -b;
    int k = up ? L1 / 2 : 0;
    float m = fabsf(b);
#pragma unroll
    for (int j = 0; j < L1 / 2 - 1; ++j) {
        const float c = xcross(aa, bb, t[j]);
        k += c >= 0.0f ? 1 : 0;
        m = fminf(m, fabsf(c));
    }
    flag |= !(m >= g);
    return k;
}

// A level >= 2 angle from the squared radii A = a^2, B = b^2 (no square
// root anywhere in the tree): for a, b >= 0 and t in (0, pi/2) the cross
// product b cos t - a sin t has the sign of B cos^2 t - A sin^2 t, which is
// (b cos t - a sin t)(b cos t + a sin t) with a second factor of at most
// sqrt(A + B). So |b cos t - a sin t| < g implies (B cos^2 t - A sin^2 t)^2 <
// g^2 (A + B): flagging on the latter (or on equality, which also catches an
// all-zero block) flags every decision the fp32 values cannot make.
// t2[j] = (cos^2 t_(j+1), sin^2 t_(j+1)); L = 0: the width from Lr.
template <int L>
__device__ __forceinline__ int upper_code_sq(float A, float B, int Lr, const float2* t2, float g2, bool& flag) {
    const int n = (L > 0 ? L : Lr) - 1;
    const float thr = g2 * (A + B);
    int k = 0;
    bool f = false;
#pragma unroll
    for (int j = 0; j < (L > 0 ? L - 1 : 15); ++j) {
        if (L == 0 && j >= n) break;
        const float c = fmaf(B, t2[j].x, -A * t2[j].y);
        k += c >= 0.0f ? 1 : 0;
        f |= !(c * c > thr);
    }
    flag |= f;
    return k;
}

// The same decisions in fp64, with atan2's answers where a component is
// zero: psi = atan2(b, a) lies in the lower half exactly when b < 0 or b is
// -0 with a < 0 or a = -0 (psi = -pi); the origin's angle is +-0 (code
// L1 / 2) or +-pi (code L1 - 1 or 0).
__device__ __forceinline__ int level1_code64(double a, double b, int L1, const double* tc, const double* ts) {
    const bool down = b < 0.0 || (b == 0.0 && signbit(b) && signbit(a));
    if (a == 0.0 && b == 0.0) return down ? 0 : (signbit(a) ? L1 - 1 : L1 / 2);
    int lo = down ? 0 : L1 / 2;
    for (int step = L1 / 4; step >= 1; step >>= 1) {
        const int j = lo + step;
        if (cross(a, b, tc[j - 1], ts[j - 1]) >= 0.0) lo = j;
    }
    return lo;
}

__device__ __forceinline__ int upper_code64(double a, double b, int L, const double* tc, const double* ts) {
    if (a == 0.0 && b == 0.0) return 0;  // atan2(0, 0) = 0: below every boundary
    int lo = 0;
    for (int step = L / 2; step >= 1; step >>= 1) {
        const int j = lo + step;
        if (cross(a, b, tc[j - 1], ts[j - 1]) >= 0.0) lo = j;
    }
    return lo;
}

// B1T, B2T: compile-time code widths (the default 4 / 2), or 0 to take them
// from the parameters
template <typename XT, bool RHT, int B1T, int B2T>
__global__ void __launch_bounds__(kPqWarps * 32) polar_quantize_kernel(const __grid_constant__ PolarQuantParams P) {
    const QuantParams& p = P.q;
    __shared__ __align__(16) uint32_t s_w[kPqWarps][16];
    __shared__ float s_x[kPqWarps][128];
    __shared__ float2 s_t[16];                    // level 1: (cos t_j, sin t_j)
    __shared__ float2 s_t2[kPolarLevels][16];     // levels >= 2: (cos^2 t_j, sin^2 t_j)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kPolarLevels * 15; i += blockDim.x) {
        const int lv = i / 15, j = i % 15;
        if (lv == 0) s_t[j] = make_float2(P.cb.tc[0][j], P.cb.ts[0][j]);
        else s_t2[lv][j] = make_float2((float)(P.cb.tc64[lv][j] * P.cb.tc64[lv][j]),
                                       (float)(P.cb.ts64[lv][j] * P.cb.ts64[lv][j]));
    }
    __syncthreads();
    const int B1 = B1T > 0 ? B1T : P.bits1, B2 = B2T > 0 ? B2T : P.bits2;
    const int L1 = 1 << B1, L2 = 1 << B2;
    const float g = P.guard, g2 = g * g;
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
        float R[2];  // squared level-1 radii
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float a = y[2 * q], b = y[2 * q + 1];
            if constexpr (B1T > 0)
                c1[q] = level1_code_lin<(1 << B1T)>(a, b, &s_t[(1 << B1T) / 2], g, flag);
            else
                c1[q] = level1_code(a, b, L1, s_t, g, flag);
            R[q] = fmaf(a, a, b * b);
        }
        int cl[kPolarLevels];  // codes of levels 2 .. 7 at index 1 .. 6
        // level 2: node `lane` from the lane's two level-1 radii
        cl[1] = upper_code_sq<(B2T > 0 ? (1 << B2T) : 0)>(R[0], R[1], L2, s_t2[1], g2, flag);
        float r_cur = R[0] + R[1];  // squared radius of the lane's level-2 node
#pragma unroll
        for (int lev = 3; lev <= kPolarLevels; ++lev) {
            const int sh = lev - 3;
            const float o = __shfl_xor_sync(TQ_FULL_MASK, r_cur, 1 << sh);
            const bool left = ((lane >> sh) & 1) == 0;
            const float a = left ? r_cur : o, b = left ? o : r_cur;
            cl[lev - 1] = upper_code_sq<(B2T > 0 ? (1 << B2T) : 0)>(a, b, L2, s_t2[lev - 1], g2, flag);
            r_cur = a + b;
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
                    c1[q] = level1_code64(a, b, L1, P.cb.tc64[0], P.cb.ts64[0]);
                    rr[q] = sqrt(fma(a, a, b * b));
                }
                cl[1] = upper_code64(rr[0], rr[1], L2, P.cb.tc64[1], P.cb.ts64[1]);
                double r64 = sqrt(fma(rr[0], rr[0], rr[1] * rr[1]));
#pragma unroll
                for (int lev = 3; lev <= kPolarLevels; ++lev) {
                    const int sh = lev - 3;
                    const double o = __shfl_xor_sync(TQ_FULL_MASK, r64, 1 << sh);
                    const bool left = ((lane >> sh) & 1) == 0;
                    const double a = left ? r64 : o, b = left ? o : r64;
                    cl[lev - 1] = upper_code64(a, b, L2, P.cb.tc64[lev - 1], P.cb.ts64[lev - 1]);
                    r64 = sqrt(fma(a, a, b * b));
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
    const bool fast = p.bits1 == 4 && p.bits2 == 2;  // the default widths: compile-time
#define TQ_PQ(XT, R)                                                              \
    if (fast) polar_quantize_kernel<XT, R, 4, 2><<<grid, block, 0, s>>>(p);       \
    else polar_quantize_kernel<XT, R, 0, 0><<<grid, block, 0, s>>>(p);
    if (dtype == 1) {
        if (rht) { TQ_PQ(__nv_bfloat16, true) } else { TQ_PQ(__nv_bfloat16, false) }
    } else {
        if (rht) { TQ_PQ(float, true) } else { TQ_PQ(float, false) }
    }
#undef TQ_PQ
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
