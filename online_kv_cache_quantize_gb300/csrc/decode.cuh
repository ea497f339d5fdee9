// Decode attention around the split-K scan: query preparation (the query is
// rotated once, q' = Pi q, and projected, u = S q') and the merge of the
// splits followed by the single un-rotation o = Pi^T (a / Z).
//
// Follows: A2A TurboQuant explainer, end of "Stage 2" and "How to implement"
// (the fused kernel rotates the query once and scores from the indices). The
// softmax merge and the un-rotation of the value sum are this library's
// reading of how the output is formed.
#pragma once

#include "common.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kPrepWarps = 8;

// The decode scan's B operands of one query row (d = m = 128), in the order
// its threads load them: word ((ks * 2 + lo) * 4 + c) * 16 + 2 * kk + r holds
// the fp16 pair (coordinates i, i + 1), i = 32c + 4kk + 2r, of the hi (lo =
// 0) or lo (lo = 1) split of q' (ks = 0) or of qjl_scale * u (ks = 1). Writes
// word `wi` (0 .. kFragWords - 1) from q' and u in shared memory; u == NULL
// gives zero words.
__device__ __forceinline__ void write_frag(const PrepParams& p, int64_t row, const float* s_q, const float* s_u,
                                           int wi) {
    if (wi >= kFragWords) return;
    const int ks = wi >> 7, lo = (wi >> 6) & 1, c = (wi >> 4) & 3, kk = (wi >> 1) & 7, r = wi & 1;
    const int i = 32 * c + 4 * kk + 2 * r;
    uint32_t w = 0u;
    if (ks == 0) {
        w = half_split(s_q[i], lo) | (half_split(s_q[i + 1], lo) << 16);
    } else if (s_u) {
        w = half_split(s_u[i] * p.qjl_scale, lo) | (half_split(s_u[i + 1] * p.qjl_scale, lo) << 16);
    }
    p.frag[row * kFragWords + wi] = w;
}

// ---------------------------------------------------------------------------
// The search's query prep (any d <= 256): one CTA (256 threads) per query
// row. Lane l of every warp owns outputs VPL*l..VPL*l+VPL-1
// and warp w accumulates the inputs j = w, w+8, ...: the rows of the
// transposed matrices are read with independent loads, all in flight at once,
// and the 8 partial vectors are summed through shared memory.
// ---------------------------------------------------------------------------
template <int VPL>
__device__ __forceinline__ void prep_row(const PrepParams& p, int64_t row) {
    constexpr int DMAX = 32 * VPL;
    __shared__ float s_x[256];
    __shared__ float s_y[256];
    __shared__ float s_part[kPrepWarps][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int d = p.d;
    for (int i = tid; i < d; i += blockDim.x) {
        s_x[i] = p.q_dtype == 1 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.q)[row * d + i])
                                : reinterpret_cast<const float*>(p.q)[row * d + i];
    }
    __syncthreads();
    if (p.rht) {
        // y = H (s * x) / sqrt(d) by butterflies, warp 0 only (d = 32 * VPL exactly)
        if (warp == 0) {
            float y[VPL];
#pragma unroll
            for (int r = 0; r < VPL; ++r) y[r] = s_x[VPL * lane + r] * p.sgn[VPL * lane + r];
#pragma unroll
            for (int h = 1; h < VPL; h <<= 1)
#pragma unroll
                for (int r = 0; r < VPL; ++r)
                    if ((r & h) == 0) {
                        float a = y[r], b = y[r + h];
                        y[r] = a + b;
                        y[r + h] = a - b;
                    }
#pragma unroll
            for (int hb = 1; hb < 32; hb <<= 1) {
                const bool upper = (lane & hb) != 0;
#pragma unroll
                for (int r = 0; r < VPL; ++r) {
                    float o = __shfl_xor_sync(TQ_FULL_MASK, y[r], hb);
                    y[r] = upper ? (o - y[r]) : (y[r] + o);
                }
            }
#pragma unroll
            for (int r = 0; r < VPL; ++r) s_y[VPL * lane + r] = y[r] * p.inv_sqrt_d;
        }
    } else {
        float acc[VPL];
#pragma unroll
        for (int r = 0; r < VPL; ++r) acc[r] = 0.0f;
#pragma unroll 32
        for (int j = warp; j < d; j += kPrepWarps) {
            const float xj = s_x[j];
            const float* rowp = p.pit32 + (size_t)j * d;
            bool vec = false;
            if constexpr (VPL == 4) {
                if (d == 128) {
                    const float4 t = __ldg(reinterpret_cast<const float4*>(rowp) + lane);
                    acc[0] = fmaf(t.x, xj, acc[0]);
                    acc[1] = fmaf(t.y, xj, acc[1]);
                    acc[2] = fmaf(t.z, xj, acc[2]);
                    acc[3] = fmaf(t.w, xj, acc[3]);
                    vec = true;
                }
            }
            if (!vec) {
#pragma unroll
                for (int r = 0; r < VPL; ++r) {
                    const int e = VPL * lane + r;
                    if (e < d) acc[r] = fmaf(__ldg(rowp + e), xj, acc[r]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < VPL; ++r)
            if (VPL * lane + r < DMAX) s_part[warp][VPL * lane + r] = acc[r];
        __syncthreads();
        for (int i = tid; i < d; i += blockDim.x) {
            float y = 0.0f;
#pragma unroll
            for (int w = 0; w < kPrepWarps; ++w) y += s_part[w][i];
            s_y[i] = y;
        }
    }
    __syncthreads();
    if (p.qprime)
        for (int i = tid; i < d; i += blockDim.x) p.qprime[row * d + i] = s_y[i];
    if (p.st32 == nullptr) return;
    // u = S q': warp w takes inputs i = w, w+8, ...; lane owns outputs MPL*lane + r
    const int m = p.m, mpl = (m + 31) >> 5;
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
#pragma unroll 32
    for (int i = warp; i < d; i += kPrepWarps) {
        const float qi = s_y[i];
        const float* rowp = p.st32 + (size_t)i * m;
        if (m == 128) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(rowp) + lane);
            acc[0] = fmaf(t.x, qi, acc[0]);
            acc[1] = fmaf(t.y, qi, acc[1]);
            acc[2] = fmaf(t.z, qi, acc[2]);
            acc[3] = fmaf(t.w, qi, acc[3]);
        } else {
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int j = mpl * lane + r;
                if (r < mpl && j < m) acc[r] = fmaf(__ldg(rowp + j), qi, acc[r]);
            }
        }
    }
    __syncthreads();  // s_part reuse
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int j = mpl * lane + r;
        if (r < mpl && j < m) s_part[warp][j] = acc[r];
    }
    __syncthreads();
    for (int j = tid; j < m; j += blockDim.x) {
        float u = 0.0f;
#pragma unroll
        for (int w = 0; w < kPrepWarps; ++w) u += s_part[w][j];
        if (p.u) p.u[row * m + j] = u;
    }
}

template <int VPL>
__global__ void __launch_bounds__(kPrepWarps * 32) query_prep_kernel(const __grid_constant__ PrepParams p) {
    prep_row<VPL>(p, blockIdx.x);
}

// ---------------------------------------------------------------------------
// Merge the splits of one query row and un-rotate: o = Pi^T (a / Z).
// CTA of 1024 threads = 1024 / (d / 4) groups of d / 4 threads, thread c4 of
// a group owning coordinates 4 c4 .. 4 c4 + 3. Group k merges the splits
// k, k + groups, ... (online max, sum and a), loading kCombinePer of them at
// once so that their loads are in flight together; then the groups are
// merged through shared memory. d in {64, 128, 256}.
// ---------------------------------------------------------------------------
constexpr int kCombineThreads = 1024;
constexpr int kCombinePer = 4;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __grid_constant__ CombineParams p) {
    __shared__ float s_m[64];
    __shared__ float s_z[64];
    __shared__ __align__(16) float s_v[kCombineThreads * 4];
    __shared__ float s_a[256];
    // launched as a programmatic dependent of the scan: wait for its grid to
    // complete and its partials to be visible (a no-op on a plain launch)
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int row = blockIdx.x, tid = threadIdx.x, d = p.d, ns = p.n_splits;
    const int tpr = d >> 2, groups = kCombineThreads / tpr;
    const int grp = tid / tpr, c4 = tid % tpr;
    const int stride = d + kPartPad;
    const float* base = p.partial + (int64_t)row * ns * stride;

    float m = -INFINITY, z = 0.0f;
    float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int s0 = grp; s0 < ns; s0 += groups * kCombinePer) {
        float4 av[kCombinePer];
        float mv[kCombinePer], zv[kCombinePer];
#pragma unroll
        for (int k = 0; k < kCombinePer; ++k) {
            const int s = s0 + k * groups;
            mv[k] = -INFINITY;
            zv[k] = 0.0f;
            av[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (s < ns) {
                const float* ps = base + (int64_t)s * stride;
                av[k] = *reinterpret_cast<const float4*>(ps + 4 * c4);
                mv[k] = ps[d];
                zv[k] = ps[d + 1];
            }
        }
#pragma unroll
        for (int k = 0; k < kCombinePer; ++k) {
            const float ms = mv[k];
            if (ms > m) {
                const float sc = (m == -INFINITY) ? 0.0f : exp2f(m - ms);
                z *= sc;
                a.x *= sc;
                a.y *= sc;
                a.z *= sc;
                a.w *= sc;
                m = ms;
            }
            if (ms != -INFINITY) {
                const float w = exp2f(ms - m);
                z = fmaf(zv[k], w, z);
                a.x = fmaf(av[k].x, w, a.x);
                a.y = fmaf(av[k].y, w, a.y);
                a.z = fmaf(av[k].z, w, a.z);
                a.w = fmaf(av[k].w, w, a.w);
            }
        }
    }
    *reinterpret_cast<float4*>(&s_v[grp * d + 4 * c4]) = a;
    if (c4 == 0) {
        s_m[grp] = m;
        s_z[grp] = z;
    }
    __syncthreads();
    if (tid < d) {
        float mstar = -INFINITY;
        for (int k = 0; k < groups; ++k) mstar = fmaxf(mstar, s_m[k]);
        float zt = 0.0f, at = 0.0f;
        for (int k = 0; k < groups; ++k) {
            const float mk = s_m[k];
            if (mk == -INFINITY) continue;
            const float w = exp2f(mk - mstar);
            zt = fmaf(s_z[k], w, zt);
            at = fmaf(s_v[k * d + tid], w, at);
        }
        s_a[tid] = (zt > 0.0f) ? at / zt : 0.0f;
    }
    __syncthreads();
    float o = 0.0f;
    if (p.rht) {
        // o = s * (H a) / sqrt(d): strides 1..16 across the lanes of a warp,
        // the rest as one (d / 32)-point transform over the first d / 32
        // warps through shared memory (s_v is free again)
        if (tid < d) {
            const int lane = tid & 31, w = tid >> 5;
            float y = s_a[tid];
#pragma unroll
            for (int h = 1; h < 32; h <<= 1) {
                const float t = __shfl_xor_sync(TQ_FULL_MASK, y, h);
                y = (lane & h) ? (t - y) : (y + t);
            }
            s_v[tid] = y;
            asm volatile("bar.sync 1, %0;\n" ::"r"(d) : "memory");  // the first d threads only
            float acc = 0.0f;
            for (int k = 0; k < (d >> 5); ++k) {
                const float t = s_v[lane + 32 * k];
                acc += (__popc(w & k) & 1) ? -t : t;
            }
            o = acc * p.sgn[tid] * p.inv_sqrt_d;
        }
    } else {
        // o_i = sum_k Pi[k][i] a_k, the k range split over 1024 / d groups of d threads
        const int ug = kCombineThreads / d, i = tid % d, ugrp = tid / d;
        const int nk = d / ug;  // rows of Pi a thread takes: 4, 16 or 64 for d = 64, 128, 256
        float part = 0.0f;
        // 16 independent loads into registers first, then the products: one
        // round of memory latency per 16 rows, not one per row
        for (int k0 = 0; k0 < nk; k0 += 16) {
            float pv[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                pv[j] = k0 + j < nk ? __ldg(p.pi32 + (size_t)(ugrp + (k0 + j) * ug) * d + i) : 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (k0 + j < nk) part = fmaf(pv[j], s_a[ugrp + (k0 + j) * ug], part);
        }
        s_v[tid] = part;
        __syncthreads();
        if (tid < d)
            for (int k = 0; k < ug; ++k) o += s_v[k * d + tid];
    }
    if (tid < d) {
        if (p.out_dtype == 1)
            reinterpret_cast<__nv_bfloat16*>(p.out)[(int64_t)row * d + tid] = __float2bfloat16_rn(o);
        else
            reinterpret_cast<float*>(p.out)[(int64_t)row * d + tid] = o;
    }
}

// ---------------------------------------------------------------------------
// Merge of a few splits per row (the chunked prefill: thousands of rows, a
// handful of splits each): one warp per row, lane l owning coordinates
// 4l .. 4l+3 (d = 128). The same arithmetic as combine_kernel: M* = max M_s,
// Z = sum Z_s 2^(M_s - M*), a = sum a_s 2^(M_s - M*) / Z, then o = Pi^T a
// (RHT: s * (H a) / sqrt(d) with H by butterflies in the thread for
// strides 1, 2 and shuffles for 4 .. 64; dense: coalesced rows of Pi).
// ---------------------------------------------------------------------------
constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeWarps * 32) merge_rows_kernel(const __grid_constant__ CombineParams p) {
    __shared__ __align__(16) float s_a[kMergeWarps][128];
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.x * kMergeWarps + warp;
    if (row >= p.rows) return;
    const int ns = p.n_splits, stride = 128 + kPartPad;
    const float* base = p.partial + (int64_t)row * ns * stride;
    float mstar = -INFINITY;
    for (int s = 0; s < ns; ++s) mstar = fmaxf(mstar, base[(int64_t)s * stride + 128]);
    float z = 0.0f;
    float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (mstar != -INFINITY) {
        for (int s = 0; s < ns; ++s) {
            const float* ps = base + (int64_t)s * stride;
            const float ms = ps[128];
            if (ms == -INFINITY) continue;
            const float w = exp2f(ms - mstar);
            const float4 av = *reinterpret_cast<const float4*>(ps + 4 * lane);
            z = fmaf(ps[129], w, z);
            a.x = fmaf(av.x, w, a.x);
            a.y = fmaf(av.y, w, a.y);
            a.z = fmaf(av.z, w, a.z);
            a.w = fmaf(av.w, w, a.w);
        }
    }
    const float inv = z > 0.0f ? 1.0f / z : 0.0f;
    float y[4] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv};
    float o[4];
    if (p.rht) {
        // strides 1 and 2 inside the thread, then 4 .. 64 across the lanes
        float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
        y[0] = t0 + t2; y[2] = t0 - t2; y[1] = t1 + t3; y[3] = t1 - t3;
#pragma unroll
        for (int h = 1; h < 32; h <<= 1)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float t = __shfl_xor_sync(TQ_FULL_MASK, y[r], h);
                y[r] = (lane & h) ? (t - y[r]) : (y[r] + t);
            }
#pragma unroll
        for (int r = 0; r < 4; ++r) o[r] = y[r] * p.sgn[4 * lane + r] * p.inv_sqrt_d;
    } else {
        *reinterpret_cast<float4*>(&s_a[warp][4 * lane]) = make_float4(y[0], y[1], y[2], y[3]);
        __syncwarp();
        o[0] = o[1] = o[2] = o[3] = 0.0f;
#pragma unroll 32
        for (int k = 0; k < 128; ++k) {
            const float ak = s_a[warp][k];
            const float4 pk = __ldg(reinterpret_cast<const float4*>(p.pi32 + (size_t)k * 128) + lane);
            o[0] = fmaf(pk.x, ak, o[0]);
            o[1] = fmaf(pk.y, ak, o[1]);
            o[2] = fmaf(pk.z, ak, o[2]);
            o[3] = fmaf(pk.w, ak, o[3]);
        }
    }
    if (p.out_dtype == 1) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (int64_t)row * 128 + 4 * lane;
        const __nv_bfloat162 lo = __floats2bfloat162_rn(o[0], o[1]), hi = __floats2bfloat162_rn(o[2], o[3]);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t*>(&lo);
        w.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out) = w;
    } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + (int64_t)row * 128 + 4 * lane) =
            make_float4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace tqk
