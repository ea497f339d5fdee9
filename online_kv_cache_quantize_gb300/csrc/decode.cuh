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
#include "pipeline.cuh"
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
// once so that their loads are in flight together. The groups are then
// merged in parallel, not one after another: one warp reduction gives M* and
// the groups' weights 2^(m_k - M*), and the 1024 threads sum the weighted
// group vectors as 1024 / d parts per coordinate. The RHT signs the
// un-rotation needs are loaded before the wait for the scan. d in {64, 128,
// 256}.
// ---------------------------------------------------------------------------
constexpr int kCombineThreads = 1024;
constexpr int kCombinePer = 4;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __grid_constant__ CombineParams p) {
    __shared__ float s_m[64];
    __shared__ float s_z[64];
    __shared__ float s_w[64];
    __shared__ float s_zt;
    __shared__ __align__(16) float s_v[kCombineThreads * 4];
    __shared__ float s_p[kCombineThreads];
    __shared__ float s_a[256];
    const int row = blockIdx.x, tid = threadIdx.x, d = p.d, ns = p.n_splits;
    const int tpr = d >> 2, groups = kCombineThreads / tpr;
    const int grp = tid / tpr, c4 = tid % tpr;
    const int stride = d + kPartPad;
    // dense Pi: thread (ugrp, ci) takes rows ugrp + k ug of column ci
    const int ug = kCombineThreads / d, ci = tid % d, ugrp = tid / d;
    const int nk = d / ug;  // rows of Pi a thread takes: 4, 16 or 64 for d = 64, 128, 256
    const float sg = (p.rht && tid < d) ? p.sgn[tid] : 0.0f;
    // launched as a programmatic dependent of the scan: wait for its grid to
    // complete and its partials to be visible (a no-op on a plain launch)
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const float* base = p.partial + (int64_t)row * ns * stride;

    float m = -INFINITY, z = 0.0f;
    float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int s0 = grp; s0 < ns; s0 += groups * kCombinePer) {
        float4 av[kCombinePer];
        float mv[kCombinePer], zv[kCombinePer];
        // unconditional loads (an index past the last split reads the last
        // one again and is then dropped): a load behind a branch is waited
        // for where the paths merge, which would serialise them
#pragma unroll
        for (int k = 0; k < kCombinePer; ++k) {
            const int s = s0 + k * groups;
            const float* ps = base + (int64_t)min(s, ns - 1) * stride;
            av[k] = *reinterpret_cast<const float4*>(ps + 4 * c4);
            const float2 mz = *reinterpret_cast<const float2*>(ps + d);
            mv[k] = s < ns ? mz.x : -INFINITY;
            zv[k] = mz.y;
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
    if (tid < 32) {
        // M* over the groups (lane l holds groups l and l + 32), their weights
        // and Z = sum_k z_k 2^(m_k - M*)
        const int lane = tid;
        const float m0 = lane < groups ? s_m[lane] : -INFINITY;
        const float m1 = lane + 32 < groups ? s_m[lane + 32] : -INFINITY;
        const float mstar = warp_max(fmaxf(m0, m1));
        const float w0 = (m0 == -INFINITY) ? 0.0f : exp2f(m0 - mstar);
        const float w1 = (m1 == -INFINITY) ? 0.0f : exp2f(m1 - mstar);
        float zt = 0.0f;
        if (lane < groups) {
            s_w[lane] = w0;
            zt = s_z[lane] * w0;
        }
        if (lane + 32 < groups) {
            s_w[lane + 32] = w1;
            zt = fmaf(s_z[lane + 32], w1, zt);
        }
        zt = warp_sum(zt);
        if (lane == 0) s_zt = zt;
    }
    __syncthreads();
    {
        // part q of coordinate ci: the groups q, q + ug, ... (groups / ug of them)
        float acc = 0.0f;
        for (int k = ugrp; k < groups; k += ug) acc = fmaf(s_v[k * d + ci], s_w[k], acc);
        s_p[tid] = acc;
    }
    __syncthreads();
    if (tid < d) {
        float at = 0.0f;
        for (int q = 0; q < ug; ++q) at += s_p[q * d + tid];
        const float zt = s_zt;
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
            o = acc * sg * p.inv_sqrt_d;
        }
    } else {
        // o_i = sum_k Pi[k][i] a_k, the k range split over ug groups of d threads
        float part = 0.0f;
        // 16 independent loads into registers first, then the products: one
        // round of memory latency per 16 rows, not one per row
        for (int k0 = 0; k0 < nk; k0 += 16) {
            float pv[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                pv[j] = k0 + j < nk ? __ldg(p.pi32 + (size_t)(ugrp + (k0 + j) * ug) * d + ci) : 0.0f;
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
// The same merge for d = 128 with the random-sign Hadamard un-rotation and at
// most kCombBulkMaxSplits splits (a decode step): one CTA of 128 threads per
// query row. The row's partials are contiguous (n_splits x (d + pad)
// floats), so one bulk copy brings all of them into shared memory at once,
// one round of latency for the whole row. Then thread t takes split t for
// M* = max M_s (a block reduction), the weights w_s = 2^(M_s - M*) (0 for a
// split that saw no token) and Z = sum w_s Z_s, and thread i sums
// a_i = sum_s w_s a_s[i] over the splits in order; o = s * (H a) / sqrt(d)
// with H by warp butterflies and one exchange through shared memory. The CTA
// is small (128 threads, the partials in shared memory), so it fits beside
// the scan's CTAs and is resident, waiting, before the scan ends.
// ---------------------------------------------------------------------------
constexpr int kCombBulkThreads = 128;
constexpr int kCombBulkMaxSplits = 93;  // (d + pad) * 4 bytes per split: at most 48 KB of shared memory

__global__ void __launch_bounds__(kCombBulkThreads) combine_bulk_kernel(const __grid_constant__ CombineParams p) {
    constexpr int D = 128, stride = D + kPartPad;
    extern __shared__ __align__(128) unsigned char cb_smem[];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ float s_w[kCombBulkThreads];
    __shared__ float s_red[2][4];
    __shared__ float s_y[D];
    const float* part = reinterpret_cast<const float*>(cb_smem);
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, ns = p.n_splits;
    const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&s_bar);
    const float sg = p.sgn[tid];  // does not depend on the scan: read while it runs
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    // launched as a programmatic dependent of the scan: wait for its grid to
    // complete and its partials to be visible (a no-op on a plain launch)
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)(ns * stride * 4);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s((uint32_t)__cvta_generic_to_shared(cb_smem), p.partial + (int64_t)row * ns * stride, bytes, bar);
    }
    if (!__syncthreads_and(mbar_wait_bounded(bar, 0, kWaitLimitNs, p.err, kErrScanWait))) {
        // the copy did not land in time (the error word says so): it must
        // still land before the shared memory is released
        mbar_wait_bounded(bar, 0, kWaitLimitNs, p.err, kErrScanWait);
        return;
    }
    // M* over the splits (thread t holds split t)
    const float ms = tid < ns ? part[tid * stride + D] : -INFINITY;
    const float mw = warp_max(ms);
    if (lane == 0) s_red[0][warp] = mw;
    __syncthreads();
    const float mstar = fmaxf(fmaxf(s_red[0][0], s_red[0][1]), fmaxf(s_red[0][2], s_red[0][3]));
    const float w = (ms == -INFINITY) ? 0.0f : exp2f(ms - mstar);
    const float zw = warp_sum(tid < ns ? part[tid * stride + D + 1] * w : 0.0f);
    s_w[tid] = w;
    if (lane == 0) s_red[1][warp] = zw;
    __syncthreads();
    const float z = (s_red[1][0] + s_red[1][1]) + (s_red[1][2] + s_red[1][3]);
    float at = 0.0f;
#pragma unroll 8
    for (int k = 0; k < ns; ++k) at = fmaf(part[k * stride + tid], s_w[k], at);
    // o = s * (H a) / sqrt(d): strides 1..16 across the lanes, 32 and 64 as a
    // 4-point transform over the warps through shared memory
    float y = z > 0.0f ? at / z : 0.0f;
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
        const float t = __shfl_xor_sync(TQ_FULL_MASK, y, h);
        y = (lane & h) ? (t - y) : (y + t);
    }
    s_y[tid] = y;
    __syncthreads();
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float t = s_y[lane + 32 * k];
        acc += (__popc(warp & k) & 1) ? -t : t;
    }
    const float o = acc * sg * p.inv_sqrt_d;
    if (p.out_dtype == 1)
        reinterpret_cast<__nv_bfloat16*>(p.out)[(int64_t)row * D + tid] = __float2bfloat16_rn(o);
    else
        reinterpret_cast<float*>(p.out)[(int64_t)row * D + tid] = o;
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
    // 8 splits at a time, every load unconditional (an index past the last
    // split reads the last one again; a branch around a load would serialise
    // the loads), the splits summed in order with weight 0 for the dropped
    constexpr int kB = 8;
    float mstar = -INFINITY;
    for (int s0 = 0; s0 < ns; s0 += kB) {
        float mv[kB];
#pragma unroll
        for (int k = 0; k < kB; ++k) mv[k] = base[(int64_t)min(s0 + k, ns - 1) * stride + 128];
#pragma unroll
        for (int k = 0; k < kB; ++k) mstar = fmaxf(mstar, mv[k]);
    }
    float z = 0.0f;
    float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (mstar != -INFINITY) {
        for (int s0 = 0; s0 < ns; s0 += kB) {
            float4 av[kB];
            float2 mz[kB];
#pragma unroll
            for (int k = 0; k < kB; ++k) {
                const float* ps = base + (int64_t)min(s0 + k, ns - 1) * stride;
                av[k] = *reinterpret_cast<const float4*>(ps + 4 * lane);
                mz[k] = *reinterpret_cast<const float2*>(ps + 128);
            }
#pragma unroll
            for (int k = 0; k < kB; ++k) {
                const bool use = s0 + k < ns && mz[k].x != -INFINITY;
                const float w = exp2f(use ? mz[k].x - mstar : -INFINITY);
                z = use ? fmaf(mz[k].y, w, z) : z;
                a.x = use ? fmaf(av[k].x, w, a.x) : a.x;
                a.y = use ? fmaf(av[k].y, w, a.y) : a.y;
                a.z = use ? fmaf(av[k].z, w, a.z) : a.z;
                a.w = use ? fmaf(av[k].w, w, a.w) : a.w;
            }
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
