// Decode attention scored from the packed codes: query preparation, split-K
// scan with online softmax, and the split merge + un-rotation.
//
// Follows: A2A TurboQuant explainer, end of "Stage 2" (logits straight from
// the compressed indices, no full de-quantization) and "How to implement"
// (the fused kernel rotates the query once); Qiita TurboQuant article, "One
// more stage so attention does not break" (residual sign term). The softmax,
// the value sum in the rotated domain and the single un-rotation are this
// library's reading of how the output is formed.
#pragma once

#include "common.cuh"
#include "tq_launch.h"

namespace tqk {

// ---------------------------------------------------------------------------
// q' = Pi q and u = S q', one warp per query row. Lane owns coordinates
// VPL*lane .. VPL*lane + VPL - 1.
// ---------------------------------------------------------------------------
template <int VPL>
__global__ void __launch_bounds__(256) query_prep_kernel(const __grid_constant__ PrepParams p) {
    __shared__ float s_buf[8][32 * VPL];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = (int64_t)blockIdx.x * 8 + warp;
    if (row >= p.rows) return;
    const int d = p.d;
    float x[VPL];
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
        int e = VPL * lane + r;
        float v = 0.0f;
        if (e < d) {
            if (p.q_dtype == 1)
                v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.q)[row * d + e]);
            else
                v = reinterpret_cast<const float*>(p.q)[row * d + e];
        }
        x[r] = v;
    }
    float y[VPL];
    if (p.rht) {
#pragma unroll
        for (int r = 0; r < VPL; ++r) y[r] = x[r] * p.sgn[VPL * lane + r];
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
        for (int r = 0; r < VPL; ++r) y[r] *= p.inv_sqrt_d;
    } else {
#pragma unroll
        for (int r = 0; r < VPL; ++r) {
            int e = VPL * lane + r;
            if (e < d) s_buf[warp][e] = x[r];
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < VPL; ++r) y[r] = 0.0f;
        for (int j = 0; j < d; ++j) {
            const float xj = s_buf[warp][j];
            const float* rowp = p.pit32 + (size_t)j * d;
#pragma unroll
            for (int r = 0; r < VPL; ++r) {
                int e = VPL * lane + r;
                if (e < d) y[r] = fmaf(__ldg(rowp + e), xj, y[r]);
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
        int e = VPL * lane + r;
        if (e < d) {
            p.qprime[row * d + e] = y[r];
            s_buf[warp][e] = y[r];
        }
    }
    __syncwarp();
    if (p.u) {
        const int m = p.m, mpl = (m + 31) >> 5;
        float acc[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
        for (int i = 0; i < d; ++i) {
            const float qi = s_buf[warp][i];
            const float* rowp = p.st32 + (size_t)i * m;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                int j = mpl * lane + r;
                if (r < mpl && j < m) acc[r] = fmaf(__ldg(rowp + j), qi, acc[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            int j = mpl * lane + r;
            if (r < mpl && j < m) p.u[row * m + j] = acc[r];
        }
    }
}

// ---------------------------------------------------------------------------
// Split-K decode scan (d = 128, m = 128): CTA = (split, KV head, batch), 4
// warps; a warp takes one token at a time, its lanes own 4 coordinates each.
// Writes per query head (M, Z, a[128]) for its token range (log2 domain).
// ---------------------------------------------------------------------------
constexpr int kDecWarps = 4;

template <int KB, int VB, int G>
__global__ void __launch_bounds__(kDecWarps * 32) decode_kernel(const __grid_constant__ DecodeParams p) {
    constexpr int D = 128;
    __shared__ float s_kc[kMaxLevels], s_vc[kMaxLevels];
    __shared__ float s_acc[kDecWarps][G][D];
    __shared__ float s_mz[kDecWarps][G][2];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int split = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;
    if (threadIdx.x < kMaxLevels) {
        s_kc[threadIdx.x] = p.kc[threadIdx.x];
        s_vc[threadIdx.x] = p.vc[threadIdx.x];
    }
    __syncthreads();

    // a length outside [0, min(capacity, max_seq_len)] is clamped into it
    const int L = max(0, (int)min((int64_t)p.seq_lens[b], min(p.capacity, (int64_t)p.max_seq_len)));
    const int t0 = split * p.chunk;
    const int t1 = min(t0 + p.chunk, L);

    int qrow[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        int h = p.use_table ? (int)p.head_table[kv * G + j] : kv * G + j;
        qrow[j] = b * p.hq + h;
    }
    float4 qv[G], uv[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        qv[j] = reinterpret_cast<const float4*>(p.qprime + (int64_t)qrow[j] * D)[lane];
        uv[j] = reinterpret_cast<const float4*>(p.u + (int64_t)qrow[j] * D)[lane];
    }
    float M[G], Z[G], acc[G][4];
#pragma unroll
    for (int j = 0; j < G; ++j) {
        M[j] = -INFINITY;
        Z[j] = 0.0f;
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[j][r] = 0.0f;
    }

    const int64_t rowbase = ((int64_t)b * p.hkv + kv) * p.capacity;
    const int kwords = p.kcode_stride >> 2, vwords = p.vcode_stride >> 2;
    for (int t = t0 + warp; t < t1; t += kDecWarps) {
        const int64_t slot = rowbase + t;
        const uint32_t* kw = reinterpret_cast<const uint32_t*>(p.kcodes + slot * p.kcode_stride);
        const uint32_t* sw = reinterpret_cast<const uint32_t*>(p.ksigns + slot * p.ksign_stride);
        const uint32_t* vw = reinterpret_cast<const uint32_t*>(p.vcodes + slot * p.vcode_stride);
        const uint32_t kchunk = stream_bits(kw, KB * 4 * lane, KB * 4, kwords);
        const uint32_t schunk = (sw[lane >> 3] >> ((lane & 7) * 4)) & 0xFu;
        const uint32_t vchunk = stream_bits(vw, VB * 4 * lane, VB * 4, vwords);
        const float kn = f16_bits_to_f32(p.knorm[slot]);
        const float kg = f16_bits_to_f32(p.krnorm[slot]);
        const float vn = f16_bits_to_f32(p.vnorm[slot]);
        float kd[4], pm[4], vd[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            kd[r] = s_kc[(kchunk >> (KB * r)) & ((1u << KB) - 1u)];
            pm[r] = ((schunk >> r) & 1u) ? 1.0f : -1.0f;
            vd[r] = vn * s_vc[(vchunk >> (VB * r)) & ((1u << VB) - 1u)];
        }
        const float gs = p.qjl_scale * kg;
        float part[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float c = qv[j].x * kd[0] + qv[j].y * kd[1] + qv[j].z * kd[2] + qv[j].w * kd[3];
            float s = uv[j].x * pm[0] + uv[j].y * pm[1] + uv[j].z * pm[2] + uv[j].w * pm[3];
            part[j] = fmaf(gs, s, c);
        }
#pragma unroll
        for (int j = 0; j < G; ++j) part[j] = warp_sum(part[j]);
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float logit = kn * part[j];
            if (p.logits != nullptr && lane == j)
                p.logits[(int64_t)qrow[j] * p.max_seq_len + t] = logit;
            const float s = logit * p.scale_log2;
            const float mn = fmaxf(M[j], s);
            const float corr = exp2f(M[j] - mn);
            const float pr = exp2f(s - mn);
            Z[j] = fmaf(Z[j], corr, pr);
            M[j] = mn;
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[j][r] = fmaf(acc[j][r], corr, pr * vd[r]);
        }
    }

    // merge the 4 warps of the CTA, then write this split's partials
#pragma unroll
    for (int j = 0; j < G; ++j) {
#pragma unroll
        for (int r = 0; r < 4; ++r) s_acc[warp][j][4 * lane + r] = acc[j][r];
        if (lane == 0) {
            s_mz[warp][j][0] = M[j];
            s_mz[warp][j][1] = Z[j];
        }
    }
    __syncthreads();
    const int i = threadIdx.x;  // coordinate 0..127
#pragma unroll
    for (int j = 0; j < G; ++j) {
        float mstar = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) mstar = fmaxf(mstar, s_mz[w][j][0]);
        float z = 0.0f, a = 0.0f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            const float mw = s_mz[w][j][0];
            const float wt = (mw == -INFINITY) ? 0.0f : exp2f(mw - mstar);
            z = fmaf(s_mz[w][j][1], wt, z);
            a = fmaf(s_acc[w][j][i], wt, a);
        }
        float* out = p.partial + ((int64_t)qrow[j] * p.n_splits + split) * (D + 2);
        out[i] = a;
        if (i == 0) {
            out[D] = mstar;
            out[D + 1] = z;
        }
    }
}

// ---------------------------------------------------------------------------
// Merge the splits of one query row and un-rotate: o = Pi^T (a / Z).
// Block = d threads (d <= 256).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineParams p) {
    __shared__ float s_a[256];
    __shared__ float s_w[1024];
    const int row = blockIdx.x;
    const int i = threadIdx.x, d = p.d;
    const float* base = p.partial + (int64_t)row * p.n_splits * (d + 2);
    float mstar = -INFINITY;
    for (int s = 0; s < p.n_splits; ++s) mstar = fmaxf(mstar, base[(int64_t)s * (d + 2) + d]);
    float z = 0.0f, a = 0.0f;
    for (int s0 = 0; s0 < p.n_splits; s0 += 1024) {
        const int cnt = min(1024, p.n_splits - s0);
        __syncthreads();
        for (int s = i; s < cnt; s += blockDim.x) {
            const float ms = base[(int64_t)(s0 + s) * (d + 2) + d];
            s_w[s] = (ms == -INFINITY) ? 0.0f : exp2f(ms - mstar);
        }
        __syncthreads();
        for (int s = 0; s < cnt; ++s) {
            const float* ps = base + (int64_t)(s0 + s) * (d + 2);
            z = fmaf(ps[d + 1], s_w[s], z);
            a = fmaf(ps[i], s_w[s], a);
        }
    }
    s_a[i] = (z > 0.0f) ? a / z : 0.0f;
    __syncthreads();
    float o = 0.0f;
    if (p.rht) {
        // o = s * (H a) / sqrt(d): in-place Walsh-Hadamard on shared memory
        for (int h = 1; h < d; h <<= 1) {
            float v = s_a[i], w = s_a[i ^ h];
            __syncthreads();
            s_a[i] = (i & h) ? (w - v) : (v + w);
            __syncthreads();
        }
        o = s_a[i] * p.sgn[i] * p.inv_sqrt_d;
    } else {
        for (int k = 0; k < d; ++k) o = fmaf(__ldg(p.pi32 + (size_t)k * d + i), s_a[k], o);
    }
    if (p.out_dtype == 1)
        reinterpret_cast<__nv_bfloat16*>(p.out)[(int64_t)row * d + i] = __float2bfloat16_rn(o);
    else
        reinterpret_cast<float*>(p.out)[(int64_t)row * d + i] = o;
}

}  // namespace tqk
