// Inner-product search scored from the codes, with a streaming top-k.
//
// Follows: A2A TurboQuant explainer, "Benchmarks and real-world performance"
// (GloVe d = 200 top-k recall) and "Applications" (vector databases). Each
// database row is scored with the decode logit estimator; the k best rows
// per query are kept, ties broken toward the lower row id.
#pragma once

#include "common.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kTopkWarps = 8;
constexpr int kTopkQ = 8;   // queries per CTA
constexpr int kTopkMaxK = 32;

// a ranks before b: higher score, or equal score and lower id
__device__ __forceinline__ bool better(float sa, int ia, float sb, int ib) {
    return sa > sb || (sa == sb && ia < ib);
}

// Insert (s, id) into a list sorted best-first of length k (kept in smem).
__device__ __forceinline__ void list_insert(float* ls, int* li, int k, float s, int id) {
    if (!better(s, id, ls[k - 1], li[k - 1])) return;
    int pos = k - 1;
    while (pos > 0 && better(s, id, ls[pos - 1], li[pos - 1])) {
        ls[pos] = ls[pos - 1];
        li[pos] = li[pos - 1];
        --pos;
    }
    ls[pos] = s;
    li[pos] = id;
}

// grid: (chunks, ceil(nq / kTopkQ)); each warp scores one database row at a
// time for the CTA's kTopkQ queries; lane q keeps query q's list for the warp.
template <int VPL, int CB, bool PROD>
__global__ void __launch_bounds__(kTopkWarps * 32) topk_scan_kernel(const __grid_constant__ TopkParams p) {
    constexpr int DMAX = 32 * VPL;
    __shared__ float s_q[kTopkQ][DMAX];
    __shared__ float s_u[kTopkQ][DMAX];
    __shared__ float s_c[kMaxLevels];
    __shared__ float s_ls[kTopkWarps][kTopkQ][kTopkMaxK];
    __shared__ int s_li[kTopkWarps][kTopkQ][kTopkMaxK];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int chunk = blockIdx.x;
    const int q0 = blockIdx.y * kTopkQ;
    const int nq_here = min(kTopkQ, p.nq - q0);
    const int d = p.d, m = p.m, k = p.k;
    if (threadIdx.x < kMaxLevels) s_c[threadIdx.x] = p.c[threadIdx.x];
    for (int e = threadIdx.x; e < kTopkQ * DMAX; e += blockDim.x) {
        const int q = e / DMAX, i = e % DMAX;
        const bool ok = q < nq_here && i < d;
        s_q[q][i] = ok ? p.qprime[(int64_t)(q0 + q) * d + i] : 0.0f;
        if (PROD) s_u[q][i] = (q < nq_here && i < m) ? p.u[(int64_t)(q0 + q) * m + i] : 0.0f;
    }
    for (int e = threadIdx.x; e < kTopkWarps * kTopkQ * kTopkMaxK; e += blockDim.x) {
        (&s_ls[0][0][0])[e] = -INFINITY;
        (&s_li[0][0][0])[e] = 0x7fffffff;
    }
    __syncthreads();

    const int64_t r0 = (int64_t)chunk * p.chunk_rows;
    const int64_t r1 = min(r0 + p.chunk_rows, p.n_db);
    const int cwords = p.code_stride >> 2;
    const int mpl = (m + 31) >> 5;
    for (int64_t row = r0 + warp; row < r1; row += kTopkWarps) {
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(p.codes + row * p.code_stride);
        float cd[VPL];
        if (VPL * lane < d) {
            const uint32_t chunkbits = stream_bits(cw, CB * VPL * lane, CB * VPL, cwords);
#pragma unroll
            for (int r = 0; r < VPL; ++r)
                cd[r] = (VPL * lane + r < d) ? s_c[(chunkbits >> (CB * r)) & ((1u << CB) - 1u)] : 0.0f;
        } else {
#pragma unroll
            for (int r = 0; r < VPL; ++r) cd[r] = 0.0f;
        }
        float pm[8];
        float gs = 0.0f;
        if (PROD) {
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(p.signs + row * p.sign_stride);
            uint32_t sb = 0;
            if (mpl * lane < m) sb = stream_bits(sw, mpl * lane, mpl, p.sign_stride >> 2);
#pragma unroll
            for (int r = 0; r < 8; ++r) pm[r] = (r < mpl && mpl * lane + r < m) ? (((sb >> r) & 1u) ? 1.0f : -1.0f) : 0.0f;
            gs = p.qjl_scale * f16_bits_to_f32(p.rnorm[row]);
        }
        const float nrm = f16_bits_to_f32(p.norm[row]);
        float sc[kTopkQ];
#pragma unroll
        for (int q = 0; q < kTopkQ; ++q) {
            float a = 0.0f;
#pragma unroll
            for (int r = 0; r < VPL; ++r) {
                const int e = VPL * lane + r;
                if (e < DMAX) a = fmaf(s_q[q][e], cd[r], a);
            }
            if (PROD) {
                float s = 0.0f;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int j = mpl * lane + r;
                    if (r < mpl && j < DMAX) s = fmaf(s_u[q][j], pm[r], s);
                }
                a = fmaf(gs, s, a);
            }
            sc[q] = a;
        }
#pragma unroll
        for (int q = 0; q < kTopkQ; ++q) sc[q] = warp_sum(sc[q]) * nrm;
        // lane q inserts into query q's list
        float mine = sc[0];
#pragma unroll
        for (int q = 1; q < kTopkQ; ++q)
            if (lane == q) mine = sc[q];
        if (lane < nq_here) list_insert(s_ls[warp][lane], s_li[warp][lane], k, mine, (int)row);
        __syncwarp();
    }
    __syncthreads();
    // merge the warps' lists: warp q merges query q
    if (warp < nq_here) {
        const int q = warp;
        if (lane == 0) {
            for (int w = 1; w < kTopkWarps; ++w)
                for (int e = 0; e < k; ++e) list_insert(s_ls[0][q], s_li[0][q], k, s_ls[w][q][e], s_li[w][q][e]);
        }
        __syncwarp();
        for (int e = lane; e < k; e += 32) {
            const int64_t o = ((int64_t)(q0 + q) * p.n_chunks + chunk) * p.k + e;
            p.cand_score[o] = s_ls[0][q][e];
            p.cand_id[o] = s_li[0][q][e];
        }
    }
}

// One warp per query: select the k best of n_chunks * k candidates.
static __global__ void __launch_bounds__(256) topk_merge_kernel(const __grid_constant__ TopkParams p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int q = blockIdx.x * 8 + warp;
    if (q >= p.nq) return;
    const int64_t n = (int64_t)p.n_chunks * p.k;
    float* cs = p.cand_score + (int64_t)q * n;
    int32_t* ci = p.cand_id + (int64_t)q * n;
    for (int e = 0; e < p.k; ++e) {
        float bs = -INFINITY;
        int bi = 0x7fffffff;
        int64_t bpos = -1;
        for (int64_t j = lane; j < n; j += 32) {
            if (better(cs[j], ci[j], bs, bi)) {
                bs = cs[j];
                bi = ci[j];
                bpos = j;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float os = __shfl_xor_sync(TQ_FULL_MASK, bs, o);
            int oi = __shfl_xor_sync(TQ_FULL_MASK, bi, o);
            long long op = __shfl_xor_sync(TQ_FULL_MASK, (long long)bpos, o);
            if (better(os, oi, bs, bi)) {
                bs = os;
                bi = oi;
                bpos = op;
            }
        }
        if (lane == 0) {
            p.ids[(int64_t)q * p.k + e] = bi;
            p.scores[(int64_t)q * p.k + e] = bs;
            if (bpos >= 0) {
                cs[bpos] = -INFINITY;
                ci[bpos] = 0x7fffffff;
            }
        }
        __syncwarp();
    }
}

}  // namespace tqk
