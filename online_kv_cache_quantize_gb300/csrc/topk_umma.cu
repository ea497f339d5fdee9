// Inner-product search on the 5th-generation tensor cores (tcgen05).
//
// Same scores as topk.cuh (A2A TurboQuant explainer, "Benchmarks and
// real-world performance" and "Applications"; the decode logit estimator
// l = n (<q', c[idx]> + sqrt(pi/2)/m * gamma <u, 2z - 1>) per database row),
// computed as a dense contraction: for a tile of 128 database rows and a
// block of 32 queries,
//     D[row][2j + s] = sum_i A[row][i] B[2j + s][i]
// with A the de-quantized rows (lam * centroid as fp16, from a pair table;
// the fp16 residual of lam * centroid as a second table when the codebook
// has 8 or more cells; gamma * (2z - 1) for the sign part) and B the queries
// split into fp16 hi (s = 0) and lo (s = 1) halves (q' against the centroid
// parts, lam * kappa * u against the sign part). The score is
// n * (D[row][2j] + D[row][2j + 1]) / lam.
//
// Per CTA: 32 queries (B resident in shared memory for the whole chunk) and a
// chunk of database rows. Per 128-row tile: the packed codes and signs land
// in a staging buffer by bulk copy (double-buffered, one tile ahead); 256
// threads de-quantize each A segment into a core-matrix tile (two buffers,
// so the next segment is built while the tensor core runs on the previous
// one); one thread issues the MMAs into a 128 x 64 fp32 TMEM accumulator;
// the epilogue reads it back with tcgen05.ld and keeps per-warp top-k lists,
// merged per query at the end into the chunk's candidates.
#include "pipeline.cuh"
#include "tcgen05.cuh"
#include "topk.cuh"

namespace tqk {

constexpr int kTuRows = 128;    // database rows per tile (MMA M)
constexpr int kTuQ = 32;        // queries per CTA
constexpr int kTuN = 2 * kTuQ;  // MMA N: hi and lo column per query
constexpr int kTuWarps = 16;
constexpr int kTuThreads = 32 * kTuWarps;
constexpr int kTuQpw = kTuQ / (kTuWarps / 4);  // queries per warp in the epilogue (8)
constexpr int kTuParts = kTuThreads / kTuRows;  // threads per row in the de-quantize (4)
constexpr int kTuSmemLimit = 227 * 1024 - 4096;  // dynamic part; static tables stay below 4 KB

struct TuLayout {
    size_t b, a0, a1, st0, st1, sgn, nrm, ls, li, total;
    int kcb, stage_bytes;
};

__host__ __device__ inline TuLayout tu_layout(int ks, int nseg_b, int code_stride, int sign_stride, int k) {
    TuLayout L;
    L.kcb = nseg_b * ks;
    const size_t bb = (size_t)kTuN * L.kcb * 2;
    const size_t ab = (size_t)kTuRows * ks * 2;
    L.stage_bytes = kTuRows * (code_stride + sign_stride) + 16;  // + slack for the 8-byte reads at a row end
    L.b = 0;
    L.a0 = bb;
    L.a1 = L.a0 + ab;
    L.st0 = L.a1 + ab;
    L.st1 = L.st0 + ((L.stage_bytes + 127) / 128) * 128;
    L.sgn = L.st1 + ((L.stage_bytes + 127) / 128) * 128;
    L.nrm = L.sgn + 256 * 16;  // [2 buffers][128 rows] norm, then [2][128] gamma (fp32)
    L.ls = L.nrm + 4 * kTuRows * 4;
    L.li = L.ls + (size_t)kTuWarps * kTuQpw * k * 4;
    L.total = L.li + (size_t)kTuWarps * kTuQpw * k * 4;
    return L;
}

template <int CB, bool PROD, bool LO>
__global__ void __launch_bounds__(kTuThreads, 1) topk_umma_kernel(const __grid_constant__ TopkParams p) {
    constexpr int NSEG_A = 1 + (LO ? 1 : 0) + (PROD ? 1 : 0);
    constexpr int NSEG_B = 1 + (PROD ? 1 : 0);
    constexpr int NT = 1 << (2 * CB);
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t s_bar[2];    // MMA completion per A buffer
    __shared__ __align__(8) uint64_t s_sbar[2];   // staging copies per buffer
    __shared__ __align__(8) uint64_t s_abar[2];   // all MMAs of a tile done, per TMEM accumulator
    __shared__ uint32_t s_tmem;
    __shared__ uint32_t s_ktab[NT];
    __shared__ uint32_t s_klo[LO ? NT : 1];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ks = p.ks, k = p.k, d = p.d, m = p.m;
    const int cs = p.code_stride, ss = PROD ? p.sign_stride : 0;
    const TuLayout Lo = tu_layout(ks, NSEG_B, cs, ss, k);
    const int kcb = Lo.kcb;
    unsigned char* sB = smem + Lo.b;
    // buffer x of a pair at base + x * stride (no arrays indexed at run time)
    unsigned char* const sA0 = smem + Lo.a0;
    const size_t sA_stride = Lo.a1 - Lo.a0;
    unsigned char* const sSt0 = smem + Lo.st0;
    const size_t sSt_stride = Lo.st1 - Lo.st0;
    const uint4* s_sgn = reinterpret_cast<const uint4*>(smem + Lo.sgn);
    float* s_nrm = reinterpret_cast<float*>(smem + Lo.nrm);          // [2][128]: n of each row
    float* s_gam = s_nrm + 2 * kTuRows;                              // [2][128]: gamma (PROD)
    float* s_ls = reinterpret_cast<float*>(smem + Lo.ls);  // [warps][queries per warp][k]
    int* s_li = reinterpret_cast<int*>(smem + Lo.li);

    const int chunk = blockIdx.x;
    const int q0 = blockIdx.y * kTuQ;
    const int nq_here = min(kTuQ, p.nq - q0);
    const int64_t r0 = (int64_t)chunk * p.chunk_rows;
    const int64_t r1 = min(r0 + p.chunk_rows, p.n_db);
    const float lam_kappa = p.qjl_scale / p.inv_lam;

    // ---- tables, lists, B tile ----
    for (int i = tid; i < NT; i += blockDim.x) {
        s_ktab[i] = p.ktab[i];
        if constexpr (LO) s_klo[i] = p.ktab_lo[i];
    }
    for (int i = tid; i < 256; i += blockDim.x) {
        // flips that make the fp16 pair (-g, -g) positive where sign bits 2w, 2w+1 of byte i are set
        uint4 v;
        v.x = ((uint32_t)(i & 1) << 15) | ((uint32_t)((i >> 1) & 1) << 31);
        v.y = ((uint32_t)((i >> 2) & 1) << 15) | ((uint32_t)((i >> 3) & 1) << 31);
        v.z = ((uint32_t)((i >> 4) & 1) << 15) | ((uint32_t)((i >> 5) & 1) << 31);
        v.w = ((uint32_t)((i >> 6) & 1) << 15) | ((uint32_t)((i >> 7) & 1) << 31);
        reinterpret_cast<uint4*>(smem + Lo.sgn)[i] = v;
    }
    // B tile: row 2j + s holds query j's hi (s = 0) or lo (s = 1) fp16 half;
    // columns [0, ks) are q', [ks, 2 ks) lam * kappa * u (PROD)
    for (int j = 0; j < kTuQ; ++j) {
        const bool qv = j < nq_here;
        const float* qp = p.qprime + (int64_t)(q0 + (qv ? j : 0)) * d;
        const float* up = PROD ? p.u + (int64_t)(q0 + (qv ? j : 0)) * m : nullptr;
        for (int col = 2 * tid; col < kcb; col += 2 * blockDim.x) {
            const bool sgn = col >= ks;
            const int i = sgn ? col - ks : col;
            const int lim = sgn ? m : d;
            const float* src = sgn ? up : qp;
            const float sc_ = sgn ? lam_kappa : 1.0f;
            const float v0 = (qv && i < lim) ? sc_ * src[i] : 0.0f;
            const float v1 = (qv && i + 1 < lim) ? sc_ * src[i + 1] : 0.0f;
            *reinterpret_cast<uint32_t*>(sB + umma_off(2 * j, col, kcb)) = half_split(v0, 0) | (half_split(v1, 0) << 16);
            *reinterpret_cast<uint32_t*>(sB + umma_off(2 * j + 1, col, kcb)) =
                half_split(v0, 1) | (half_split(v1, 1) << 16);
        }
    }
    // mbarrier x of each pair at base + 8 x
    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(&s_bar[0]);
    const uint32_t sbar0 = (uint32_t)__cvta_generic_to_shared(&s_sbar[0]);
    const uint32_t abar0 = (uint32_t)__cvta_generic_to_shared(&s_abar[0]);
    if (tid == 0) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar0 + 8 * x, 1);
            mbar_init(sbar0 + 8 * x, 1);
            mbar_init(abar0 + 8 * x, 1);
        }
        mbar_init_fence();
    }
    if (warp == 0) {  // two accumulators: tile t's MMAs run while tile t - 1's epilogue reads the other
        tmem_alloc((uint32_t)__cvta_generic_to_shared(&s_tmem), 2 * kTuN);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;

    // staging of tile t (codes then signs of its rows) into buffer t & 1, by thread 0
    const int64_t ntile = r1 > r0 ? (r1 - r0 + kTuRows - 1) / kTuRows : 0;
    auto stage = [&](int64_t t) {
        const int64_t t0 = r0 + t * kTuRows;
        const int rows = (int)min((int64_t)kTuRows, r1 - t0);
        const int b = (int)(t & 1);
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(sSt0 + b * sSt_stride);
        const uint32_t sb_ = sbar0 + 8 * b;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(sb_, (uint32_t)rows * (cs + ss));
        bulk_g2s(dst, p.codes + t0 * cs, (uint32_t)rows * cs, sb_);
        if constexpr (PROD) bulk_g2s(dst + kTuRows * cs, p.signs + t0 * ss, (uint32_t)rows * ss, sb_);
    };
    if (tid == 0 && ntile > 0) stage(0);

    const uint32_t idesc = umma_idesc_f16(kTuRows, kTuN);
    const uint32_t sA_a0 = (uint32_t)__cvta_generic_to_shared(sA0);
    // MMA descriptors of k-step 0; k-step s starts 256 s bytes (16 s in the
    // descriptor's address field) further on
    const uint64_t descA0 = umma_desc(sA_a0, 128, ks * 16);
    const uint64_t descB0 = umma_desc((uint32_t)__cvta_generic_to_shared(sB), 128, kcb * 16);
    // de-quantize: warp w takes rows 8w .. 8w+7 (lane & 7) and a quarter of their
    // 8-coordinate units (lane >> 3): a quarter warp stores 8 rows of one unit
    // (all banks) and the warp reads 8 rows x 4 units of the staged codes
    const int r = 8 * warp + (lane & 7);
    const int part = lane >> 3;
    const int units = ks / 8, upp = (units + kTuParts - 1) / kTuParts;
    const int u0 = part * upp, u1 = min(units, u0 + upp);
    const int er = 32 * (warp & 3) + lane;  // epilogue: this thread's row (TMEM lane)
    const int ecol = 2 * kTuQpw * (warp >> 2);  // ... and its 2 * kTuQpw columns (kTuQpw queries)
    int step = 0;
    bool ok = true;
    // this warp's top-k list of each of its kTuQpw queries, spread over the
    // lanes: lane e holds entry e (best first; lanes >= k hold nothing)
    float lsc[kTuQpw];
    int lid[kTuQpw];
    // the k-th entry of each list (the admission threshold), the same in every lane
    float thr_s[kTuQpw];
    int thr_i[kTuQpw];
#pragma unroll
    for (int jj = 0; jj < kTuQpw; ++jj) {
        lsc[jj] = -INFINITY;
        lid[jj] = 0x7fffffff;
        thr_s[jj] = -INFINITY;
        thr_i[jj] = 0x7fffffff;
    }

    // norms of a tile's rows: threads 0..127 load tile t + 1's into registers
    // during tile t and publish them into the other smem buffer at its end
    auto load_norms = [&](int64_t t, uint16_t& nv, uint16_t& gv) {
        const int64_t row = r0 + t * kTuRows + tid;
        nv = gv = 0;
        if (tid < kTuRows && t < ntile && row < r1) {
            nv = p.norm[row];
            if constexpr (PROD) gv = p.rnorm[row];
        }
    };
    uint16_t nxt_n = 0, nxt_g = 0;
    load_norms(0, nxt_n, nxt_g);
    if (tid < kTuRows) {
        s_nrm[tid] = f16_bits_to_f32(nxt_n);
        s_gam[tid] = __uint_as_float((uint32_t)nxt_g);  // raw fp16 bits of gamma, carried in a float slot
    }

    // epilogue of tile te: wait for its MMAs, read its accumulator, update the lists
    auto epilogue = [&](int64_t te) -> bool {
        if (__syncthreads_or(!mbar_wait_bounded(abar0 + 8 * (uint32_t)(te & 1), (uint32_t)((te >> 1) & 1), kWaitLimitNs, p.err,
                                                kErrScanWait)))
            return false;
        tc_fence_after_sync();
        float v[2 * kTuQpw];
        static_assert(2 * kTuQpw == 16, "one 16-column TMEM load per warp");
        tmem_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((te & 1) * kTuN + ecol), v);
        tmem_ld_wait();
        const int64_t erow = r0 + te * kTuRows + er;
        const bool evalid = erow < r1;
        const float scale = s_nrm[(te & 1) * kTuRows + er] * p.inv_lam;
        const int id = (int)erow;
#pragma unroll
        for (int jj = 0; jj < kTuQpw; ++jj) {
            const int j = (ecol >> 1) + jj;
            if (j < nq_here) {  // warp-uniform
                const float sc = scale * (v[2 * jj] + v[2 * jj + 1]);
                float ts = thr_s[jj];
                int ti = thr_i[jj];
                // cheap filter (>=); the exact rule (equal scores: lower id first) is applied below
                unsigned cand = __ballot_sync(TQ_FULL_MASK, evalid && sc >= ts);
                while (cand) {
                    const int src = __ffs(cand) - 1;
                    cand &= cand - 1;
                    const float cs_ = __shfl_sync(TQ_FULL_MASK, sc, src);
                    const int ci = __shfl_sync(TQ_FULL_MASK, id, src);
                    if (!better(cs_, ci, ts, ti)) continue;  // the list moved on since the ballot
                    // entries better than the candidate stay, the rest move one lane down
                    const int pos = __popc(__ballot_sync(TQ_FULL_MASK, lane < k && better(lsc[jj], lid[jj], cs_, ci)));
                    const float us = __shfl_up_sync(TQ_FULL_MASK, lsc[jj], 1);
                    const int ui = __shfl_up_sync(TQ_FULL_MASK, lid[jj], 1);
                    if (lane == pos) {
                        lsc[jj] = cs_;
                        lid[jj] = ci;
                    } else if (lane > pos) {
                        lsc[jj] = us;
                        lid[jj] = ui;
                    }
                    ts = __shfl_sync(TQ_FULL_MASK, lsc[jj], k - 1);
                    ti = __shfl_sync(TQ_FULL_MASK, lid[jj], k - 1);
                }
                thr_s[jj] = ts;
                thr_i[jj] = ti;
            }
        }
        return true;
    };

    for (int64_t t = 0; t < ntile && ok; ++t) {
        const int64_t t0 = r0 + t * kTuRows;
        const int sb = (int)(t & 1);
        if (tid == 0 && t + 1 < ntile) stage(t + 1);  // its buffer was last read in tile t - 1
        load_norms(t + 1, nxt_n, nxt_g);
        ok = !__syncthreads_or(!mbar_wait_bounded(sbar0 + 8 * sb, (uint32_t)((t >> 1) & 1), kWaitLimitNs, p.err, kErrScanWait));
        if (!ok) break;
        const float* t_nrm = s_nrm + sb * kTuRows;
        const float* t_gam = s_gam + sb * kTuRows;
        for (int seg = 0; seg < NSEG_A; ++seg) {
            const int buf = step & 1;
            if (step >= 2) {
                ok = !__syncthreads_or(
                    !mbar_wait_bounded(bar0 + 8 * buf, (uint32_t)(((step - 2) >> 1) & 1), kWaitLimitNs, p.err, kErrScanWait));
                if (!ok) break;
            }
            const bool sign_seg = PROD && seg == NSEG_A - 1;
            unsigned char* dstA = sA0 + buf * sA_stride;
            const bool rvalid = t0 + r < r1;
            const unsigned char* crow = sSt0 + sb * sSt_stride + r * cs;
            const unsigned char* srow = sSt0 + sb * sSt_stride + kTuRows * cs + r * ss;
            uint32_t g2 = 0u;
            if (sign_seg) {
                const uint32_t g16 = __float_as_uint(t_gam[r]);
                g2 = (g16 | 0x8000u) | ((g16 | 0x8000u) << 16);  // (-gamma, -gamma)
            }
            static_assert(256 / 8 / kTuParts <= 8, "at most 8 units per thread");
#pragma unroll
            for (int q = 0; q < 8; ++q) {  // fixed trip count: predicated, no loop branches
                const int u = u0 + q;
                if (u >= u1) break;
                uint4 w;
                if (sign_seg) {
                    const uint4 f = s_sgn[rvalid ? srow[u] : 0];
                    w = make_uint4(g2 ^ f.x, g2 ^ f.y, g2 ^ f.z, g2 ^ f.w);
                } else {
                    // 8 codes: CB bytes starting at byte CB * u of the row
                    uint32_t bits = 0u;
                    if (rvalid) {
                        if constexpr (CB == 1) bits = crow[u];
                        else if constexpr (CB == 2) bits = *reinterpret_cast<const uint16_t*>(crow + 2 * u);
                        else if constexpr (CB == 4) bits = *reinterpret_cast<const uint32_t*>(crow + 4 * u);
                        else {
                            const int o = CB * u;
                            const uint32_t* wp = reinterpret_cast<const uint32_t*>(crow + (o & ~3));
                            bits = __funnelshift_r(wp[0], wp[1], 8 * (o & 3));
                        }
                    }
                    const uint32_t* tab = (LO && seg == 1) ? s_klo : s_ktab;
                    constexpr uint32_t M2 = (1u << (2 * CB)) - 1u;
                    w.x = tab[bits & M2];
                    w.y = tab[(bits >> (2 * CB)) & M2];
                    w.z = tab[(bits >> (4 * CB)) & M2];
                    w.w = tab[CB == 4 ? (bits >> 24) : ((bits >> (6 * CB)) & M2)];
                }
                *reinterpret_cast<uint4*>(dstA + umma_off(r, 8 * u, ks)) = w;
            }
            fence_proxy_async_smem();  // the tile is read by the tensor core next
            __syncthreads();
            if (tid == 0) {
                tc_fence_after_sync();
                const int bseg = sign_seg ? 1 : 0;
                const uint32_t dacc = tmem + (uint32_t)((t & 1) * kTuN);
                for (int s = 0; s < ks / 16; ++s)
                    umma_f16(dacc, descA0 + (uint64_t)((buf * sA_stride + 256 * s) >> 4),
                             descB0 + (uint64_t)((bseg * ks / 8 + 2 * s) * 8), idesc, seg > 0 || s > 0);
                umma_commit(bar0 + 8 * buf);
                if (seg == NSEG_A - 1) umma_commit(abar0 + 8 * (uint32_t)(t & 1));
            }
            ++step;
        }
        if (!ok) break;
        // the previous tile's epilogue runs while the tensor core works on this tile
        if (t > 0 && !(ok = epilogue(t - 1))) break;
        tc_fence_before_sync();
        __syncthreads();  // the accumulator just read is overwritten by tile t + 1's first MMA
        if (tid < kTuRows) {  // the norms of tile t + 1 into the buffer tile t - 1 used
            s_nrm[(sb ^ 1) * kTuRows + tid] = f16_bits_to_f32(nxt_n);
            s_gam[(sb ^ 1) * kTuRows + tid] = __uint_as_float((uint32_t)nxt_g);
        }
    }
    if (ok && ntile > 0) ok = epilogue(ntile - 1);
    if (!ok) {
        // a wait ran out (the error word says so): let the copies and MMAs
        // still in flight finish, bounded, before TMEM and smem are released
        for (int b = 0; b < 2; ++b) {
            mbar_wait_bounded(sbar0 + 8 * b, 0, kWaitLimitNs, p.err, kErrScanWait);
            mbar_wait_bounded(sbar0 + 8 * b, 1, kWaitLimitNs, p.err, kErrScanWait);
        }
        if (step > 0)
            mbar_wait_bounded(bar0 + 8 * ((step - 1) & 1), (uint32_t)(((step - 1) >> 1) & 1), kWaitLimitNs, p.err, kErrScanWait);
        if (step >= 2)
            mbar_wait_bounded(bar0 + 8 * ((step - 2) & 1), (uint32_t)(((step - 2) >> 1) & 1), kWaitLimitNs, p.err, kErrScanWait);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 2 * kTuN);

    // ---- merge the four warp lists of each query, write the chunk's candidates ----
    {
        float* wls = s_ls + warp * kTuQpw * k;
        int* wli = s_li + warp * kTuQpw * k;
#pragma unroll
        for (int jj = 0; jj < kTuQpw; ++jj)
            if (lane < k) {
                wls[jj * k + lane] = lsc[jj];
                wli[jj * k + lane] = lid[jj];
            }
    }
    __syncthreads();
    if (tid < nq_here) {
        const int j = tid;
        const int base_w = 4 * (j / kTuQpw), jj = j % kTuQpw;
        float* ls0 = s_ls + (base_w * kTuQpw + jj) * k;
        int* li0 = s_li + (base_w * kTuQpw + jj) * k;
        for (int w4 = 1; w4 < 4; ++w4) {
            const float* ls = s_ls + ((base_w + w4) * kTuQpw + jj) * k;
            const int* li = s_li + ((base_w + w4) * kTuQpw + jj) * k;
            for (int e = 0; e < k; ++e) list_insert(ls0, li0, k, ls[e], li[e]);
        }
        for (int e = 0; e < k; ++e) {
            const int64_t o = ((int64_t)(q0 + j) * p.n_chunks + chunk) * p.k + e;
            p.cand_score[o] = ls0[e];
            p.cand_id[o] = li0[e];
        }
    }
}

template <int CB, bool PROD, bool LO>
static cudaError_t go_tu(const TopkParams& p, size_t smem, cudaStream_t s) {
    auto kern = topk_umma_kernel<CB, PROD, LO>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_chunks, (p.nq + kTuQ - 1) / kTuQ);
    kern<<<grid, kTuThreads, smem, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    topk_merge_kernel<<<(p.nq + 7) / 8, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_topk_umma(const TopkParams& p, int cb, int prod, int lo, cudaStream_t s) {
    if (p.ks < 16 || p.ks > 256 || p.ks % 16 || p.chunk_rows % kTuRows || p.code_stride % 16 ||
        (prod && p.sign_stride % 16) || p.k < 1 || p.k > kTopkMaxK)
        return cudaErrorNotSupported;
    // every 8-code unit the kernel reads lies inside a staged row
    if (cb * p.ks / 8 > p.code_stride || (prod && p.ks / 8 > p.sign_stride)) return cudaErrorNotSupported;
    const TuLayout L = tu_layout(p.ks, prod ? 2 : 1, p.code_stride, prod ? p.sign_stride : 0, p.k);
    if (L.total > (size_t)kTuSmemLimit) return cudaErrorNotSupported;
    if (p.nq <= 0 || p.n_chunks <= 0) return cudaSuccess;
#define TQ_TU(CBV)                                                                      \
    case CBV:                                                                           \
        if (prod) return lo ? go_tu<CBV, true, true>(p, L.total, s) : go_tu<CBV, true, false>(p, L.total, s); \
        return lo ? go_tu<CBV, false, true>(p, L.total, s) : go_tu<CBV, false, false>(p, L.total, s);
    switch (cb) {
        TQ_TU(1)
        TQ_TU(2)
        TQ_TU(3)
        TQ_TU(4)
    }
#undef TQ_TU
    return cudaErrorNotSupported;
}

}  // namespace tqk
