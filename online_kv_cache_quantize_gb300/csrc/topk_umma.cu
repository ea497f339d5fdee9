// Inner-product search on the 5th-generation tensor cores (tcgen05).
//
// Same scores as topk.cuh (A2A TurboQuant explainer, "Benchmarks and
// real-world performance" and "Applications"; the decode logit estimator
// l = n (<q', c[idx]> + sqrt(pi/2)/m * gamma <u, 2z - 1>) per database row),
// computed as a dense contraction: for a tile of 128 database rows and a
// block of 64 queries,
//     D[row][2j + s] = sum_i A[row][i] B[2j + s][i]
// with A the de-quantized rows (lam * centroid as fp16, from a pair table;
// the fp16 residual of lam * centroid as a second table when the codebook
// has 8 or more cells; gamma * (2z - 1) for the sign part) and B the queries
// split into fp16 hi (s = 0) and lo (s = 1) halves (q' against the centroid
// parts, lam * kappa * u against the sign part). The score is
// n * (D[row][2j] + D[row][2j + 1]) / lam.
//
// Warp-specialised CTA (64 queries, a chunk of database rows, 128-row tiles):
//  * copy warp: bulk copies of each tile's packed codes and signs into a
//    ring of staging buffers;
//  * MMA warp: the MMAs (tcgen05.mma, A read from tensor memory, B = the
//    queries resident in shared memory) into one of two 128 x 128 fp32 TMEM
//    accumulators, committed to mbarriers (kept free of other work, since
//    its thread waits while the tensor core takes each MMA);
//  * 8 producer warps: de-quantize each A segment of a tile straight into
//    tensor memory (tcgen05.st; row r in TMEM lane r, two fp16 per column)
//    through a ring of segment slots, so the de-quantized tile never touches
//    shared memory;
//  * 16 epilogue warps: read a finished accumulator (tcgen05.ld) and keep
//    per-warp top-k lists of their rows (in shared memory, with the k-th
//    score of each in registers as the admission threshold), merged per
//    query at the end of the chunk into its candidates.
// The roles hand over through mbarriers (full / empty pairs); every wait is
// bounded, and a wait that runs out stops the CTA after draining what it has
// in flight.
#include "pipeline.cuh"
#include "tcgen05.cuh"
#include "topk.cuh"

namespace tqk {

constexpr int kTuRows = 128;            // database rows per tile (MMA M, TMEM lanes)
constexpr int kTuQ = 64;                // queries per CTA
constexpr int kTuN = 2 * kTuQ;          // MMA N: hi and lo column per query
constexpr int kTuProd = 8;              // producer warps
constexpr int kTuEpi = 16;              // epilogue warps (4 per TMEM lane quarter)
constexpr int kTuCtl = kTuProd + kTuEpi;  // the MMA warp's index
constexpr int kTuCopy = kTuCtl + 1;       // the copy warp's index
constexpr int kTuWarps = kTuCopy + 1;
constexpr int kTuThreads = 32 * kTuWarps;
constexpr int kTuQpw = kTuQ / 4;        // queries per epilogue warp (16)
constexpr int kTuStages = 4;            // staging buffers
constexpr int kTuASlots = 2;            // A segment slots in TMEM (after the two accumulators)
constexpr uint32_t kTuCols = 512;       // TMEM columns held by the CTA
constexpr int kTuSmemLimit = 227 * 1024 - 4096;  // dynamic part; static part below 4 KB
constexpr int kTuSmemMin = 116 * 1024;  // at most one CTA per SM: it holds all of TMEM

struct TuLayout {
    size_t b, st, sgn, kb, ls, li, total;
    int kcb, stage_bytes;
};

__host__ __device__ inline TuLayout tu_layout(int ks, int nseg_b, int code_stride, int sign_stride, int k) {
    TuLayout L;
    L.kcb = nseg_b * ks;
    const size_t bb = (size_t)kTuN * L.kcb * 2;
    // + 128: a half-row read may run past the last row's codes (into unused bytes)
    L.stage_bytes = (kTuRows * (code_stride + sign_stride) + 128 + 127) / 128 * 128;
    L.b = 0;
    L.st = (bb + 127) / 128 * 128;
    L.sgn = L.st + (size_t)kTuStages * L.stage_bytes;
    L.kb = L.sgn + 256 * 16;  // byte table of the codes (1- and 2-bit codes)
    L.ls = L.kb + 256 * 16;
    L.li = L.ls + (size_t)kTuEpi * kTuQpw * k * 4;
    L.total = L.li + (size_t)kTuEpi * kTuQpw * k * 4;
    return L;
}

// bits [8 * byte0, 8 * byte0 + nb) of a little-endian word array (folded to
// constants inside unrolled loops)
__device__ __forceinline__ uint32_t tu_bits(const uint32_t* w, int bit0, int nb) {
    const int W = bit0 >> 5, S = bit0 & 31;
    const uint32_t v = (S == 0) ? w[W] : __funnelshift_r(w[W], w[W + 1], S);
    return nb >= 32 ? v : (v & ((1u << nb) - 1u));
}

template <int CB, bool PROD, bool LO>
__global__ void __launch_bounds__(kTuThreads, 1) topk_umma_kernel(const __grid_constant__ TopkParams p) {
    constexpr int NSEG_A = 1 + (LO ? 1 : 0) + (PROD ? 1 : 0);
    constexpr int NSEG_B = 1 + (PROD ? 1 : 0);
    constexpr int NT = 1 << (2 * CB);
    constexpr int HW = 4 * CB;  // words of codes per half row (8 pairs of 16 codes)
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t s_stf[kTuStages], s_ste[kTuStages];  // staging full / empty
    __shared__ __align__(8) uint64_t s_af[kTuASlots], s_ae[kTuASlots];    // A slot full / empty
    __shared__ __align__(8) uint64_t s_cf[2], s_ce[2];                    // accumulator full / empty
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ uint32_t s_ktab[NT];
    __shared__ uint32_t s_klo[LO ? NT : 1];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ks = p.ks, k = p.k, d = p.d, m = p.m;
    const int cs = p.code_stride, ss = PROD ? p.sign_stride : 0;
    const TuLayout Lo = tu_layout(ks, NSEG_B, cs, ss, k);
    const int kcb = Lo.kcb;
    const int npair = ks / 16;  // pairs of 8-coordinate units per segment
    const uint32_t scols = (uint32_t)(ks / 2);  // TMEM columns per A segment
    unsigned char* sB = smem + Lo.b;
    unsigned char* const sSt0 = smem + Lo.st;
    const uint4* s_sgn = reinterpret_cast<const uint4*>(smem + Lo.sgn);
    // 1- and 2-bit codes: one code byte -> its 8 / 4 coordinates' pair-table
    // words in one lookup (16 / 8 bytes), instead of 4 / 2 lookups of pairs
    constexpr bool KBYTE = CB <= 2;
    const unsigned char* s_kb = smem + Lo.kb;
    float* s_ls = reinterpret_cast<float*>(smem + Lo.ls);  // [epilogue warp][query][k]
    int* s_li = reinterpret_cast<int*>(smem + Lo.li);

    const int chunk = blockIdx.x;
    const int q0 = blockIdx.y * kTuQ;
    const int nq_here = min(kTuQ, p.nq - q0);
    const int64_t r0 = (int64_t)chunk * p.chunk_rows;
    const int64_t r1 = min(r0 + p.chunk_rows, p.n_db);
    const int64_t ntile = r1 > r0 ? (r1 - r0 + kTuRows - 1) / kTuRows : 0;
    const float lam_kappa = p.qjl_scale / p.inv_lam;

    // ---- tables, B tile, barriers, TMEM (all threads) ----
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
    if constexpr (KBYTE)
        for (int i = tid; i < 256; i += blockDim.x) {
            if constexpr (CB == 1)
                reinterpret_cast<uint4*>(smem + Lo.kb)[i] =
                    make_uint4(p.ktab[i & 3], p.ktab[(i >> 2) & 3], p.ktab[(i >> 4) & 3], p.ktab[i >> 6]);
            else
                reinterpret_cast<uint2*>(smem + Lo.kb)[i] = make_uint2(p.ktab[i & 15], p.ktab[i >> 4]);
        }
    // B tile: row 2j + s holds query j's hi (s = 0) or lo (s = 1) fp16 half;
    // columns [0, ks) are q', [ks, 2 ks) lam * kappa * u (PROD)
    for (int e = tid; e < kTuQ * (kcb / 2); e += blockDim.x) {
        const int j = e / (kcb / 2), col = 2 * (e % (kcb / 2));
        const bool qv = j < nq_here;
        const bool sgn = col >= ks;
        const int i = sgn ? col - ks : col;
        const int lim = sgn ? m : d;
        const float* src = sgn ? p.u + (int64_t)(q0 + (qv ? j : 0)) * m : p.qprime + (int64_t)(q0 + (qv ? j : 0)) * d;
        const float sc_ = sgn ? lam_kappa : 1.0f;
        const float v0 = (qv && i < lim) ? sc_ * src[i] : 0.0f;
        const float v1 = (qv && i + 1 < lim) ? sc_ * src[i + 1] : 0.0f;
        *reinterpret_cast<uint32_t*>(sB + umma_off(2 * j, col, kcb)) = half_split(v0, 0) | (half_split(v1, 0) << 16);
        *reinterpret_cast<uint32_t*>(sB + umma_off(2 * j + 1, col, kcb)) = half_split(v0, 1) | (half_split(v1, 1) << 16);
    }
    const uint32_t stf0 = (uint32_t)__cvta_generic_to_shared(&s_stf[0]);
    const uint32_t ste0 = (uint32_t)__cvta_generic_to_shared(&s_ste[0]);
    const uint32_t af0 = (uint32_t)__cvta_generic_to_shared(&s_af[0]);
    const uint32_t ae0 = (uint32_t)__cvta_generic_to_shared(&s_ae[0]);
    const uint32_t cf0 = (uint32_t)__cvta_generic_to_shared(&s_cf[0]);
    const uint32_t ce0 = (uint32_t)__cvta_generic_to_shared(&s_ce[0]);
    if (tid == 0) {
        for (int x = 0; x < kTuStages; ++x) {
            mbar_init(stf0 + 8 * x, 1);
            mbar_init(ste0 + 8 * x, kTuProd);
        }
        for (int x = 0; x < kTuASlots; ++x) {
            mbar_init(af0 + 8 * x, kTuProd);
            mbar_init(ae0 + 8 * x, 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(cf0 + 8 * x, 1);
            mbar_init(ce0 + 8 * x, kTuEpi);
        }
        s_abort = 0;
        mbar_init_fence();
    }
    if (warp == kTuCtl) {
        tmem_alloc((uint32_t)__cvta_generic_to_shared(&s_tmem), kTuCols);
        tmem_relinquish();
    }
    fence_proxy_async_smem();  // the B tile is read by the tensor core
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;

    // staging of tile t (codes then signs of its rows) into buffer t % kTuStages
    auto stage = [&](int64_t t) {
        const int64_t t0 = r0 + t * kTuRows;
        const int rows = (int)min((int64_t)kTuRows, r1 - t0);
        const int b = (int)(t % kTuStages);
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(sSt0 + (size_t)b * Lo.stage_bytes);
        const uint32_t bar = stf0 + 8 * b;
        mbar_arrive_expect_tx(bar, (uint32_t)rows * (cs + ss));
        bulk_g2s(dst, p.codes + t0 * cs, (uint32_t)rows * cs, bar);
        if constexpr (PROD) bulk_g2s(dst + kTuRows * cs, p.signs + t0 * ss, (uint32_t)rows * ss, bar);
    };

    if (warp < kTuProd) {
        // ================= producers =================
        // thread: row r (its TMEM lane) and half h of every segment (pairs
        // 8h .. 8h + 7 of 16-code pairs; pairs >= npair are not written)
        const int r = 32 * (warp & 3) + lane;
        const int h = warp >> 2;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        uint16_t g_next = 0;
        if (PROD && ntile > 0 && r0 + r < r1) g_next = p.rnorm[r0 + r];
        for (int64_t t = 0; t < ntile; ++t) {
            const int b = (int)(t % kTuStages);
            if (!mbar_wait_bounded(stf0 + 8 * b, (uint32_t)((t / kTuStages) & 1), kWaitLimitNs, p.err, kErrScanWait)) {
                *abort_flag = 1;
                break;
            }
            const bool rvalid = r0 + t * kTuRows + r < r1;
            const unsigned char* st = sSt0 + (size_t)b * Lo.stage_bytes;
            // this thread's half row of codes (16 CB bytes) and of sign bits (16
            // bytes); a row past the end reads stale staging bytes, cleared by
            // the mask (the loads stay unconditional: a load that a branch may
            // skip is waited for where the paths merge)
            const uint32_t rmask = rvalid ? 0xFFFFFFFFu : 0u;
            uint32_t cw[HW + 1];
            {
                const uint4* src = reinterpret_cast<const uint4*>(st + (size_t)r * cs + 16 * CB * h);
#pragma unroll
                for (int q = 0; q < CB; ++q) {
                    const uint4 v = src[q];
                    cw[4 * q] = v.x & rmask;
                    cw[4 * q + 1] = v.y & rmask;
                    cw[4 * q + 2] = v.z & rmask;
                    cw[4 * q + 3] = v.w & rmask;
                }
                cw[HW] = 0u;
            }
            uint4 sgw = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (PROD) {
                const uint4 v = *reinterpret_cast<const uint4*>(st + (size_t)kTuRows * cs + (size_t)r * ss + 16 * h);
                sgw = make_uint4(v.x & rmask, v.y & rmask, v.z & rmask, v.w & rmask);
            }
            const uint16_t g16 = g_next;  // gamma of row r of this tile (fp16 bits)
            if (PROD && t + 1 < ntile && r0 + (t + 1) * kTuRows + r < r1) g_next = p.rnorm[r0 + (t + 1) * kTuRows + r];
            __syncwarp();
            if (lane == 0) mbar_arrive(ste0 + 8 * b);  // the staged rows were read into registers
            bool ok = true;
#pragma unroll
            for (int seg = 0; seg < NSEG_A; ++seg) {
                const int64_t g = t * NSEG_A + seg;
                const int x = (int)(g % kTuASlots);
                if (g >= kTuASlots &&
                    !mbar_wait_bounded(ae0 + 8 * x, (uint32_t)(((g / kTuASlots) - 1) & 1), kWaitLimitNs, p.err,
                                       kErrScanWait)) {
                    ok = false;
                    break;
                }
                const bool sign_seg = PROD && seg == NSEG_A - 1;
                const uint32_t* tab = (LO && seg == 1) ? s_klo : s_ktab;
                const uint32_t g2 = (sign_seg && rvalid) ? ((g16 | 0x8000u) | ((uint32_t)(g16 | 0x8000u) << 16)) : 0u;
                const uint32_t sb[4] = {sgw.x, sgw.y, sgw.z, sgw.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (8 * h + j >= npair) break;
                    uint32_t v[8];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int u = 2 * j + e;  // unit within the half row
                        if (sign_seg) {
                            const uint4 f = s_sgn[(sb[u >> 2] >> (8 * (u & 3))) & 0xFFu];
                            v[4 * e] = g2 ^ f.x;
                            v[4 * e + 1] = g2 ^ f.y;
                            v[4 * e + 2] = g2 ^ f.z;
                            v[4 * e + 3] = g2 ^ f.w;
                        } else if constexpr (KBYTE && CB == 1) {
                            const uint4 f = reinterpret_cast<const uint4*>(s_kb)[(cw[u >> 2] >> (8 * (u & 3))) & 0xFFu];
                            v[4 * e] = f.x;
                            v[4 * e + 1] = f.y;
                            v[4 * e + 2] = f.z;
                            v[4 * e + 3] = f.w;
                        } else if constexpr (KBYTE) {
                            const uint32_t w16 = cw[u >> 1] >> (16 * (u & 1));
                            const uint2 f0 = reinterpret_cast<const uint2*>(s_kb)[w16 & 0xFFu];
                            const uint2 f1 = reinterpret_cast<const uint2*>(s_kb)[(w16 >> 8) & 0xFFu];
                            v[4 * e] = f0.x;
                            v[4 * e + 1] = f0.y;
                            v[4 * e + 2] = f1.x;
                            v[4 * e + 3] = f1.y;
                        } else {
                            constexpr uint32_t M2 = (1u << (2 * CB)) - 1u;
                            const uint32_t bits = tu_bits(cw, 8 * CB * u, 8 * CB);
                            v[4 * e] = tab[bits & M2];
                            v[4 * e + 1] = tab[(bits >> (2 * CB)) & M2];
                            v[4 * e + 2] = tab[(bits >> (4 * CB)) & M2];
                            v[4 * e + 3] = tab[CB == 4 ? (bits >> 24) : ((bits >> (6 * CB)) & M2)];
                        }
                    }
                    tmem_st8(lane_addr + kTuN * 2u + (uint32_t)x * scols + 8u * (uint32_t)(8 * h + j), v);
                }
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(af0 + 8 * x);
            }
            if (!ok || *abort_flag) {
                *abort_flag = 1;
                break;
            }
        }
    } else if (warp < kTuCtl) {
        // ================= epilogue =================
        const int ew = warp - kTuProd;           // 0..15: quarter ew % 4, query group ew / 4
        const int er = 32 * (warp & 3) + lane;   // this thread's row (TMEM lane)
        const int jq0 = kTuQpw * (ew >> 2);      // its queries jq0 .. jq0 + kTuQpw - 1
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        // top-k list of each query over this warp's rows in shared memory
        // (entries best first) and, in registers, its k-th score: the
        // admission threshold
        float* const wls = s_ls + ew * kTuQpw * k;
        int* const wli = s_li + ew * kTuQpw * k;
        for (int e = lane; e < kTuQpw * k; e += 32) {
            wls[e] = -INFINITY;
            wli[e] = 0x7fffffff;
        }
        __syncwarp();
        float thr_s[kTuQpw];
#pragma unroll
        for (int jj = 0; jj < kTuQpw; ++jj) thr_s[jj] = -INFINITY;
        uint16_t n_next = 0;
        if (ntile > 0 && r0 + er < r1) n_next = p.norm[r0 + er];
        for (int64_t t = 0; t < ntile; ++t) {
            const int ab = (int)(t & 1);
            const int64_t erow = r0 + t * kTuRows + er;
            const bool evalid = erow < r1;
            const float scale = f16_bits_to_f32(n_next) * p.inv_lam;
            if (t + 1 < ntile && erow + kTuRows < r1) n_next = p.norm[erow + kTuRows];
            if (!mbar_wait_bounded(cf0 + 8 * ab, (uint32_t)((t >> 1) & 1), kWaitLimitNs, p.err, kErrScanWait)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after_sync();
            const int id = (int)erow;
            // two groups of 8 queries (16 columns) each, so that only 16
            // accumulator values are live at a time (releasing the accumulator
            // before any compute was measured slower)
#pragma unroll
            for (int hf = 0; hf < kTuQpw / 8; ++hf) {
                float v[16];
                tmem_ld16(lane_addr + (uint32_t)(ab * kTuN + 2 * jq0 + 16 * hf), v);
                tmem_ld_wait();
                if (hf == kTuQpw / 8 - 1) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ce0 + 8 * ab);  // the accumulator may be overwritten
                }
                // lane-local admission test of the 8 queries first (one compare
                // each with the list's k-th score), so that a tile where no
                // row beats any list costs one vote for the 8 queries
                float sc[8];
                uint32_t mine = 0u;
#pragma unroll
                for (int j8 = 0; j8 < 8; ++j8) {
                    const int jj = 8 * hf + j8;
                    sc[j8] = scale * (v[2 * j8] + v[2 * j8 + 1]);
                    if (evalid && jq0 + jj < nq_here && sc[j8] >= thr_s[jj]) mine |= 1u << j8;
                }
                if (!__any_sync(TQ_FULL_MASK, mine != 0u)) continue;
#pragma unroll
                for (int j8 = 0; j8 < 8; ++j8) {
                    const int jj = 8 * hf + j8;
                    unsigned cand = __ballot_sync(TQ_FULL_MASK, (mine >> j8) & 1u);
                    if (!cand) continue;
                    float* const ls = wls + jj * k;
                    int* const li = wli + jj * k;
                    while (cand) {
                        const int src = __ffs(cand) - 1;
                        cand &= cand - 1;
                        const float cs_ = __shfl_sync(TQ_FULL_MASK, sc[j8], src);
                        const int ci = __shfl_sync(TQ_FULL_MASK, id, src);
                        // lane e holds entry e; the exact rule (equal scores:
                        // lower id first) decides against the k-th entry
                        const float my = lane < k ? ls[lane] : -INFINITY;
                        const int myi = lane < k ? li[lane] : 0x7fffffff;
                        const float ts = __shfl_sync(TQ_FULL_MASK, my, k - 1);
                        const int ti = __shfl_sync(TQ_FULL_MASK, myi, k - 1);
                        if (!better(cs_, ci, ts, ti)) continue;  // the list moved on since the test
                        // entries better than the candidate stay, the rest move one slot down
                        const int pos = __popc(__ballot_sync(TQ_FULL_MASK, lane < k && better(my, myi, cs_, ci)));
                        if (lane >= pos && lane < k - 1) {
                            ls[lane + 1] = my;
                            li[lane + 1] = myi;
                        }
                        if (lane == pos) {
                            ls[lane] = cs_;
                            li[lane] = ci;
                        }
                        __syncwarp();
                    }
                    thr_s[jj] = ls[k - 1];
                }
            }
            if (*abort_flag) break;
        }
    } else if (warp == kTuCtl && lane == 0) {
        // ================= MMA issue =================
        const uint32_t idesc = umma_idesc_f16(kTuRows, kTuN);
        const uint64_t descB0 = umma_desc((uint32_t)__cvta_generic_to_shared(sB), 128, kcb * 16);
        int64_t seg_done = 0;  // segments whose MMAs were issued and committed
        bool ok = true;
        for (int64_t t = 0; t < ntile && ok; ++t) {
            const int ab = (int)(t & 1);
            // the epilogue has read this accumulator's previous tile
            if (t >= 2 && !mbar_wait_bounded(ce0 + 8 * ab, (uint32_t)(((t >> 1) - 1) & 1), kWaitLimitNs, p.err,
                                             kErrScanWait)) {
                ok = false;
                break;
            }
            const uint32_t dacc = tmem + (uint32_t)(ab * kTuN);
            for (int seg = 0; seg < NSEG_A; ++seg) {
                const int64_t g = t * NSEG_A + seg;
                const int x = (int)(g % kTuASlots);
                if (!mbar_wait_bounded(af0 + 8 * x, (uint32_t)((g / kTuASlots) & 1), kWaitLimitNs, p.err,
                                       kErrScanWait)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const int bseg = (PROD && seg == NSEG_A - 1) ? 1 : 0;
                const uint32_t a_col = tmem + kTuN * 2u + (uint32_t)x * scols;
                for (int s = 0; s < ks / 16; ++s)
                    umma_f16_ta(dacc, a_col + 8u * s, descB0 + (uint64_t)((bseg * ks / 8 + 2 * s) * 8), idesc,
                                seg > 0 || s > 0);
                umma_commit(ae0 + 8 * x);
                ++seg_done;
            }
            if (!ok) break;
            umma_commit(cf0 + 8 * ab);
            if (*abort_flag) ok = false;
        }
        if (!ok) *abort_flag = 1;
        // the MMAs in flight finish (bounded wait on the last commit) before
        // TMEM is released
        if (seg_done > 0) {
            const int64_t g = seg_done - 1;
            mbar_wait_bounded(ae0 + 8 * (int)(g % kTuASlots), (uint32_t)((g / kTuASlots) & 1), kWaitLimitNs, p.err,
                              kErrScanWait);
        }
    } else if (warp == kTuCopy && lane == 0) {
        // ================= bulk copies =================
        // tile t goes into buffer t % kTuStages once the producers released
        // it (right after reading it into registers) for tile t - kTuStages
        int64_t issued = 0;
        for (int64_t t = 0; t < ntile; ++t) {
            const int64_t prev = t - kTuStages;
            if (prev >= 0 && !mbar_wait_bounded(ste0 + 8 * (int)(prev % kTuStages), (uint32_t)((prev / kTuStages) & 1),
                                                kWaitLimitNs, p.err, kErrScanWait)) {
                *abort_flag = 1;
                break;
            }
            fence_proxy_async_smem();
            stage(t);
            issued = t + 1;
            if (*abort_flag) break;
        }
        // every copy issued has landed (bounded) before the staging buffers
        // are released: at once when the producers consumed them, and on the
        // way out of a wait that ran out
        for (int64_t t = max((int64_t)0, issued - kTuStages); t < issued; ++t)
            mbar_wait_bounded(stf0 + 8 * (int)(t % kTuStages), (uint32_t)((t / kTuStages) & 1), kWaitLimitNs, p.err,
                              kErrScanWait);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kTuCtl) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTuCols);
    }

    // ---- merge the four warp lists of each query, write the chunk's candidates ----
    if (tid < nq_here) {
        const int j = tid;
        const int qh = j / kTuQpw, jj = j % kTuQpw;  // epilogue warps 4 qh .. 4 qh + 3 hold query j
        float* ls0 = s_ls + ((4 * qh) * kTuQpw + jj) * k;
        int* li0 = s_li + ((4 * qh) * kTuQpw + jj) * k;
        for (int w4 = 1; w4 < 4; ++w4) {
            const float* ls = s_ls + ((4 * qh + w4) * kTuQpw + jj) * k;
            const int* li = s_li + ((4 * qh + w4) * kTuQpw + jj) * k;
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
    // at least kTuSmemMin: one CTA per SM, since each holds all 512 TMEM columns
    smem = smem < (size_t)kTuSmemMin ? (size_t)kTuSmemMin : smem;
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
