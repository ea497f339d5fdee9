// Chunked-prefill attention over the packed cache on the 5th-generation
// tensor cores (tcgen05.mma kind::f16, fp32 accumulators in TMEM).
//
// The same logit estimator and value sum as the decode scan (A2A TurboQuant
// explainer, end of "Stage 2": scores straight from the stored indices with
// the query rotated once; Qiita TurboQuant article, "One more stage ...":
// the residual sign term), for the C tokens x G query heads of a chunk
// against the cache, causal (query i of the chunk sees the slots 0 ..
// q_start + i), FlashAttention style: per 128-token tile an S = Q Bs^T
// contraction into TMEM, an online softmax over its rows, and O += P V
// accumulated in TMEM.
//
// Work split (stream-K): a unit is 128 query rows (the MMA M dimension, row r
// in TMEM lane r) of one KV head with all its 128-token tiles; the units'
// tiles form one sequence, and each CTA (one per SM) takes an equal run of
// it, which may start and end inside units. Each unit the run touches is a
// segment with its own query operands, softmax state and partial slot; the
// barrier phases run on across segments and the copy ring prefetches into
// the next one. Operands:
//  * A of S (loaded once): fp16 hi/lo limbs of q' for the key part and of
//    kappa lam_k u for the sign part (K = 128 + 128), the hi limbs in TMEM,
//    the lo limbs in shared memory;
//  * Bs (shared memory, rebuilt per tile): token t's row holds lam_k cK[idx]
//    for the 128 coordinates, then +-gamma_t for the 128 sign bits, so that
//        S[r][t] = lam_k (<q'_r, cK[idx_t]> + kappa gamma_t <u_r, 2 z_t - 1>)
//    and the logit is n_t / lam_k * S[r][t]. The sign part's K is permuted
//    (positions 2i, 2i + 1 of each 32-bit sign word hold bits i and i + 16),
//    so that one shift and one logic op build a register of two signs; A
//    carries the same permutation;
//  * P (TMEM, written by the softmax): fp16 hi/lo limbs of p * nV_t, the A
//    operand of O += P V, so that this contraction reads only V from shared
//    memory (with P there too it read at nearly the full shared-memory
//    bandwidth, and the de-quantization stores queued behind it);
//  * V (shared memory, rebuilt per tile): lam_v cV[idx], coordinates x tokens,
//    written through stmatrix with transposition from pair-table lookups.
// All shared-memory operands use the K-major layout without swizzle of
// tcgen05.cuh (8-row core matrices of 16 bytes along K).
//
// Warp roles (512 threads, four warps per scheduler):
//  * warps 0-7: softmax, two threads per query row (warps w and w + 4 share
//    TMEM lane quarter w and take S columns 0-63 and 64-127; they agree on
//    the row maximum of each tile through shared memory and an mbarrier);
//  * warps 8-11: Bs, thread = token;
//  * warps 12-14: V, token groups of 8 round robin, through stmatrix fragments;
//  * warp 15: one thread issues the MMAs and the bulk copies of each tile's
//    cache planes into a 3-deep ring (a stage is refilled once the softmax, Bs
//    and V warps are done with its tile); the warp owns the TMEM allocation.
// Per tile T the MMA thread issues S(T + 1) as soon as Bs(T + 1) is written
// and the softmax has read S(T), then O += P(T) V(T), so the tensor pipe runs
// the next tile's scores while the softmax works (a segment's first scores
// wait for its query operands); Bs and V are written by
// separate warps, so neither waits for the other's buffer. Every wait is
// bounded; a wait that runs out sets the library's error word and the CTA
// drains and returns.
#pragma once

#include "decode_mma.cuh"
#include "tcgen05.cuh"

namespace tqk {

constexpr int kPuStages = 3;                     // tiles of cache planes in flight
constexpr int kPuThreads = 512;                  // 16 warps
constexpr int kPuBsBytes = kPuTok * 256 * 2;     // Bs: 128 tokens x 256 fp16
constexpr int kPuVBytes = kPuTok * 128 * 2;      // V: 128 coordinates x 128 tokens fp16
constexpr int kPuQloBytes = kPuRows * 256 * 2;   // lo limbs of the A operand of S: 128 rows x 256 fp16
constexpr uint32_t kPuColQ = 0;    // TMEM: hi limbs of the A operand of S, q' then kappa lam u (64 columns each)
constexpr uint32_t kPuColS = 128;  // S: 128 columns
constexpr uint32_t kPuColO = 256;  // O: 128 columns
constexpr uint32_t kPuColP = 384;  // P: hi limb (64 columns), lo limb (64 columns)

// One ring stage: the six cache planes of 128 tokens as the bulk copies
// deliver them, then the per-token factors the de-quantization warps write
// for the softmax (n_t / lam_k * scale * log2 e, and nV_t) as floats.
template <int KB, int VB, int KB2, int VB2>
struct PuStage {
    static constexpr int KS = 8 * (KB + KB2), VS = 8 * (VB + VB2);
    static constexpr int OFF_KC = 0;
    static constexpr int OFF_SG = OFF_KC + kPuTok * KS;
    static constexpr int OFF_KN = OFF_SG + kPuTok * 16;
    static constexpr int OFF_KR = OFF_KN + kPuTok * 2;
    static constexpr int OFF_VC = OFF_KR + kPuTok * 2;
    static constexpr int OFF_VN = OFF_VC + kPuTok * VS;
    static constexpr int OFF_FK = OFF_VN + kPuTok * 2;
    static constexpr int OFF_FV = OFF_FK + kPuTok * 4;
    static constexpr int BYTES = OFF_FV + kPuTok * 4;
};

// bit offset of coordinate i in a token's code row (two channel groups:
// i % 16 < 8 at B bits, the rest at B2 bits, 16 coordinates per 8 (B + B2) bits)
template <int B, int B2>
__device__ __forceinline__ constexpr int code_bit(int i) {
    return (i >> 4) * 8 * (B + B2) + ((i & 15) < 8 ? B * (i & 15) : 8 * B + B2 * ((i & 15) - 8));
}

// Stores of operand tiles that only the tensor cores read, after the
// writer's fence.proxy.async and an mbarrier arrival (both volatile asm with
// memory clobbers, which keep their order relative to these): no memory
// clobber here, so that the compiler may hoist the table lookups of later
// stores above earlier ones (shared-memory loads take hundreds of cycles
// while the tensor cores stream their operands).
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(r0),
                 "r"(r1), "r"(r2), "r"(r3));
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d));
}

// fp16 hi/lo limbs of two floats (hi = fp16(x), lo = fp16(x - hi)), packed
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Bounded wait for the warps of this kernel: between polls the waiting warp
// sleeps, so that the de-quantization warps' shared-memory lookups do not
// queue behind a stream of mbarrier polls (a suspended try_wait wakes on every
// phase any barrier of the CTA completes, which here is often). At most
// kWaitLimitNs, then the error word and false.
__device__ __forceinline__ bool pu_wait(uint32_t bar, uint32_t parity, uint32_t* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(64);
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 0 && global_ns() - t0 > kWaitLimitNs) {
            if (err) atomicOr(err, kErrScanWait);
            return false;
        }
    }
}

// S(T) = Q Bs(T)^T over K = 256, issued by one thread once Bs(T) is written
// and the softmax has read S(T - 1): the key part (k-steps 0..7) against q',
// the sign part (8..15) against kappa lam_k u; the hi limbs from TMEM, the lo
// limbs from shared memory
__device__ __forceinline__ bool pu_issue_s(int T, uint32_t tmem, uint32_t qlo_s, uint32_t bs_s, uint32_t bs_full,
                                           uint32_t s_empty, uint32_t s_done, uint32_t idesc, uint32_t* err) {
    if (!pu_wait(bs_full, (uint32_t)(T & 1), err)) return false;
    if (T > 0 && !pu_wait(s_empty, (uint32_t)((T - 1) & 1), err)) return false;
    tc_fence_after_sync();
    const uint32_t dS = tmem + kPuColS;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint64_t bd = umma_desc(bs_s + 256u * k, 128, 4096);
        umma_f16_ta(dS, tmem + kPuColQ + 8u * k, bd, idesc, k > 0);           // hi limb
        umma_f16(dS, umma_desc(qlo_s + 256u * k, 128, 4096), bd, idesc, true);  // lo limb
    }
    umma_commit(s_done);
    return true;
}

// O += P(T) V(T) over K = 128 tokens, P in two fp16 limbs in TMEM, issued
// by one thread once P(T) and V(T) are written (T counts the CTA's tiles;
// first: the segment's first tile, which starts O afresh)
__device__ __forceinline__ bool pu_issue_o(int T, bool first, uint32_t tmem, uint32_t v_s, uint32_t p_full,
                                           uint32_t v_full, uint32_t o_done, uint32_t idesc, uint32_t* err) {
    if (!pu_wait(p_full, (uint32_t)(T & 1), err)) return false;
    if (!pu_wait(v_full, (uint32_t)(T & 1), err)) return false;
    tc_fence_after_sync();
    const uint32_t dO = tmem + kPuColO;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint64_t bd = umma_desc(v_s + 256u * k, 128, 2048);
        umma_f16_ta(dO, tmem + kPuColP + 8u * k, bd, idesc, !first || k > 0);
        umma_f16_ta(dO, tmem + kPuColP + 64u + 8u * k, bd, idesc, true);
    }
    umma_commit(o_done);
    return true;
}

// One unit's share of a CTA's tile range (stream-K): query block qb of KV
// head kv of batch row b, tokens [t0, t_end) of its sequence, visible up to
// t1 (the causal limit of the block's last chunk token), ntiles tiles with
// visible tokens; tg0 = the CTA's tiles before this segment (the barrier
// phases run on across segments); the unit's rows' partials go to slot, and
// the unit spans nslot slots.
struct PuSeg {
    int qb, b, kv;
    int t0, t_end, t1;
    int ntiles, tg0, slot, nslot;
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

template <int KB, int VB, int KB2, int VB2>
__global__ void __launch_bounds__(kPuThreads, 1) prefill_umma_kernel(const __grid_constant__ PrefillParams p) {
    using ST = PuStage<KB, VB, KB2, VB2>;
    constexpr bool K2 = KB2 != KB, V2 = VB2 != VB;
    constexpr int KL = 1 << (2 * KB), VL = 1 << (2 * VB);
    constexpr int KL2 = K2 ? 1 << (2 * KB2) : 1, VL2 = V2 ? 1 << (2 * VB2) : 1;
    constexpr int D = 128;

    extern __shared__ __align__(1024) unsigned char pu_smem[];
    unsigned char* sQlo = pu_smem;
    unsigned char* sBs = sQlo + kPuQloBytes;
    unsigned char* sV = sBs + kPuBsBytes;
    unsigned char* ring = sV + kPuVBytes;

    __shared__ uint32_t klut[KL];
    __shared__ uint32_t klut2[KL2];
    // 2-bit keys at one width: four codes (one byte of the row) per lookup,
    // entry x = the pair entries of its low and high nibbles
    constexpr bool KQ = KB == 2 && !K2;
    __shared__ __align__(8) uint2 kquad[KQ ? 256 : 1];
    __shared__ uint32_t vlut[VL];
    __shared__ uint32_t vlut2[VL2];
    __shared__ float s_xv[2][2][kPuRows];  // softmax pair exchange: [slot][column half][row]
    __shared__ int s_xok[2][2][kPuRows];
    __shared__ __align__(8) uint64_t s_bar[3 * kPuStages + 7 + 4];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ PuSeg s_seg[kPuMaxSeg];
    __shared__ int s_nseg, s_ntot;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.group;

    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(&s_bar[0]);
    auto ring_full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto ring_empty = [&](int s) { return bar0 + 8u * (uint32_t)(kPuStages + s); };
    auto fac_full = [&](int s) { return bar0 + 8u * (uint32_t)(2 * kPuStages + s); };
    const uint32_t bs_full = bar0 + 8u * (3 * kPuStages + 0);  // Bs(T) written (2 warps)
    const uint32_t s_done = bar0 + 8u * (3 * kPuStages + 1);   // S(T) complete (commit)
    const uint32_t v_full = bar0 + 8u * (3 * kPuStages + 2);   // V(T) written (2 warps)
    const uint32_t o_done = bar0 + 8u * (3 * kPuStages + 3);   // O += P(T) V(T) complete (commit)
    const uint32_t s_empty = bar0 + 8u * (3 * kPuStages + 4);  // S(T) read by the softmax (8 warps)
    const uint32_t p_full = bar0 + 8u * (3 * kPuStages + 5);   // P(T) written, O rescaled (8 warps)
    const uint32_t q_full = bar0 + 8u * (3 * kPuStages + 6);   // A of S in TMEM (8 warps)
    auto pair_bar = [&](int quarter) { return bar0 + 8u * (uint32_t)(3 * kPuStages + 7 + quarter); };  // 2 warps

    for (int i = tid; i < KL; i += kPuThreads) klut[i] = p.klut[i];
    if constexpr (KQ)
        for (int i = tid; i < 256; i += kPuThreads) kquad[i] = make_uint2(p.klut[i & 15], p.klut[i >> 4]);
    for (int i = tid; i < VL; i += kPuThreads) vlut[i] = p.vlut[i];
    if constexpr (K2)
        for (int i = tid; i < KL2; i += kPuThreads) klut2[i] = p.klut2[i];
    if constexpr (V2)
        for (int i = tid; i < VL2; i += kPuThreads) vlut2[i] = p.vlut2[i];
    if (tid == 0) {
        for (int s = 0; s < kPuStages; ++s) {
            mbar_init(ring_full(s), 1);
            mbar_init(ring_empty(s), 15);  // 4 Bs + 3 V + 8 softmax warps
            mbar_init(fac_full(s), 4);
        }
        mbar_init(bs_full, 4);
        mbar_init(s_done, 1);
        mbar_init(v_full, 3);
        mbar_init(o_done, 1);
        mbar_init(s_empty, 8);
        mbar_init(p_full, 8);
        mbar_init(q_full, 8);
        for (int i = 0; i < 4; ++i) mbar_init(pair_bar(i), 2);
        s_abort = 0;
        mbar_init_fence();
        // this CTA's segments: tiles [g0, g1) of the (unit, tile) sequence
        const int64_t total = (int64_t)p.qbs * p.batch * p.hkv * p.unit_tiles;
        const int64_t g0 = (int64_t)blockIdx.x * p.tiles_per_cta;
        const int64_t g1 = min(g0 + p.tiles_per_cta, total);
        int n = 0, tg = 0;
        int64_t g = g0;
        for (; g < g1 && n < kPuMaxSeg; ++n) {
            const int64_t u = g / p.unit_tiles;
            const int a = (int)(g - u * p.unit_tiles);
            const int bend = (int)min((int64_t)p.unit_tiles, a + (g1 - g));
            PuSeg sg;
            sg.qb = (int)(u % p.qbs);
            const int bkv = (int)(u / p.qbs);
            sg.b = bkv / p.hkv;
            sg.kv = bkv % p.hkv;
            // rows see at most the slots before the limit of the block's last chunk token
            const int i_last = min(p.chunk - 1, (sg.qb * kPuRows + kPuRows - 1) / G);
            const int lim = max(0, min(p.q_start[sg.b] + i_last + 1, p.lim_cap));
            sg.t0 = a * kPuTok;
            sg.t_end = bend * kPuTok;
            sg.t1 = min(sg.t_end, lim);
            sg.ntiles = sg.t1 > sg.t0 ? (sg.t1 - sg.t0 + kPuTok - 1) / kPuTok : 0;
            sg.tg0 = tg;
            const int64_t fc = (u * p.unit_tiles) / p.tiles_per_cta;
            sg.slot = (int)(blockIdx.x - fc);
            sg.nslot = (int)(((u + 1) * p.unit_tiles - 1) / p.tiles_per_cta - fc + 1);
            s_seg[n] = sg;
            tg += sg.ntiles;
            g += bend - a;
        }
        if (g < g1) {  // more units than the plan allows (the host bounds it): report, do nothing
            if (p.err) atomicOr(p.err, kErrScanWait);
            n = 0;
            tg = 0;
        }
        s_nseg = n;
        s_ntot = tg;
    }
    if (warp == 15) {
        tmem_alloc((uint32_t)__cvta_generic_to_shared(&s_tmem), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;

    const int nseg = s_nseg;      // segments of this CTA
    const int ntot = s_ntot;      // tiles over all of them
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
    const uint32_t bs_s = (uint32_t)__cvta_generic_to_shared(sBs);
    const uint32_t v_s = (uint32_t)__cvta_generic_to_shared(sV);
    const uint32_t qlo_s = (uint32_t)__cvta_generic_to_shared(sQlo);

    // the six bulk copies of the tile starting at cache slot `slot` with
    // ntok (whole 16-slot rows) to fetch into ring stage Tg % kPuStages (the
    // CTA's tile Tg)
    auto issue_copies = [&](int64_t slot, uint32_t ntok, int Tg) {  // one thread
        const int s = Tg % kPuStages;
        const uint32_t dst = ring_s + (uint32_t)(s * ST::BYTES), bar = ring_full(s);
        fence_proxy_async_smem();  // the consumers' reads of this stage come first
        mbar_arrive_expect_tx(bar, ntok * (uint32_t)(ST::KS + 16 + 2 + 2 + ST::VS + 2));
        bulk_g2s(dst + ST::OFF_KC, p.kcodes + slot * ST::KS, ntok * ST::KS, bar);
        bulk_g2s(dst + ST::OFF_SG, p.ksigns + slot * 16, ntok * 16, bar);
        bulk_g2s(dst + ST::OFF_KN, p.knorm + slot, ntok * 2, bar);
        bulk_g2s(dst + ST::OFF_KR, p.krnorm + slot, ntok * 2, bar);
        bulk_g2s(dst + ST::OFF_VC, p.vcodes + slot * ST::VS, ntok * ST::VS, bar);
        bulk_g2s(dst + ST::OFF_VN, p.vnorm + slot, ntok * 2, bar);
    };

    if (warp == 15) {
        // ======================= MMA issue and bulk copies (one thread) =======================
        if (lane == 0 && ntot > 0) {
            // the copy cursor: the next tile to fetch is tile ct of segment
            // cs (its fields cached in registers: this thread also issues the
            // MMAs, so its per-tile path stays short), the CTA's tile issued
            int cs = -1, ct = 0, cnt = 0, issued = 0, ctb = 0, ct1 = 0;
            int64_t crow = 0;
            auto next_copy = [&]() {
                while (ct >= cnt) {
                    const PuSeg& sg = s_seg[++cs];
                    ct = 0;
                    cnt = sg.ntiles;
                    ctb = sg.t0;
                    ct1 = sg.t1;
                    crow = ((int64_t)sg.b * p.hkv + sg.kv) * p.capacity;
                }
                const int tb = ctb + ct * kPuTok;
                issue_copies(crow + tb, (uint32_t)((min(kPuTok, ct1 - tb) + 15) & ~15), issued);
                ++ct;
                ++issued;
            };
            while (issued < kPuStages && issued < ntot) next_copy();
            const uint32_t idesc = umma_idesc_f16(kPuRows, kPuTok);
            uint32_t last_bar = 0, last_par = 0;
            int qn = 0;  // segments whose query operands were loaded
            bool ok = true;
            for (int si = 0; ok && si < nseg; ++si) {
                const PuSeg sg = s_seg[si];
                if (sg.ntiles == 0) continue;
                // the softmax warps loaded this segment's query operands
                if (!(ok = pu_wait(q_full, (uint32_t)(qn & 1), p.err))) break;
                ++qn;
                if (!(ok = pu_issue_s(sg.tg0, tmem, qlo_s, bs_s, bs_full, s_empty, s_done, idesc, p.err))) break;
                last_bar = s_done;
                last_par = (uint32_t)(sg.tg0 & 1);
                for (int T = 0; ok && T < sg.ntiles; ++T) {
                    const int Tg = sg.tg0 + T;
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    // the next tile's scores go in while the softmax works on this one
                    if (T + 1 < sg.ntiles) {
                        if (!(ok = pu_issue_s(Tg + 1, tmem, qlo_s, bs_s, bs_full, s_empty, s_done, idesc, p.err)))
                            break;
                        last_bar = s_done;
                        last_par = (uint32_t)((Tg + 1) & 1);
                    }
                    if (!(ok = pu_issue_o(Tg, T == 0, tmem, v_s, p_full, v_full, o_done, idesc, p.err))) break;
                    last_bar = o_done;
                    last_par = (uint32_t)(Tg & 1);
                    // tile Tg's stage is free once its softmax, Bs and V warps are
                    // done with it (just after P(Tg) and V(Tg), waited for above):
                    // refill it with tile Tg + kPuStages, possibly of a later segment
                    if (issued < ntot) {
                        if (!(ok = pu_wait(ring_empty(Tg % kPuStages), (uint32_t)((Tg / kPuStages) & 1), p.err)))
                            break;
                        next_copy();
                    }
                }
            }
            if (!ok) *abort_flag = 1;
            // the MMAs in flight complete (bounded) before TMEM is released:
            // the last commit covers every MMA issued before it; every copy
            // issued lands (bounded) before the shared memory is released
            if (last_bar != 0) pu_wait(last_bar, last_par, p.err);
            for (int T = max(0, issued - kPuStages); T < issued; ++T)
                pu_wait(ring_full(T % kPuStages), (uint32_t)((T / kPuStages) & 1), p.err);
        }
    } else if (warp >= 12) {
        // ======================= V: values through stmatrix =======================
        // warp vw writes the token groups J = vw, vw + 3, ... (8 tokens each,
        // 16 groups). Fragments: matrix m of a stmatrix = token group J x
        // coordinate block b (8 coordinates); this thread holds token 8 J +
        // lane / 4 at coordinates 8 b + 2q, 8 b + 2q + 1, and lane l addresses
        // row l % 8 of matrix l / 8, which after the transposition is
        // coordinate 8 b + l % 8 over tokens 8 J .. 8 J + 7 (one 16-byte row of
        // the K-major B operand).
        const int vw = warp - 12;
        const int q = lane & 3;
        constexpr int VW = ST::VS / 4;
        // T: the CTA's tile count over all its segments (the values need no
        // per-segment state)
        for (int T = 0; T < ntot; ++T) {
            const int s = T % kPuStages;
            bool ok = !*abort_flag && pu_wait(ring_full(s), (uint32_t)((T / kPuStages) & 1), p.err);
            // O += P(T - 1) V(T - 1) has read V(T - 1)
            if (ok && T > 0)
                ok = pu_wait(o_done, (uint32_t)((T - 1) & 1), p.err);
            if (!__all_sync(TQ_FULL_MASK, ok)) {
                *abort_flag = 1;
                break;
            }
            const unsigned char* st = ring + s * ST::BYTES;
            // the code words of this thread's token in group J (the next
            // group's are loaded while this one's lookups are in flight)
            auto load_row = [&](int J, uint32_t (&w)[VW + 1]) {
                const unsigned char* vr = st + ST::OFF_VC + (8 * J + (lane >> 2)) * ST::VS;
                if constexpr (ST::VS % 16 == 0) {
#pragma unroll
                    for (int i = 0; i < VW / 4; ++i) {
                        const uint4 x = reinterpret_cast<const uint4*>(vr)[i];
                        w[4 * i] = x.x; w[4 * i + 1] = x.y; w[4 * i + 2] = x.z; w[4 * i + 3] = x.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < VW / 2; ++i) {
                        const uint2 x = reinterpret_cast<const uint2*>(vr)[i];
                        w[2 * i] = x.x; w[2 * i + 1] = x.y;
                    }
                }
                w[VW] = 0u;
            };
            // one token group: 16 lookups, then the next group's row loads,
            // then the four stmatrix stores (a rolled loop over pairs of
            // groups keeps the code in the instruction cache)
            auto group = [&](int J, const uint32_t (&w)[VW + 1], uint32_t (&wn)[VW + 1]) {
                // Tokens past the split end (stale staging bytes) still index
                // inside the table, so their values are finite centroids; their
                // P is exactly 0, so they add nothing, and no mask is needed.
                // The loads are unconditional: a load that a branch may skip is
                // waited for where the paths merge.
                uint32_t f[16];
#pragma unroll
                for (int bb = 0; bb < 16; ++bb) {
                    const bool first = !V2 || (bb & 1) == 0;
                    const int wd = first ? VB : VB2;
                    const int base = code_bit<VB, VB2>(8 * bb);
                    uint32_t off;
                    if (8 * wd + 2 <= 32 && base >= 2) {
                        // the window starts 2 bits early, so the field lands
                        // pre-scaled to a byte offset (the 2 low bits masked off)
                        const int b2 = base - 2;
                        const uint32_t y2 = (b2 & 31) == 0 ? w[b2 >> 5]
                                                           : __funnelshift_r(w[b2 >> 5], w[(b2 >> 5) + 1], b2 & 31);
                        off = (y2 >> (2 * wd * q)) & (((1u << (2 * wd)) - 1u) << 2);
                    } else {
                        const uint32_t y = (base & 31) == 0 ? w[base >> 5]
                                                            : __funnelshift_r(w[base >> 5], w[(base >> 5) + 1], base & 31);
                        off = ((y >> (2 * wd * q)) & ((1u << (2 * wd)) - 1u)) << 2;
                    }
                    f[bb] = lds_at<uint32_t>(first ? vlut : vlut2, off);
                }
                if (J + 3 < 16) load_row(J + 3, wn);
                const uint32_t rowaddr = v_s + (uint32_t)((lane >> 3) * 2048 + J * 128 + (lane & 7) * 16);
#pragma unroll
                for (int bq = 0; bq < 4; ++bq)
                    stmatrix_x4_trans(rowaddr + (uint32_t)(4 * bq * 2048), f[4 * bq], f[4 * bq + 1], f[4 * bq + 2],
                                      f[4 * bq + 3]);
            };
            uint32_t wa[VW + 1], wb[VW + 1];
            load_row(vw, wa);
            int J = vw;
#pragma unroll 1
            for (; J + 3 < 16; J += 6) {
                group(J, wa, wb);
                group(J + 3, wb, wa);
            }
            if (J < 16) group(J, wa, wb);
            fence_proxy_async_smem();  // the MMA reads V through the async proxy
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(v_full);
                mbar_arrive(ring_empty(s));
            }
        }
    } else if (warp >= 8) {
        // ======================= Bs: keys and signs, thread = token =======================
        const int tau = 32 * (warp - 8) + lane;
        const float kfac = p.inv_lam_k * p.scale_log2;
        constexpr int KW = ST::KS / 4;
        // T: the CTA's tile count; the segment cursor (si, Tl) gives the
        // tile's tokens (the segment's fields cached in registers)
        int si = -1, Tl = 0, snt = 0, st0 = 0, st1 = 0;
        for (int T = 0; T < ntot; ++T, ++Tl) {
            while (Tl >= snt) {
                const PuSeg& sg = s_seg[++si];
                Tl = 0;
                snt = sg.ntiles;
                st0 = sg.t0;
                st1 = sg.t1;
            }
            const int s = T % kPuStages;
            bool ok = !*abort_flag && pu_wait(ring_full(s), (uint32_t)((T / kPuStages) & 1), p.err);
            if (!__all_sync(TQ_FULL_MASK, ok)) {
                *abort_flag = 1;
                break;
            }
            unsigned char* st = ring + s * ST::BYTES;
            const int nval = min(kPuTok, st1 - (st0 + Tl * kPuTok));
            {  // the softmax's per-token factors
                const bool valid = tau < nval;
                const float kn = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(st + ST::OFF_KN)[tau]);
                const float vn = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(st + ST::OFF_VN)[tau]);
                reinterpret_cast<float*>(st + ST::OFF_FK)[tau] = valid ? kn * kfac : 0.0f;
                reinterpret_cast<float*>(st + ST::OFF_FV)[tau] = valid ? vn : 0.0f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(fac_full(s));
            // S(T - 1) has read Bs(T - 1)
            if (T > 0 && !__all_sync(TQ_FULL_MASK, pu_wait(s_done, (uint32_t)((T - 1) & 1), p.err))) {
                *abort_flag = 1;
                break;
            }
            {
                // a token past the split end gets finite key values and signs
                // of stale gamma bits: its logits are masked (a select, not
                // arithmetic) before the softmax uses them, so no mask here
                const uint32_t row = bs_s + (uint32_t)((tau >> 3) * 4096 + (tau & 7) * 16);
                uint32_t kw[KW + 1];
                const unsigned char* kr = st + ST::OFF_KC + tau * ST::KS;
                if constexpr (ST::KS % 16 == 0) {
#pragma unroll
                    for (int i = 0; i < KW / 4; ++i) {
                        const uint4 x = reinterpret_cast<const uint4*>(kr)[i];
                        kw[4 * i] = x.x; kw[4 * i + 1] = x.y; kw[4 * i + 2] = x.z; kw[4 * i + 3] = x.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < KW / 2; ++i) {
                        const uint2 x = reinterpret_cast<const uint2*>(kr)[i];
                        kw[2 * i] = x.x; kw[2 * i + 1] = x.y;
                    }
                }
                kw[KW] = 0u;
                const uint4 sg = *reinterpret_cast<const uint4*>(st + ST::OFF_SG + tau * 16);
                const uint32_t gb = reinterpret_cast<const uint16_t*>(st + ST::OFF_KR)[tau];
                // key part: chunk c holds coordinates 8c .. 8c + 7 (four pairs);
                // every lookup of the row goes out before the first store
                uint32_t x[16][4];
                if constexpr (KQ) {
                    // byte b of the row = codes 4b .. 4b + 3; chunk c = bytes 2c, 2c + 1
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int bit = 8 * (2 * c + h);
                            const uint32_t wv = kw[bit >> 5];
                            const int sh = bit & 31;
                            const uint32_t off = (sh >= 3 ? (wv >> (sh - 3)) : (wv << (3 - sh))) & 0x7F8u;
                            const uint2 e = lds_at<uint2>(kquad, off);
                            x[c][2 * h] = e.x;
                            x[c][2 * h + 1] = e.y;
                        }
                    }
                } else {
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const bool first = !K2 || (c & 1) == 0;
                    const int wd = first ? KB : KB2;
                    const uint32_t* tab = first ? klut : klut2;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        x[c][j] = lds_at<uint32_t>(tab, field4(kw, code_bit<KB, KB2>(8 * c + 2 * j), 2 * wd));
                }
                }
#pragma unroll
                for (int c = 0; c < 16; ++c) sts128(row + 128u * c, x[c][0], x[c][1], x[c][2], x[c][3]);
                // sign part: positions 2i, 2i + 1 of sign word w hold bits i and
                // i + 16; a set bit is +gamma, a clear one -gamma
                const uint32_t sw[4] = {sg.x, sg.y, sg.z, sg.w};
                const uint32_t g2 = (gb | (gb << 16)) & 0x7FFF7FFFu;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint32_t w = sw[c >> 2];
                    uint32_t y[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int i = 4 * (c & 3) + j;
                        y[j] = g2 ^ ((~w << (15 - i)) & 0x80008000u);
                    }
                    sts128(row + 128u * (16 + c), y[0], y[1], y[2], y[3]);
                }
            }
            fence_proxy_async_smem();  // the MMA reads Bs through the async proxy
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bs_full);
                mbar_arrive(ring_empty(s));
            }
        }
    } else {
        // ======================= softmax: two threads per query row =======================
        const int qd = warp & 3, hc = warp >> 2;  // TMEM lane quarter, column half
        const int r = 32 * qd + lane;             // query row = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);

        // The two threads of a row swap a value and a flag through shared
        // memory and the pair's mbarrier (one arrival per warp, one phase per
        // exchange, bounded wait). Both take every exchange and decide on the
        // two flags together, so they leave the tile loop at the same point;
        // a wait that runs out counts as a failed flag.
        int xn = 0;
        auto exchange = [&](float v, int okv, float& other, int& other_ok) {
            const int slot = xn & 1;
            s_xv[slot][hc][r] = v;
            s_xok[slot][hc][r] = okv;
            __syncwarp();
            if (lane == 0) mbar_arrive(pair_bar(qd));
            const bool got = __all_sync(TQ_FULL_MASK, pu_wait(pair_bar(qd), (uint32_t)(xn & 1), p.err));
            ++xn;
            other = s_xv[slot][hc ^ 1][r];
            other_ok = got ? s_xok[slot][hc ^ 1][r] : 0;
        };

        bool ok = true;
        for (int si = 0; ok && si < nseg; ++si) {
        const PuSeg& sg = s_seg[si];  // read from shared memory where used (registers are at the cap)
        const int ntiles = sg.ntiles, t0 = sg.t0, tgb = sg.tg0;
        // CTA row r is chunk token i = (qb * 128 + r) / G and the
        // ((qb * 128 + r) % G)-th query head of KV head kv
        const int qg = sg.qb * kPuRows + r;
        const int ci = qg / G;
        const bool rok = ci < p.chunk;
        const int hj = sg.kv * G + (qg - ci * G);
        const int64_t qrow =
            rok ? ((int64_t)sg.b * p.chunk + ci) * p.hq + (p.use_table ? (int)p.head_table[hj] : hj) : -1;
        // tokens >= rlim are masked
        const int rlim = rok ? min(max(0, min(p.q_start[sg.b] + ci + 1, p.lim_cap)), sg.t_end) : 0;

        // ---- A of S: hi limbs in TMEM (columns 0..63 q', column m holding
        // coordinates 2m, 2m + 1; 64..127 kappa lam_k u, column 64 + 16 w + i
        // holding sign rows 32 w + i and 32 w + i + 16), lo limbs in shared
        // memory at the same K positions (row r of the K-major layout); the
        // hc = 0 warps write q', the hc = 1 warps kappa lam_k u. A later
        // segment overwrites them once the last scores of the one before
        // (waited for in its tile loop) are complete ----
        if (ntiles > 0) {
            const uint32_t qrow_s = qlo_s + (uint32_t)((r >> 3) * 4096 + (r & 7) * 16);
            if (hc == 0) {
                const float4* q4 = rok ? reinterpret_cast<const float4*>(p.qprime + qrow * D) : nullptr;
#pragma unroll
                for (int h = 0; h < 4; ++h) {  // coordinates 32 h .. 32 h + 31: columns 16 h .. 16 h + 15
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 a = q4 ? __ldg(q4 + 8 * h + k) : make_float4(0.f, 0.f, 0.f, 0.f);
                        split2(a.x, a.y, hi[2 * k], lo[2 * k]);
                        split2(a.z, a.w, hi[2 * k + 1], lo[2 * k + 1]);
                    }
                    tmem_st16(lane_base + kPuColQ + 16u * h, hi);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        sts128(qrow_s + 128u * (4 * h + c), lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
                }
            } else {
                const float su = p.qjl_scale / p.inv_lam_k;
                const float4* u4 = rok ? reinterpret_cast<const float4*>(p.u + qrow * D) : nullptr;
#pragma unroll
                for (int w = 0; w < 4; ++w) {  // sign word w: columns 64 + 16 w .. + 15
                    float uu[32];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 a = u4 ? __ldg(u4 + 8 * w + k) : make_float4(0.f, 0.f, 0.f, 0.f);
                        uu[4 * k] = a.x * su; uu[4 * k + 1] = a.y * su; uu[4 * k + 2] = a.z * su; uu[4 * k + 3] = a.w * su;
                    }
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) split2(uu[i], uu[i + 16], hi[i], lo[i]);
                    tmem_st16(lane_base + kPuColQ + 64u + 16u * w, hi);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        sts128(qrow_s + 128u * (16 + 4 * w + c), lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
                }
            }
            fence_proxy_async_smem();  // the MMA reads the lo limbs through the async proxy
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        }

        float M = -INFINITY, Z = 0.0f;
        for (int T = 0; T < ntiles; ++T) {
            const int Tg = tgb + T;  // the CTA's tile count: stage and barrier phases
            const int s = Tg % kPuStages;
            bool w_ok = !*abort_flag;
            w_ok = w_ok && pu_wait(fac_full(s), (uint32_t)((Tg / kPuStages) & 1), p.err);
            w_ok = w_ok && pu_wait(s_done, (uint32_t)(Tg & 1), p.err);
            w_ok = __all_sync(TQ_FULL_MASK, w_ok);
            tc_fence_after_sync();
            // this thread's 64 columns of S (read even after a failed wait:
            // TMEM reads stay in bounds, and the values are then dropped)
            float l[64];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t x[32];
                tmem_ld32(lane_base + kPuColS + 64u * hc + 32u * h, x);
#pragma unroll
                for (int k = 0; k < 32; ++k) l[32 * h + k] = __uint_as_float(x[k]);
            }
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (w_ok && lane == 0) mbar_arrive(s_empty);  // S may take the next tile's scores

            const unsigned char* st = ring + s * ST::BYTES;
            const float2* fk = reinterpret_cast<const float2*>(st + ST::OFF_FK) + 32 * hc;
            const float2* fv = reinterpret_cast<const float2*>(st + ST::OFF_FV) + 32 * hc;
            // logits in log2 units: S * n_t / lam_k * scale * log2 e
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float2 v = __fmul2_rn(make_float2(l[2 * k], l[2 * k + 1]), fk[k]);
                l[2 * k] = v.x;
                l[2 * k + 1] = v.y;
            }
            const int rl = rlim - (t0 + T * kPuTok + 64 * hc);  // columns >= rl are masked
            if (!__all_sync(TQ_FULL_MASK, rl >= 64)) {
#pragma unroll
                for (int k = 0; k < 64; ++k) l[k] = k < rl ? l[k] : -INFINITY;
            }
            float mt[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mt[k] = fmax3(l[8 * k], l[8 * k + 1], fmax3(l[8 * k + 2], l[8 * k + 3], l[8 * k + 4]));
#pragma unroll
            for (int k = 0; k < 8; ++k) mt[k] = fmax3(mt[k], l[8 * k + 5], fmax3(l[8 * k + 6], l[8 * k + 7], mt[k]));
            float mloc = fmax3(fmax3(mt[0], mt[1], mt[2]), fmax3(mt[3], mt[4], mt[5]), fmaxf(mt[6], mt[7]));
            float mo;
            int ook;
            exchange(mloc, w_ok ? 1 : 0, mo, ook);
            if (!(w_ok && ook)) {
                ok = false;
                break;
            }
            const float mn = fmax3(M, mloc, mo);
            // nothing seen yet: no rescale; first finite maximum: the (zero) sums scale by 0
            const float corr = mn == -INFINITY ? 1.0f : ex2(M - mn);
            const float mu = mn == -INFINITY ? 0.0f : mn;
            float2 z2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float2 d = __fadd2_rn(make_float2(l[2 * k], l[2 * k + 1]), make_float2(-mu, -mu));
                l[2 * k] = ex2(d.x);  // masked columns: 2^-inf = 0
                l[2 * k + 1] = ex2(d.y);
                z2[k & 3] = __fadd2_rn(z2[k & 3], make_float2(l[2 * k], l[2 * k + 1]));
            }
            const float2 zz = __fadd2_rn(__fadd2_rn(z2[0], z2[1]), __fadd2_rn(z2[2], z2[3]));
            Z = fmaf(Z, corr, zz.x + zz.y);
            M = mn;

            // P(T) and the rescale of O wait for O += P(T - 1) V(T - 1) (the
            // previous segment's last one, for a segment's first tile)
            bool o_ok = true;
            if (Tg > 0)
                o_ok = __all_sync(TQ_FULL_MASK, pu_wait(o_done, (uint32_t)((Tg - 1) & 1), p.err));
            {
                float dummy;
                int o_ook;
                exchange(0.0f, o_ok ? 1 : 0, dummy, o_ook);
                if (!(o_ok && o_ook)) {
                    ok = false;
                    break;
                }
            }
            tc_fence_after_sync();
            // P = p * nV_t as fp16 hi/lo limbs into TMEM (the A operand of
            // O += P V): tokens 64 hc + 2j, + 1 in column 32 hc + j of each limb
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int k = 32 * h2 + 2 * j;
                    const float2 pv = __fmul2_rn(make_float2(l[k], l[k + 1]), fv[16 * h2 + j]);
                    split2(pv.x, pv.y, hi[j], lo[j]);
                }
                tmem_st16(lane_base + kPuColP + 32u * hc + 16u * h2, hi);
                tmem_st16(lane_base + kPuColP + 64u + 32u * hc + 16u * h2, lo);
            }
            // the running maximum of a row rarely moves after the first tiles:
            // rescale this thread's half of O only when it moved for some row
            // of the warp
            if (T > 0 && __any_sync(TQ_FULL_MASK, corr != 1.0f)) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t x[32];
                    const uint32_t a = lane_base + kPuColO + 64u * hc + 32u * h;
                    tmem_ld32(a, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float2 v = __fmul2_rn(make_float2(__uint_as_float(x[2 * k]), __uint_as_float(x[2 * k + 1])),
                                                    make_float2(corr, corr));
                        x[2 * k] = __float_as_uint(v.x);
                        x[2 * k + 1] = __float_as_uint(v.y);
                    }
                    tmem_st32(a, x);
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(p_full);
                mbar_arrive(ring_empty(s));
            }
        }
        if (!ok) *abort_flag = 1;
        if (si == nseg - 1) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

        // ---- this segment's partials of row r: a (rotated domain) from both
        // halves, M, and Z summed over the pair ----
        if (ok && ntiles > 0) {
            ok = __all_sync(TQ_FULL_MASK, pu_wait(o_done, (uint32_t)((tgb + ntiles - 1) & 1), p.err));
            tc_fence_after_sync();
        }
        float zo;
        int zok;
        exchange(Z, ok ? 1 : 0, zo, zok);
        ok = ok && zok;
        float* out = qrow >= 0 ? p.partial + (qrow * p.n_splits + sg.slot) * (D + kPartPad) : nullptr;
        const float inv_lv = p.inv_lam_v;
        if (ok && ntiles > 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t x[32];
                tmem_ld32(lane_base + kPuColO + 64u * hc + 32u * h, x);
                tmem_ld_wait();
                if (out) {
                    float4* o4 = reinterpret_cast<float4*>(out + 64 * hc + 32 * h);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        o4[k] = make_float4(__uint_as_float(x[4 * k]) * inv_lv, __uint_as_float(x[4 * k + 1]) * inv_lv,
                                            __uint_as_float(x[4 * k + 2]) * inv_lv, __uint_as_float(x[4 * k + 3]) * inv_lv);
                }
            }
        } else if (out) {
            float4* o4 = reinterpret_cast<float4*>(out + 64 * hc);
#pragma unroll
            for (int k = 0; k < 16; ++k) o4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (out && hc == 0) {
            out[D] = M;
            out[D + 1] = Z + zo;
        }
        // the unit's first segment also writes the slots no CTA of the unit
        // fills as empty partials (M = -inf, Z = 0, a = 0)
        if (sg.slot == 0 && qrow >= 0)
            for (int e = sg.nslot; e < p.n_splits; ++e) {
                float* oe = p.partial + (qrow * p.n_splits + e) * (D + kPartPad);
                float4* o4 = reinterpret_cast<float4*>(oe + 64 * hc);
#pragma unroll
                for (int k = 0; k < 16; ++k) o4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (hc == 0) {
                    oe[D] = -INFINITY;
                    oe[D + 1] = 0.0f;
                }
            }
        }  // segments
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 15) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

template <int KB, int VB, int KB2, int VB2>
constexpr size_t prefill_umma_smem() {
    return (size_t)kPuQloBytes + kPuBsBytes + kPuVBytes +
           (size_t)kPuStages * PuStage<KB, VB, KB2, VB2>::BYTES;
}

template <int KB, int VB, int KB2, int VB2>
cudaError_t launch_prefill_umma_t(const PrefillParams& p, cudaStream_t s) {
    auto kern = prefill_umma_kernel<KB, VB, KB2, VB2>;
    constexpr size_t smem = prefill_umma_smem<KB, VB, KB2, VB2>();
    static_assert(smem <= 227 * 1024 - 4096, "prefill tile buffers exceed shared memory");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // stream-K: ceil(units x unit_tiles / tiles_per_cta) CTAs
    const int64_t total = (int64_t)p.qbs * p.batch * p.hkv * p.unit_tiles;
    if (p.tiles_per_cta < 1 || p.unit_tiles < 1 || total < 1) return cudaErrorInvalidValue;
    const int64_t ctas = (total + p.tiles_per_cta - 1) / p.tiles_per_cta;
    if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
    kern<<<dim3((unsigned)ctas), kPuThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tqk
