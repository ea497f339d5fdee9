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
// One CTA: 128 query rows (the MMA M dimension, row r in TMEM lane r) of one
// KV head against one token split. Operands:
//  * A of S (TMEM, loaded once): fp16 hi/lo limbs of q' for the key part and
//    of kappa lam_k u for the sign part (K = 128 + 128);
//  * Bs (shared memory, rebuilt per tile): token t's row holds lam_k cK[idx]
//    for the 128 coordinates, then +-gamma_t for the 128 sign bits, so that
//        S[r][t] = lam_k (<q'_r, cK[idx_t]> + kappa gamma_t <u_r, 2 z_t - 1>)
//    and the logit is n_t / lam_k * S[r][t]. The sign part's K is permuted
//    (positions 2i, 2i + 1 of each 32-bit sign word hold bits i and i + 16),
//    so that one shift and one logic op build a register of two signs; A
//    carries the same permutation;
//  * P (shared memory, written by the softmax): fp16 hi/lo limbs of
//    p * nV_t, the A operand of O += P V;
//  * V (shared memory, rebuilt per tile): lam_v cV[idx], coordinates x tokens,
//    written through stmatrix with transposition from pair-table lookups.
// All shared-memory operands use the K-major layout without swizzle of
// tcgen05.cuh (8-row core matrices of 16 bytes along K).
//
// Warp roles (320 threads): warps 0-3 run the softmax (thread = query row =
// TMEM lane), warps 4-7 de-quantize (keys: thread = token; values: stmatrix
// fragments), warp 8 issues the MMAs (one thread) and owns the TMEM
// allocation, warp 9 issues the bulk copies of each tile's cache planes into
// a 3-deep ring. Per tile T the MMA thread issues S(T + 1) as soon as the
// softmax has read S(T), then O += P(T) V(T), so the tensor pipe runs the next
// tile's scores while the softmax works. Every wait is bounded; a wait that
// runs out sets the library's error word and the CTA drains and returns.
#pragma once

#include "decode_mma.cuh"
#include "tcgen05.cuh"

namespace tqk {

constexpr int kPuStages = 3;                     // tiles of cache planes in flight
constexpr int kPuThreads = 320;                  // 10 warps
constexpr int kPuBsBytes = kPuTok * 256 * 2;     // Bs: 128 tokens x 256 fp16
constexpr int kPuVBytes = kPuTok * 128 * 2;      // V: 128 coordinates x 128 tokens fp16
constexpr int kPuPBytes = kPuRows * kPuTok * 2;  // one limb of P: 128 rows x 128 tokens fp16
constexpr uint32_t kPuColQ = 0;    // TMEM: q' hi, q' lo, kappa lam u hi, lo (64 columns each)
constexpr uint32_t kPuColS = 256;  // S: 128 columns
constexpr uint32_t kPuColO = 384;  // O: 128 columns

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

__device__ __forceinline__ void stmatrix_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(r0),
                 "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// fp16 hi/lo limbs of two floats (hi = fp16(x), lo = fp16(x - hi)), packed
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// S(T) = Q Bs(T)^T over K = 256, issued by one thread once Bs(T) is written
// and the softmax has read S(T - 1): the key part (k-steps 0..7) against the
// q' limbs, the sign part (8..15) against the kappa lam_k u limbs
__device__ __forceinline__ bool pu_issue_s(int T, uint32_t tmem, uint32_t bs_s, uint32_t bs_full, uint32_t s_empty,
                                           uint32_t s_done, uint32_t idesc, uint32_t* err) {
    if (!mbar_wait_bounded(bs_full, (uint32_t)(T & 1), kWaitLimitNs, err, kErrScanWait)) return false;
    if (T > 0 && !mbar_wait_bounded(s_empty, (uint32_t)((T - 1) & 1), kWaitLimitNs, err, kErrScanWait)) return false;
    tc_fence_after_sync();
    const uint32_t dS = tmem + kPuColS;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint64_t bd = umma_desc(bs_s + 256u * k, 128, 4096);
        const uint32_t a = tmem + kPuColQ + (k < 8 ? 0u : 128u) + 8u * (k & 7);
        umma_f16_ta(dS, a, bd, idesc, k > 0);       // hi limb
        umma_f16_ta(dS, a + 64u, bd, idesc, true);  // lo limb
    }
    umma_commit(s_done);
    return true;
}

// O += P(T) V(T) over K = 128 tokens, P in two fp16 limbs, issued by one
// thread once P(T) and V(T) are written
__device__ __forceinline__ bool pu_issue_o(int T, uint32_t tmem, uint32_t p_s, uint32_t v_s, uint32_t p_full,
                                           uint32_t v_full, uint32_t o_done, uint32_t idesc, uint32_t* err) {
    if (!mbar_wait_bounded(p_full, (uint32_t)(T & 1), kWaitLimitNs, err, kErrScanWait)) return false;
    if (!mbar_wait_bounded(v_full, (uint32_t)(T & 1), kWaitLimitNs, err, kErrScanWait)) return false;
    tc_fence_after_sync();
    const uint32_t dO = tmem + kPuColO;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint64_t bd = umma_desc(v_s + 256u * k, 128, 2048);
        umma_f16(dO, umma_desc(p_s + 256u * k, 128, 2048), bd, idesc, T > 0 || k > 0);
        umma_f16(dO, umma_desc(p_s + kPuPBytes + 256u * k, 128, 2048), bd, idesc, true);
    }
    umma_commit(o_done);
    return true;
}

template <int KB, int VB, int KB2, int VB2>
__global__ void __launch_bounds__(kPuThreads, 1) prefill_umma_kernel(const __grid_constant__ PrefillParams p) {
    using ST = PuStage<KB, VB, KB2, VB2>;
    constexpr bool K2 = KB2 != KB, V2 = VB2 != VB;
    constexpr int KL = 1 << (2 * KB), VL = 1 << (2 * VB);
    constexpr int KL2 = K2 ? 1 << (2 * KB2) : 1, VL2 = V2 ? 1 << (2 * VB2) : 1;
    constexpr int D = 128;

    extern __shared__ __align__(1024) unsigned char pu_smem[];
    unsigned char* sBs = pu_smem;
    unsigned char* sV = sBs + kPuBsBytes;
    unsigned char* sP = sV + kPuVBytes;  // hi limb, then lo limb
    unsigned char* ring = sP + 2 * kPuPBytes;

    __shared__ uint32_t klut[KL];
    __shared__ uint32_t klut2[KL2];
    __shared__ uint32_t vlut[VL];
    __shared__ uint32_t vlut2[VL2];
    __shared__ __align__(8) uint64_t s_bar[3 * kPuStages + 7];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int qb = blockIdx.x, split = blockIdx.y;
    const int b = blockIdx.z / p.hkv, kv = blockIdx.z % p.hkv;
    const int G = p.group;

    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(&s_bar[0]);
    auto ring_full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto ring_empty = [&](int s) { return bar0 + 8u * (uint32_t)(kPuStages + s); };
    auto fac_full = [&](int s) { return bar0 + 8u * (uint32_t)(2 * kPuStages + s); };
    const uint32_t bs_full = bar0 + 8u * (3 * kPuStages + 0);  // Bs(T) written (4 warps)
    const uint32_t s_done = bar0 + 8u * (3 * kPuStages + 1);   // S(T) complete (commit)
    const uint32_t v_full = bar0 + 8u * (3 * kPuStages + 2);   // V(T) written (4 warps)
    const uint32_t o_done = bar0 + 8u * (3 * kPuStages + 3);   // O += P(T) V(T) complete (commit)
    const uint32_t s_empty = bar0 + 8u * (3 * kPuStages + 4);  // S(T) read by the softmax (4 warps)
    const uint32_t p_full = bar0 + 8u * (3 * kPuStages + 5);   // P(T) written, O rescaled (4 warps)
    const uint32_t q_full = bar0 + 8u * (3 * kPuStages + 6);   // A of S in TMEM (4 warps)

    for (int i = tid; i < KL; i += kPuThreads) klut[i] = p.klut[i];
    for (int i = tid; i < VL; i += kPuThreads) vlut[i] = p.vlut[i];
    if constexpr (K2)
        for (int i = tid; i < KL2; i += kPuThreads) klut2[i] = p.klut2[i];
    if constexpr (V2)
        for (int i = tid; i < VL2; i += kPuThreads) vlut2[i] = p.vlut2[i];
    if (tid == 0) {
        for (int s = 0; s < kPuStages; ++s) {
            mbar_init(ring_full(s), 1);
            mbar_init(ring_empty(s), 8);  // 4 de-quantization + 4 softmax warps
            mbar_init(fac_full(s), 4);
        }
        mbar_init(bs_full, 4);
        mbar_init(s_done, 1);
        mbar_init(v_full, 4);
        mbar_init(o_done, 1);
        mbar_init(s_empty, 4);
        mbar_init(p_full, 4);
        mbar_init(q_full, 4);
        s_abort = 0;
        mbar_init_fence();
    }
    if (warp == 8) {
        tmem_alloc((uint32_t)__cvta_generic_to_shared(&s_tmem), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;

    // ---- the CTA's tokens: rows see at most the slots before the limit of
    // its last chunk token; the split covers [t0, t0 + split_tokens) ----
    const int qs = p.q_start[b];
    const int i_last = min(p.chunk - 1, (qb * kPuRows + kPuRows - 1) / G);
    const int cta_lim = max(0, min(qs + i_last + 1, p.lim_cap));
    const int t0 = split * p.split_tokens;
    const int t_end = t0 + p.split_tokens;
    const int t1 = min(t_end, cta_lim);
    const int ntiles = t1 > t0 ? (t1 - t0 + kPuTok - 1) / kPuTok : 0;
    const int64_t rowbase = ((int64_t)b * p.hkv + kv) * p.capacity;
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
    const uint32_t bs_s = (uint32_t)__cvta_generic_to_shared(sBs);
    const uint32_t v_s = (uint32_t)__cvta_generic_to_shared(sV);
    const uint32_t p_s = (uint32_t)__cvta_generic_to_shared(sP);

    if (warp == 9) {
        // ======================= bulk copies of the cache planes =======================
        if (lane == 0 && ntiles > 0) {
            int issued = 0;
            for (int T = 0; T < ntiles; ++T) {
                const int s = T % kPuStages;
                if (T >= kPuStages && !mbar_wait_bounded(ring_empty(s), (uint32_t)((T / kPuStages - 1) & 1),
                                                         kWaitLimitNs, p.err, kErrScanWait)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const int tb = t0 + T * kPuTok;
                const uint32_t ntok = (uint32_t)((min(kPuTok, t1 - tb) + 15) & ~15);  // whole 16-slot rows
                const int64_t slot = rowbase + tb;
                const uint32_t dst = ring_s + (uint32_t)(s * ST::BYTES), bar = ring_full(s);
                fence_proxy_async_smem();  // the consumers' reads of this stage come first
                mbar_arrive_expect_tx(bar, ntok * (uint32_t)(ST::KS + 16 + 2 + 2 + ST::VS + 2));
                bulk_g2s(dst + ST::OFF_KC, p.kcodes + slot * ST::KS, ntok * ST::KS, bar);
                bulk_g2s(dst + ST::OFF_SG, p.ksigns + slot * 16, ntok * 16, bar);
                bulk_g2s(dst + ST::OFF_KN, p.knorm + slot, ntok * 2, bar);
                bulk_g2s(dst + ST::OFF_KR, p.krnorm + slot, ntok * 2, bar);
                bulk_g2s(dst + ST::OFF_VC, p.vcodes + slot * ST::VS, ntok * ST::VS, bar);
                bulk_g2s(dst + ST::OFF_VN, p.vnorm + slot, ntok * 2, bar);
                issued = T + 1;
            }
            // every copy issued lands (bounded) before the CTA's shared memory is released
            for (int T = max(0, issued - kPuStages); T < issued; ++T)
                mbar_wait_bounded(ring_full(T % kPuStages), (uint32_t)((T / kPuStages) & 1), kWaitLimitNs, p.err,
                                  kErrScanWait);
        }
    } else if (warp == 8) {
        // ======================= MMA issue (one thread) =======================
        if (lane == 0 && ntiles > 0) {
            const uint32_t idesc = umma_idesc_f16(kPuRows, kPuTok);
            uint32_t last_bar = 0, last_par = 0;
            bool ok = mbar_wait_bounded(q_full, 0, kWaitLimitNs, p.err, kErrScanWait);
            if (ok) {
                ok = pu_issue_s(0, tmem, bs_s, bs_full, s_empty, s_done, idesc, p.err);
                last_bar = s_done;
                last_par = 0;
            }
            for (int T = 0; ok && T < ntiles; ++T) {
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                // the next tile's scores go in while the softmax works on this one
                if (T + 1 < ntiles) {
                    if (!(ok = pu_issue_s(T + 1, tmem, bs_s, bs_full, s_empty, s_done, idesc, p.err))) break;
                    last_bar = s_done;
                    last_par = (uint32_t)((T + 1) & 1);
                }
                if (!(ok = pu_issue_o(T, tmem, p_s, v_s, p_full, v_full, o_done, idesc, p.err))) break;
                last_bar = o_done;
                last_par = (uint32_t)(T & 1);
            }
            if (!ok) *abort_flag = 1;
            // the MMAs in flight complete (bounded) before TMEM is released:
            // the last commit covers every MMA issued before it
            if (last_bar != 0) mbar_wait_bounded(last_bar, last_par, kWaitLimitNs, p.err, kErrScanWait);
        }
    } else if (warp >= 4) {
        // ======================= de-quantization =======================
        const int dw = warp - 4;
        const int tau = 32 * dw + lane;  // the token whose Bs row this thread writes
        const float kfac = p.inv_lam_k * p.scale_log2;
        constexpr int KW = ST::KS / 4, VW = ST::VS / 4;
        const int q = lane & 3;  // value fragment: coordinates 2q, 2q + 1 of each 8-coordinate block
        for (int T = 0; T < ntiles; ++T) {
            if (*abort_flag) break;
            const int s = T % kPuStages;
            if (!__all_sync(TQ_FULL_MASK, mbar_wait_bounded(ring_full(s), (uint32_t)((T / kPuStages) & 1),
                                                            kWaitLimitNs, p.err, kErrScanWait))) {
                *abort_flag = 1;
                break;
            }
            unsigned char* st = ring + s * ST::BYTES;
            const int tb = t0 + T * kPuTok;
            const int nval = min(kPuTok, t1 - tb);  // tokens of this tile inside the split
            const bool valid = tau < nval;
            {
                const float kn = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(st + ST::OFF_KN)[tau]);
                const float vn = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(st + ST::OFF_VN)[tau]);
                reinterpret_cast<float*>(st + ST::OFF_FK)[tau] = valid ? kn * kfac : 0.0f;
                reinterpret_cast<float*>(st + ST::OFF_FV)[tau] = valid ? vn : 0.0f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(fac_full(s));

            // ---- Bs(T): S(T - 1) has read Bs(T - 1) ----
            if (T > 0 && !__all_sync(TQ_FULL_MASK, mbar_wait_bounded(s_done, (uint32_t)((T - 1) & 1), kWaitLimitNs,
                                                                     p.err, kErrScanWait))) {
                *abort_flag = 1;
                break;
            }
            {
                const uint32_t row = bs_s + (uint32_t)((tau >> 3) * 4096 + (tau & 7) * 16);
                uint32_t kw[KW + 1];
                const unsigned char* kr = st + ST::OFF_KC + tau * ST::KS;
                if constexpr (ST::KS % 16 == 0) {
#pragma unroll
                    for (int w = 0; w < KW / 4; ++w) {
                        const uint4 x = reinterpret_cast<const uint4*>(kr)[w];
                        kw[4 * w] = x.x; kw[4 * w + 1] = x.y; kw[4 * w + 2] = x.z; kw[4 * w + 3] = x.w;
                    }
                } else {
#pragma unroll
                    for (int w = 0; w < KW / 2; ++w) {
                        const uint2 x = reinterpret_cast<const uint2*>(kr)[w];
                        kw[2 * w] = x.x; kw[2 * w + 1] = x.y;
                    }
                }
                kw[KW] = 0u;
                // key part: chunk c holds coordinates 8c .. 8c + 7 (four pairs)
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const bool first = !K2 || (c & 1) == 0;
                    const int wd = first ? KB : KB2;
                    const uint32_t* tab = first ? klut : klut2;
                    uint32_t e[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        e[j] = valid ? lds_at<uint32_t>(tab, field4(kw, code_bit<KB, KB2>(8 * c + 2 * j), 2 * wd)) : 0u;
                    sts128(row + 128u * c, e[0], e[1], e[2], e[3]);
                }
                // sign part: positions 2i, 2i + 1 of sign word w hold bits i and
                // i + 16; a set bit is +gamma, a clear one -gamma
                const uint4 sg = *reinterpret_cast<const uint4*>(st + ST::OFF_SG + tau * 16);
                const uint32_t sw[4] = {sg.x, sg.y, sg.z, sg.w};
                const uint32_t gb = reinterpret_cast<const uint16_t*>(st + ST::OFF_KR)[tau];
                const uint32_t g2 = valid ? (gb | (gb << 16)) & 0x7FFF7FFFu : 0u;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint32_t w = sw[c >> 2];
                    uint32_t e[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int i = 4 * (c & 3) + j;
                        e[j] = g2 ^ ((~w << (15 - i)) & 0x80008000u);
                    }
                    sts128(row + 128u * (16 + c), e[0], e[1], e[2], e[3]);
                }
            }
            fence_proxy_async_smem();  // the MMA reads Bs through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(bs_full);

            // ---- V(T): O += P(T - 1) V(T - 1) has read V(T - 1) ----
            if (T > 0 && !__all_sync(TQ_FULL_MASK, mbar_wait_bounded(o_done, (uint32_t)((T - 1) & 1), kWaitLimitNs,
                                                                     p.err, kErrScanWait))) {
                *abort_flag = 1;
                break;
            }
            // stmatrix fragments: matrix m of a group = token group J (8 tokens) x
            // coordinate block b (8 coordinates); this thread holds token
            // 32 dw + 8 J + lane / 4, coordinates 8 b + 2q, 8 b + 2q + 1, and
            // lane l addresses row l % 8 of matrix l / 8 (transposed: coordinate
            // 8 b + l % 8, tokens 8 J .. 8 J + 7)
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                const int tv = 32 * dw + 8 * J + (lane >> 2);
                const bool vv = tv < nval;
                uint32_t vw[VW + 1];
                const unsigned char* vr = st + ST::OFF_VC + tv * ST::VS;
                if constexpr (ST::VS % 16 == 0) {
#pragma unroll
                    for (int w = 0; w < VW / 4; ++w) {
                        const uint4 x = reinterpret_cast<const uint4*>(vr)[w];
                        vw[4 * w] = x.x; vw[4 * w + 1] = x.y; vw[4 * w + 2] = x.z; vw[4 * w + 3] = x.w;
                    }
                } else {
#pragma unroll
                    for (int w = 0; w < VW / 2; ++w) {
                        const uint2 x = reinterpret_cast<const uint2*>(vr)[w];
                        vw[2 * w] = x.x; vw[2 * w + 1] = x.y;
                    }
                }
                vw[VW] = 0u;
#pragma unroll
                for (int bq = 0; bq < 4; ++bq) {
                    uint32_t f[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int bb = 4 * bq + m;
                        const bool first = !V2 || (bb & 1) == 0;
                        const int wd = first ? VB : VB2;
                        const int base = code_bit<VB, VB2>(8 * bb);
                        const uint32_t y = (base & 31) == 0 ? vw[base >> 5]
                                                            : __funnelshift_r(vw[base >> 5], vw[(base >> 5) + 1], base & 31);
                        const uint32_t idx = (y >> (2 * wd * q)) & ((1u << (2 * wd)) - 1u);
                        f[m] = vv ? (first ? vlut[idx] : vlut2[idx]) : 0u;
                    }
                    const uint32_t addr = v_s + (uint32_t)((4 * bq + (lane >> 3)) * 2048 + (4 * dw + J) * 128 +
                                                           (lane & 7) * 16);
                    stmatrix_x4_trans(addr, f[0], f[1], f[2], f[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(v_full);
                mbar_arrive(ring_empty(s));
            }
        }
    } else {
        // ======================= softmax: thread = query row = TMEM lane =======================
        const int r = 32 * warp + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
        // CTA row r is chunk token i = (qb * 128 + r) / G and the
        // ((qb * 128 + r) % G)-th query head of KV head kv
        const int qg = qb * kPuRows + r;
        const int ci = qg / G;
        const bool rok = ci < p.chunk;
        const int hj = kv * G + (qg - ci * G);
        const int64_t qrow =
            rok ? ((int64_t)b * p.chunk + ci) * p.hq + (p.use_table ? (int)p.head_table[hj] : hj) : -1;
        const int rlim = rok ? min(max(0, min(qs + ci + 1, p.lim_cap)), t_end) : 0;  // tokens >= rlim are masked

        // ---- A of S into TMEM: columns 0..63 hold q' (coordinates 2m, 2m + 1
        // in column m) hi, 64..127 its lo; 128..191 / 192..255 kappa lam_k u,
        // column 16 w + i holding sign rows 32 w + i and 32 w + i + 16 ----
        if (ntiles > 0) {
            const float su = p.qjl_scale / p.inv_lam_k;
            const float4* q4 = rok ? reinterpret_cast<const float4*>(p.qprime + qrow * D) : nullptr;
            const float4* u4 = rok ? reinterpret_cast<const float4*>(p.u + qrow * D) : nullptr;
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // coordinates 64 h .. 64 h + 63
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float4 a = q4 ? __ldg(q4 + 16 * h + k) : make_float4(0.f, 0.f, 0.f, 0.f);
                    split2(a.x, a.y, hi[2 * k], lo[2 * k]);
                    split2(a.z, a.w, hi[2 * k + 1], lo[2 * k + 1]);
                }
                tmem_st32(lane_base + kPuColQ + 32u * h, hi);
                tmem_st32(lane_base + kPuColQ + 64u + 32u * h, lo);
#pragma unroll
                for (int w2 = 0; w2 < 2; ++w2) {  // sign word 2 h + w2: rows 32 w .. 32 w + 31
                    float uu[32];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 a = u4 ? __ldg(u4 + 16 * h + 8 * w2 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
                        uu[4 * k] = a.x * su; uu[4 * k + 1] = a.y * su; uu[4 * k + 2] = a.z * su; uu[4 * k + 3] = a.w * su;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) split2(uu[i], uu[i + 16], hi[16 * w2 + i], lo[16 * w2 + i]);
                }
                tmem_st32(lane_base + kPuColQ + 128u + 32u * h, hi);
                tmem_st32(lane_base + kPuColQ + 192u + 32u * h, lo);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        }

        float M = -INFINITY, Z = 0.0f;
        bool ok = true;
        int T = 0;
        for (; T < ntiles; ++T) {
            if (*abort_flag) {
                ok = false;
                break;
            }
            const int s = T % kPuStages;
            bool w_ok = mbar_wait_bounded(fac_full(s), (uint32_t)((T / kPuStages) & 1), kWaitLimitNs, p.err, kErrScanWait);
            w_ok = w_ok && mbar_wait_bounded(s_done, (uint32_t)(T & 1), kWaitLimitNs, p.err, kErrScanWait);
            if (!__all_sync(TQ_FULL_MASK, w_ok)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            float l[kPuTok];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t x[32];
                tmem_ld32(lane_base + kPuColS + 32u * h, x);
#pragma unroll
                for (int k = 0; k < 32; ++k) l[32 * h + k] = __uint_as_float(x[k]);
            }
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_empty);  // S may be overwritten by the next tile's scores

            const unsigned char* st = ring + s * ST::BYTES;
            const float4* fk = reinterpret_cast<const float4*>(st + ST::OFF_FK);
            const float4* fv = reinterpret_cast<const float4*>(st + ST::OFF_FV);
            // logits in log2 units: S * n_t / lam_k * scale * log2 e
#pragma unroll
            for (int k = 0; k < kPuTok / 4; ++k) {
                const float4 f = fk[k];
                l[4 * k] *= f.x; l[4 * k + 1] *= f.y; l[4 * k + 2] *= f.z; l[4 * k + 3] *= f.w;
            }
            const int rl = rlim - (t0 + T * kPuTok);  // columns >= rl are masked
            if (!__all_sync(TQ_FULL_MASK, rl >= kPuTok)) {
#pragma unroll
                for (int k = 0; k < kPuTok; ++k) l[k] = k < rl ? l[k] : -INFINITY;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < kPuTok; ++k) mx = fmaxf(mx, l[k]);
            const float mn = fmaxf(M, mx);
            // nothing seen yet: no rescale; first finite maximum: the (zero) sums scale by 0
            const float corr = mn == -INFINITY ? 1.0f : ex2(M - mn);
            const float mu = mn == -INFINITY ? 0.0f : mn;
            float zs = 0.0f;
#pragma unroll
            for (int k = 0; k < kPuTok; ++k) {
                l[k] = ex2(l[k] - mu);  // masked columns: 2^-inf = 0
                zs += l[k];
            }
            Z = fmaf(Z, corr, zs);
            M = mn;

            // P(T) and the rescale of O wait for O += P(T - 1) V(T - 1)
            if (T > 0) {
                if (!__all_sync(TQ_FULL_MASK, mbar_wait_bounded(o_done, (uint32_t)((T - 1) & 1), kWaitLimitNs, p.err,
                                                                kErrScanWait))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
            }
            // P = p * nV_t as fp16 hi/lo limbs, row r of the K-major A operand
            const uint32_t prow = p_s + (uint32_t)((r >> 3) * 2048 + (r & 7) * 16);
#pragma unroll
            for (int kc = 0; kc < kPuTok / 8; ++kc) {
                const float4 v0 = fv[2 * kc], v1 = fv[2 * kc + 1];
                uint32_t h[4], o[4];
                split2(l[8 * kc] * v0.x, l[8 * kc + 1] * v0.y, h[0], o[0]);
                split2(l[8 * kc + 2] * v0.z, l[8 * kc + 3] * v0.w, h[1], o[1]);
                split2(l[8 * kc + 4] * v1.x, l[8 * kc + 5] * v1.y, h[2], o[2]);
                split2(l[8 * kc + 6] * v1.z, l[8 * kc + 7] * v1.w, h[3], o[3]);
                sts128(prow + 128u * kc, h[0], h[1], h[2], h[3]);
                sts128(prow + kPuPBytes + 128u * kc, o[0], o[1], o[2], o[3]);
            }
            // the running maximum of a row rarely moves after the first tiles:
            // rescale O only when it moved for some row of the warp
            if (T > 0 && __any_sync(TQ_FULL_MASK, corr != 1.0f)) {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t x[32];
                    tmem_ld32(lane_base + kPuColO + 32u * h, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) x[k] = __float_as_uint(__uint_as_float(x[k]) * corr);
                    tmem_st32(lane_base + kPuColO + 32u * h, x);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();  // the MMA reads P through the async proxy
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(p_full);
                mbar_arrive(ring_empty(s));
            }
        }
        if (!ok) *abort_flag = 1;
        asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

        // ---- this split's partials of row r: a (rotated domain), M and Z ----
        if (ok && ntiles > 0) {
            ok = __all_sync(TQ_FULL_MASK, mbar_wait_bounded(o_done, (uint32_t)((ntiles - 1) & 1), kWaitLimitNs, p.err,
                                                           kErrScanWait));
            tc_fence_after_sync();
        }
        float* out = qrow >= 0 ? p.partial + (qrow * p.n_splits + split) * (D + kPartPad) : nullptr;
        const float inv_lv = p.inv_lam_v;
        if (ok && ntiles > 0) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t x[32];
                tmem_ld32(lane_base + kPuColO + 32u * h, x);
                tmem_ld_wait();
                if (out) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        reinterpret_cast<float4*>(out + 32 * h)[k] =
                            make_float4(__uint_as_float(x[4 * k]) * inv_lv, __uint_as_float(x[4 * k + 1]) * inv_lv,
                                        __uint_as_float(x[4 * k + 2]) * inv_lv, __uint_as_float(x[4 * k + 3]) * inv_lv);
                }
            }
        } else if (out) {
#pragma unroll
            for (int k = 0; k < D / 4; ++k) reinterpret_cast<float4*>(out)[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (out) {
            out[D] = M;
            out[D + 1] = Z;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

template <int KB, int VB, int KB2, int VB2>
constexpr size_t prefill_umma_smem() {
    return (size_t)kPuBsBytes + kPuVBytes + 2 * (size_t)kPuPBytes +
           (size_t)kPuStages * PuStage<KB, VB, KB2, VB2>::BYTES;
}

template <int KB, int VB, int KB2, int VB2>
cudaError_t launch_prefill_umma_t(const PrefillParams& p, cudaStream_t s) {
    auto kern = prefill_umma_kernel<KB, VB, KB2, VB2>;
    constexpr size_t smem = prefill_umma_smem<KB, VB, KB2, VB2>();
    static_assert(smem <= 227 * 1024 - 4096, "prefill tile buffers exceed shared memory");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned qbs = (unsigned)((p.chunk * p.group + kPuRows - 1) / kPuRows);
    dim3 grid(qbs, (unsigned)p.n_splits, (unsigned)(p.batch * p.hkv));
    kern<<<grid, kPuThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tqk
