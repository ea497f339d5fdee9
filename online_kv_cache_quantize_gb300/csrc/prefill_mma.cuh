// Chunked-prefill attention over the packed cache on the tensor cores
// (mma.sync m16n8k16, f16 x f16 -> f32).
//
// The same logit estimator and value sum as the decode scan (A2A TurboQuant
// explainer, end of "Stage 2"; Qiita TurboQuant article, "One more stage
// ..."), for many queries per KV head: the C tokens of a chunk x G query
// heads. Query i of the chunk (position q_start + i) sees the slots
// 0 .. q_start + i (causal), the chunk's own keys and values having been
// quantized into the cache first.
//
// Orientation: a warp owns 16 query rows (the MMA M dimension) and walks the
// token tiles of its split, FlashAttention-2 style:
//  * S = Q K^T: A[row][coord] = fp16 hi/lo splits of q' (and of kappa u for
//    the sign term), built once per CTA into shared memory in fragment order;
//    B[coord][token] = lam_k * cK[idx] straight from the 2-coordinate pair
//    table (one lookup = one B register: the pair lies along the MMA K
//    dimension), the sign term's B = +-1 from the 4-sign table. K is permuted
//    as in the decode scan (thread c of a quad holds coordinates
//    32c .. 32c+31), so a thread reads contiguous code bits.
//  * online softmax per row in registers (a row's 16 tile columns sit in one
//    quad).
//  * O += P V: the S accumulators of a 16-token tile are exactly the A
//    fragment of the next MMA (tokens along K), as fp16 hi/lo of p * nV;
//    B[token][coord] = lam_v * cV[idx] from the pair table: one lookup gives
//    two coordinates of one token and a byte permute pairs two tokens, so
//    four lookups make the B registers of two n-tiles. N is permuted so that
//    thread g reads coordinates 16g .. 16g+15 (contiguous bits): column n of
//    n-tile (j, h) is coordinate 16 n + 2 j + h.
// Tokens stream through a CTA-wide 4-deep ring of shared-memory stages (64
// tokens each, one bulk copy per cache plane, as in the decode scan); all
// four warps read every tile of a stage, and the last warp done with a stage
// refills it. Split-K over tokens; each (row, split) partial (a, M, Z) is
// merged and un-rotated by the decode merge kernel.
#pragma once

#include <type_traits>

#include "decode_mma.cuh"

namespace tqk {

// fp16 hi/lo splits of a pair (a in the low half): hi = fp16(a), lo =
// fp16(a - hi), each pair converted by one instruction; the same values as
// split_half
__device__ __forceinline__ void split_half2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 8 * field(w, off, n): the byte offset of an 8-byte table entry
__device__ __forceinline__ uint32_t field8(const uint32_t* w, int off, int n) {
    const int W = off >> 5, S = off & 31;
    const uint32_t mask = ((1u << n) - 1u) << 3;
    if (S + n <= 32) return (S >= 3 ? (w[W] >> (S - 3)) : (w[W] << (3 - S))) & mask;
    return (__funnelshift_r(w[W], w[W + 1], S) << 3) & mask;
}

constexpr int kPfWarps = 4;
constexpr int kPfStages = 4;
static_assert(kPfRows == 16 * kPfWarps, "a warp owns 16 query rows");

template <int KB, int VB, int KB2 = KB, int VB2 = VB>
__global__ void __launch_bounds__(kPfWarps * 32, 2) prefill_mma_kernel(const __grid_constant__ PrefillParams p) {
    using T = MmaTile<KB, VB, KB2, VB2>;
    constexpr bool K2 = KB2 != KB, V2 = VB2 != VB;
    constexpr int KL = 1 << (2 * KB), VL = 1 << (2 * VB);
    constexpr int KL2 = K2 ? 1 << (2 * KB2) : 1, VL2 = V2 ? 1 << (2 * VB2) : 1;
    constexpr bool KLO = KB >= 3;
    constexpr int D = 128;
    constexpr int SB = kPfWarps * T::BYTES;  // one stage: 4 tiles of 16 tokens

    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* stages = smem;
    // A fragments of the CTA's query rows: [warp][kk][part][lane], part 0 / 1 =
    // hi / lo of q', 2 / 3 = hi / lo of kappa u (four registers each)
    uint4* qf = reinterpret_cast<uint4*>(smem + kPfStages * SB);
    // key pair tables: 4-byte entries, or for 3-4 bit codes 8-byte entries
    // holding the fp16 pair and its lo residual pair
    __shared__ uint32_t klut[KLO ? 1 : KL];
    __shared__ __align__(8) uint2 klut8[KLO ? KL : 1];
    __shared__ uint32_t vlut[VL];
    __shared__ uint32_t klut2[(K2 && !KLO) ? KL2 : 1];
    __shared__ __align__(8) uint2 klut8_2[(K2 && KLO) ? KL2 : 1];
    __shared__ uint32_t vlut2[VL2];
    __shared__ __align__(8) uint2 slut4[16];
    __shared__ __align__(8) uint64_t s_bar[kPfStages];
    __shared__ uint32_t s_cnt[kPfStages];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int qb = blockIdx.x, split = blockIdx.y;
    const int b = blockIdx.z / p.hkv, kv = blockIdx.z % p.hkv;
    const int G = p.group;

    for (int i = threadIdx.x; i < KL; i += blockDim.x) {
        if constexpr (KLO) klut8[i] = make_uint2(p.klut[i], p.klut_lo[i]);
        else klut[i] = p.klut[i];
    }
    for (int i = threadIdx.x; i < VL; i += blockDim.x) vlut[i] = p.vlut[i];
    if constexpr (K2) {
        for (int i = threadIdx.x; i < KL2; i += blockDim.x) {
            if constexpr (KLO) klut8_2[i] = make_uint2(p.klut2[i], p.klut2_lo[i]);
            else klut2[i] = p.klut2[i];
        }
    }
    if constexpr (V2)
        for (int i = threadIdx.x; i < VL2; i += blockDim.x) vlut2[i] = p.vlut2[i];
    if (threadIdx.x < 16) {
        const uint32_t pos = 0x3C00u, neg = 0xBC00u, e = threadIdx.x;
        slut4[e].x = ((e & 1) ? pos : neg) | (((e & 2) ? pos : neg) << 16);
        slut4[e].y = ((e & 4) ? pos : neg) | (((e & 8) ? pos : neg) << 16);
    }
    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(&s_bar[0]);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int sb = 0; sb < kPfStages; ++sb) {
            mbar_init(bar0 + 8 * sb, 1);
            s_cnt[sb] = 0u;
        }
        mbar_init_fence();
    }

    // ---- the rows: CTA row q = qb * 64 + warp * 16 + rho is chunk token q / G
    // and the (q % G)-th query head of KV head kv; this thread's rows are
    // rho = g and g + 8 ----
    const int qs = p.q_start[b];
    int lim[2];
    int64_t qrow[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int q = qb * kPfRows + warp * 16 + g + 8 * r;
        const int i = q / G;
        const bool ok = i < p.chunk;
        const int j = kv * G + (q - i * G);
        qrow[r] = ok ? ((int64_t)b * p.chunk + i) * p.hq + (p.use_table ? (int)p.head_table[j] : j) : -1;
        lim[r] = ok ? max(0, min(qs + i + 1, p.lim_cap)) : 0;
    }
    // the CTA's last chunk token bounds the tokens any of its rows can see
    const int i_last = min(p.chunk - 1, (qb * kPfRows + kPfRows - 1) / G);
    const int cta_lim = max(0, min(qs + i_last + 1, p.lim_cap));
    const int t0 = split * p.split_tokens;
    const int t1 = min(t0 + p.split_tokens, cta_lim);
    const int ntiles = t1 > t0 ? (t1 - t0 + 15) >> 4 : 0;
    const int ngroups = (ntiles + kPfWarps - 1) / kPfWarps;
    const int64_t rowbase = ((int64_t)b * p.hkv + kv) * p.capacity;
    const uint32_t stages_s = (uint32_t)__cvta_generic_to_shared(stages);
    auto issue_group = [&](int gi) {  // one thread
        const int sb = gi % kPfStages;
        const int ntg = min(kPfWarps, ntiles - kPfWarps * gi);
        const int64_t slot = rowbase + t0 + 16 * kPfWarps * gi;
        const uint32_t dst = stages_s + sb * SB, bar = bar0 + 8 * sb;
        const uint32_t ntok = 16u * (uint32_t)ntg;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, (uint32_t)ntg * T::BYTES);
        bulk_g2s(dst + kPfWarps * T::OFF_KC, p.kcodes + slot * T::KS, ntok * T::KS, bar);
        bulk_g2s(dst + kPfWarps * T::OFF_SG, p.ksigns + slot * 16, ntok * 16, bar);
        bulk_g2s(dst + kPfWarps * T::OFF_KN, p.knorm + slot, ntok * 2, bar);
        bulk_g2s(dst + kPfWarps * T::OFF_KR, p.krnorm + slot, ntok * 2, bar);
        bulk_g2s(dst + kPfWarps * T::OFF_VC, p.vcodes + slot * T::VS, ntok * T::VS, bar);
        bulk_g2s(dst + kPfWarps * T::OFF_VN, p.vnorm + slot, ntok * 2, bar);
    };
    if (threadIdx.x == 0)
        for (int gi = 0; gi < kPfStages && gi < ngroups; ++gi) issue_group(gi);

    // ---- A fragments: thread (g, c) of k-step kk holds coordinates
    // 32c + 4kk + {0, 1} (registers 0, 1: rows g, g + 8) and + {2, 3}
    // (registers 2, 3) ----
    {
        const float* q0 = qrow[0] >= 0 ? p.qprime + qrow[0] * D : nullptr;
        const float* q1 = qrow[1] >= 0 ? p.qprime + qrow[1] * D : nullptr;
        const float* u0 = qrow[0] >= 0 ? p.u + qrow[0] * D : nullptr;
        const float* u1 = qrow[1] >= 0 ? p.u + qrow[1] * D : nullptr;
        const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        const float ks = p.qjl_scale;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int c0 = 32 * c + 4 * kk;
            const float4 a = q0 ? __ldg(reinterpret_cast<const float4*>(q0 + c0)) : z4;
            const float4 a8 = q1 ? __ldg(reinterpret_cast<const float4*>(q1 + c0)) : z4;
            float4 v = u0 ? __ldg(reinterpret_cast<const float4*>(u0 + c0)) : z4;
            float4 v8 = u1 ? __ldg(reinterpret_cast<const float4*>(u1 + c0)) : z4;
            v.x *= ks; v.y *= ks; v.z *= ks; v.w *= ks;
            v8.x *= ks; v8.y *= ks; v8.z *= ks; v8.w *= ks;
            uint4* dst = qf + (warp * 8 + kk) * 4 * 32 + lane;
#pragma unroll
            for (int lo = 0; lo < 2; ++lo) {
                dst[lo * 32] = make_uint4(split_half(a.x, lo) | (split_half(a.y, lo) << 16),
                                          split_half(a8.x, lo) | (split_half(a8.y, lo) << 16),
                                          split_half(a.z, lo) | (split_half(a.w, lo) << 16),
                                          split_half(a8.z, lo) | (split_half(a8.w, lo) << 16));
                dst[(2 + lo) * 32] = make_uint4(split_half(v.x, lo) | (split_half(v.y, lo) << 16),
                                                split_half(v8.x, lo) | (split_half(v8.y, lo) << 16),
                                                split_half(v.z, lo) | (split_half(v.w, lo) << 16),
                                                split_half(v8.z, lo) | (split_half(v8.w, lo) << 16));
            }
        }
    }
    // a tile at or past every row's limit is skipped by the whole warp
    const int wlim = __reduce_max_sync(TQ_FULL_MASK, max(lim[0], lim[1]));

    float M[2] = {-INFINITY, -INFINITY}, Zp[2] = {0.0f, 0.0f};
    float O[8][2][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < 4; ++r) O[j][h][r] = 0.0f;

    __syncthreads();  // tables, fragments, barriers
    const float inv_lk = p.inv_lam_k, inv_lv = p.inv_lam_v;
    const uint4* wq = qf + warp * 8 * 4 * 32 + lane;

    // One step over NS consecutive 16-token tiles of a stage (two, or one at
    // the end of a split): S for 8 NS tokens per A-fragment load, then the
    // online softmax, then O += P V one 16-token tile at a time.
    auto step = [&](auto ns_tag, const unsigned char* st, int tt, int tok0) {
        constexpr int NS = decltype(ns_tag)::value;
        constexpr int NT = 2 * NS;  // key n-tiles of 8 tokens; this thread's B column is token 8 nt + g
        const unsigned char* p_kc = st + kPfWarps * T::OFF_KC + tt * T::KC;
        const unsigned char* p_sg = st + kPfWarps * T::OFF_SG + tt * T::SG;
        const uint32_t* p_kn = reinterpret_cast<const uint32_t*>(st + kPfWarps * T::OFF_KN + tt * T::NB);
        const uint32_t* p_kr = reinterpret_cast<const uint32_t*>(st + kPfWarps * T::OFF_KR + tt * T::NB);
        const unsigned char* p_vc = st + kPfWarps * T::OFF_VC + tt * T::VC;
        const uint32_t* p_vn = reinterpret_cast<const uint32_t*>(st + kPfWarps * T::OFF_VN + tt * T::NB);

        // ---- S = Q K^T (+ the sign term) ----
        constexpr int KWN = (KB + KB2 + 1) / 2;
        uint32_t kw[NT][KWN + 1], sw[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int tok = 8 * nt + g;
            if constexpr (!K2) {
                const uint32_t* r = reinterpret_cast<const uint32_t*>(p_kc + tok * T::KS) + KB * c;
#pragma unroll
                for (int w = 0; w < KB; ++w) kw[nt][w] = r[w];
            } else {
                // an odd KB + KB2 starts odd c's run half way into a word
                constexpr int TW = T::KS / 4;
                const int wb = (c * (KB + KB2)) >> 1, sh = ((c * (KB + KB2)) & 1) * 16;
                const uint32_t* r = reinterpret_cast<const uint32_t*>(p_kc + tok * T::KS) + wb;
                uint32_t x[KWN + 1];
#pragma unroll
                for (int w = 0; w <= KWN; ++w) x[w] = wb + w < TW ? r[w] : 0u;
#pragma unroll
                for (int w = 0; w < KWN; ++w) kw[nt][w] = __funnelshift_r(x[w], x[w + 1], sh);
            }
            kw[nt][KWN] = 0u;
            sw[nt] = reinterpret_cast<const uint32_t*>(p_sg + tok * 16)[c];
        }
        float sk[NT][4], ss[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) sk[nt][r] = ss[nt][r] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint4 qh = wq[(kk * 4 + 0) * 32], ql = wq[(kk * 4 + 1) * 32];
            const uint4 uh = wq[(kk * 4 + 2) * 32], ul = wq[(kk * 4 + 3) * 32];
            const bool first = !K2 || (kk & 3) < 2;
            const int kw_ = first ? KB : KB2, ko = key_off<KB, KB2>(kk);
            uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if constexpr (KLO) {  // one 8-byte entry: (hi pair, lo pair)
                    const uint2* t8 = first ? klut8 : klut8_2;
                    const uint2 e0 = lds_at<uint2>(t8, field8(kw[nt], ko, 2 * kw_));
                    const uint2 e1 = lds_at<uint2>(t8, field8(kw[nt], ko + 2 * kw_, 2 * kw_));
                    bh[nt][0] = e0.x; bl[nt][0] = e0.y;
                    bh[nt][1] = e1.x; bl[nt][1] = e1.y;
                } else {
                    const uint32_t* tab = first ? klut : klut2;
                    bh[nt][0] = lds_at<uint32_t>(tab, field4(kw[nt], ko, 2 * kw_));
                    bh[nt][1] = lds_at<uint32_t>(tab, field4(kw[nt], ko + 2 * kw_, 2 * kw_));
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(sk[nt], qh.x, qh.y, qh.z, qh.w, bh[nt][0], bh[nt][1]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(sk[nt], ql.x, ql.y, ql.z, ql.w, bh[nt][0], bh[nt][1]);
            if constexpr (KLO) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma16816(sk[nt], qh.x, qh.y, qh.z, qh.w, bl[nt][0], bl[nt][1]);
            }
            uint2 sg[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                sg[nt] = lds_at<uint2>(slut4, kk == 0 ? (sw[nt] << 3) & 0x78u : (sw[nt] >> (4 * kk - 3)) & 0x78u);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(ss[nt], uh.x, uh.y, uh.z, uh.w, sg[nt].x, sg[nt].y);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(ss[nt], ul.x, ul.y, ul.z, ul.w, sg[nt].x, sg[nt].y);
        }

        // ---- logits and the online softmax: this thread's columns of n-tile
        // nt are tokens 8 nt + 2c and 8 nt + 2c + 1 ----
        float s_[NT][4];
        float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t knw = p_kn[4 * nt + c], krw = p_kr[4 * nt + c];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int hi = r & 1, row = r >> 1;
                const int tok = tok0 + 8 * nt + 2 * c + hi;
                const float kn = f16_bits_to_f32((uint16_t)(knw >> (16 * hi)));
                const float kg = f16_bits_to_f32((uint16_t)(krw >> (16 * hi)));
                const float l = kn * fmaf(kg, ss[nt][r], sk[nt][r] * inv_lk);
                s_[nt][r] = tok < lim[row] ? l * p.scale_log2 : -INFINITY;
                mt[row] = fmaxf(mt[row], s_[nt][r]);
            }
        }
        float corr[2];
#pragma unroll
        for (int row = 0; row < 2; ++row) {
            float m = mt[row];
            m = fmaxf(m, __shfl_xor_sync(TQ_FULL_MASK, m, 1));
            m = fmaxf(m, __shfl_xor_sync(TQ_FULL_MASK, m, 2));
            const float mn = fmaxf(M[row], m);
            corr[row] = (mn == -INFINITY) ? 1.0f : ex2(M[row] - mn);
            M[row] = mn;
        }
        float zs[2] = {0.0f, 0.0f};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t vnw = p_vn[4 * nt + c];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int hi = r & 1, row = r >> 1;
                const float pr = (s_[nt][r] == -INFINITY) ? 0.0f : ex2(s_[nt][r] - M[row]);
                zs[row] += pr;
                s_[nt][r] = pr * f16_bits_to_f32((uint16_t)(vnw >> (16 * hi)));  // now p * nV
            }
        }
        Zp[0] = fmaf(Zp[0], corr[0], zs[0]);
        Zp[1] = fmaf(Zp[1], corr[1], zs[1]);
        if (__any_sync(TQ_FULL_MASK, corr[0] != 1.0f || corr[1] != 1.0f)) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    O[j][h][0] *= corr[0];
                    O[j][h][1] *= corr[0];
                    O[j][h][2] *= corr[1];
                    O[j][h][3] *= corr[1];
                }
        }

        // ---- O += P V, one 16-token tile at a time ----
#pragma unroll
        for (int t16 = 0; t16 < NS; ++t16) {
            // A fragment (tokens along K): registers 0..3 = (row g, tokens 2c,
            // 2c+1), (row g+8, same), (row g, 8+2c, 9+2c), (row g+8, same)
            uint32_t ph[4], pl[4];
            split_half2(s_[2 * t16][0], s_[2 * t16][1], ph[0], pl[0]);
            split_half2(s_[2 * t16][2], s_[2 * t16][3], ph[1], pl[1]);
            split_half2(s_[2 * t16 + 1][0], s_[2 * t16 + 1][1], ph[2], pl[2]);
            split_half2(s_[2 * t16 + 1][2], s_[2 * t16 + 1][3], ph[3], pl[3]);
            // value codes of tokens 2c, 2c+1, 8+2c, 9+2c, coordinates 16g .. 16g+15
            uint32_t vf[4][3];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int tok = 16 * t16 + 2 * c + (q & 1) + 8 * (q >> 1);
                const uint32_t* vr = reinterpret_cast<const uint32_t*>(p_vc + tok * T::VS);
                const int bit0 = 8 * (VB + VB2) * g;
                const int wd = bit0 >> 5, sh = bit0 & 31;
                const uint32_t x0 = vr[wd];
                const uint32_t x1 = (wd + 1 < T::VS / 4) ? vr[wd + 1] : 0u;
                const uint32_t x2 = (wd + 2 < T::VS / 4) ? vr[wd + 2] : 0u;
                vf[q][0] = __funnelshift_r(x0, x1, sh);
                vf[q][1] = __funnelshift_r(x1, x2, sh);
                vf[q][2] = 0u;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t x[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    x[q] = (!V2 || j < 4) ? lds_at<uint32_t>(vlut, field4(vf[q], val_off<VB, VB2>(j), 2 * VB))
                                          : lds_at<uint32_t>(vlut2, field4(vf[q], val_off<VB, VB2>(j), 2 * VB2));
                const uint32_t e0 = prmt(x[0], x[1], 0x5410u), e1 = prmt(x[2], x[3], 0x5410u);  // coordinate 16g + 2j
                const uint32_t o0 = prmt(x[0], x[1], 0x7632u), o1 = prmt(x[2], x[3], 0x7632u);  // 16g + 2j + 1
                mma16816(O[j][0], ph[0], ph[1], ph[2], ph[3], e0, e1);
                mma16816(O[j][1], ph[0], ph[1], ph[2], ph[3], o0, o1);
                mma16816(O[j][0], pl[0], pl[1], pl[2], pl[3], e0, e1);
                mma16816(O[j][1], pl[0], pl[1], pl[2], pl[3], o0, o1);
            }
        }
    };

    int gi = 0;
    for (; gi < ngroups; ++gi) {
        const bool landed = mbar_wait_bounded(bar0 + 8 * (gi % kPfStages), (gi / kPfStages) & 1, kWaitLimitNs,
                                              p.err, kErrScanWait);
        if (!__all_sync(TQ_FULL_MASK, landed)) break;
        const unsigned char* st = stages + (gi % kPfStages) * SB;
        const int ntg = min(kPfWarps, ntiles - kPfWarps * gi);
        for (int tt = 0; tt < ntg;) {
            const int tok0 = t0 + 16 * (kPfWarps * gi + tt);
            if (tok0 >= wlim) break;
            if (tt + 1 < ntg) {
                step(std::integral_constant<int, 2>{}, st, tt, tok0);
                tt += 2;
            } else {
                step(std::integral_constant<int, 1>{}, st, tt, tok0);
                tt += 1;
            }
        }
        __syncwarp();
        if (lane == 0) {  // done with this stage; the last of the four warps refills it
            const int sb = gi % kPfStages;
            __threadfence_block();
            const uint32_t before = atomicAdd(&s_cnt[sb], 1u);
            if (before == (uint32_t)(kPfWarps * (gi / kPfStages + 1)) - 1u && gi + kPfStages < ngroups)
                issue_group(gi + kPfStages);
        }
    }
    if (gi < ngroups) {
        // a copy did not land in time (the error word says so; the partials
        // are not valid): wait, bounded, for the copies still in flight
        for (int j = gi; j < ngroups && j < gi + kPfStages; ++j)
            mbar_wait_bounded(bar0 + 8 * (j % kPfStages), (j / kPfStages) & 1, kWaitLimitNs, p.err, kErrScanWait);
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    // ---- this split's partials of the two rows: a (column n of n-tile (j, h)
    // is coordinate 16 n + 2 j + h), M and Z ----
#pragma unroll
    for (int row = 0; row < 2; ++row) {
        float z = Zp[row];
        z += __shfl_xor_sync(TQ_FULL_MASK, z, 1);
        z += __shfl_xor_sync(TQ_FULL_MASK, z, 2);
        if (qrow[row] < 0) continue;
        float* out = p.partial + (qrow[row] * p.n_splits + split) * (D + kPartPad);
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                out[16 * (2 * c) + 2 * j + h] = O[j][h][2 * row] * inv_lv;
                out[16 * (2 * c + 1) + 2 * j + h] = O[j][h][2 * row + 1] * inv_lv;
            }
        if (c == 0) {
            out[D] = M[row];
            out[D + 1] = z;
        }
    }
}

template <int KB, int VB, int KB2 = KB, int VB2 = VB>
size_t prefill_mma_smem() {
    using T = MmaTile<KB, VB, KB2, VB2>;
    return (size_t)kPfStages * kPfWarps * T::BYTES + (size_t)kPfWarps * 8 * 4 * 32 * sizeof(uint4);
}

template <int KB, int VB, int KB2 = KB, int VB2 = VB>
cudaError_t launch_prefill_mma_t(const PrefillParams& p, cudaStream_t s) {
    auto kern = prefill_mma_kernel<KB, VB, KB2, VB2>;
    const size_t smem = prefill_mma_smem<KB, VB, KB2, VB2>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned qbs = (unsigned)((p.chunk * p.group + kPfRows - 1) / kPfRows);
    dim3 grid(qbs, (unsigned)p.n_splits, (unsigned)(p.batch * p.hkv));
    kern<<<grid, kPfWarps * 32, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tqk
