// Split-K decode scan on the tensor cores (mma.sync m16n8k16, f16 x f16 -> f32).
//
// Same computation as the logit estimator and softmax-weighted value sum of
// the A2A TurboQuant explainer (end of "Stage 2": scores straight from the
// stored indices with the query rotated once) and the Qiita TurboQuant
// article ("One more stage ...": residual sign term):
//   l_t = n_t ( <q', cK[idx_t]> + sqrt(pi/2)/m * gamma_t <u, 2 z_t - 1> )
//   a   = sum_t exp(s_t - M) nV_t cV[idxV_t]          (rotated domain)
// computed per 16-token tile of one KV head for all G query heads at once.
//
// Operands are built in registers, never staged as de-quantized tiles:
//  * keys   A[token][coord] = lam_k * cK[idx] as fp16 (a 2-coordinate lookup
//           table; lam_k is chosen on the host so that every centroid is very
//           close to an fp16 value), B[coord][2h+s] = hi/lo fp16 split of
//           q'_h (s = 0 hi, 1 lo), so the f32 accumulator holds the dot
//           product to about fp32 accuracy;
//  * signs  A[token][j] = +-1 (exact), B[j][2h+s] = hi/lo of kappa u_h;
//  * values A[coord][token] = lam_v * cV[idx] (fp16 table), B[token][2h+s] =
//           hi/lo of p_t nV_t.
// The MMA K dimension is permuted (keys: thread c of a quad holds coordinates
// 32c..32c+31; values: tokens 4c..4c+3) and the value M dimension too (row g
// holds coordinates 16g..16g+15), so each thread reads contiguous code bits.
//
// Tiles are staged in a 4-deep ring of CTA-wide shared-memory stages, each
// holding one tile per warp (64 tokens) and filled by six bulk (TMA) copies
// -- one per cache plane -- that complete on the stage's mbarrier. The capacity
// of the cache must be a multiple of 16 so that a tile never leaves its row.
//
// Fractional-rate caches (two channel groups, the Qiita article's 2.5 / 3.5
// bit rows): coordinate i has KB code bits when i % 16 < 8 and KB2 otherwise
// (values VB / VB2), codes packed in coordinate order, 8 (KB + KB2) bytes per
// token. With the K permutation above, thread c's k-steps kk = 0, 1, 4, 5 hold
// first-group coordinates and kk = 2, 3, 6, 7 second-group ones; with the M
// permutation, value m-tiles 0..3 are first-group and 4..7 second-group.
// Each group has its own pair table, both scaled by one lam.
#pragma once

#include "common.cuh"
#include "pipeline.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kMmaWarps = 4;
constexpr int kMmaStages = 4;

template <int KB, int VB, int KB2 = KB, int VB2 = VB>
struct MmaTile {
    static constexpr int KS = 8 * (KB + KB2);  // key code bytes per token
    static constexpr int VS = 8 * (VB + VB2);  // value code bytes per token
    static constexpr int KC = 16 * KS;         // key code bytes (16 tokens)
    static constexpr int SG = 16 * 16;         // sign bytes (m = 128)
    static constexpr int NB = 32;              // 16 fp16 scalars
    static constexpr int VC = 16 * VS;         // value code bytes
    static constexpr int OFF_KC = 0;
    static constexpr int OFF_SG = OFF_KC + KC;
    static constexpr int OFF_KN = OFF_SG + SG;
    static constexpr int OFF_KR = OFF_KN + NB;
    static constexpr int OFF_VC = OFF_KR + NB;
    static constexpr int OFF_VN = OFF_VC + VC;
    static constexpr int BYTES = OFF_VN + NB;
    static constexpr int CHUNKS = BYTES / 16;
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// hi/lo fp16 split of v: the fp16 bits of the hi part, or of v - hi
__device__ __forceinline__ uint32_t split_half(float v, int lo) {
    __half h = __float2half_rn(v);
    if (lo) h = __float2half_rn(v - __half2float(h));
    return (uint32_t)__half_as_ushort(h);
}

// bits [off, off+n) of a little-endian word array; called inside fully
// unrolled loops so that off and n fold to constants
__device__ __forceinline__ uint32_t field(const uint32_t* w, int off, int n) {
    const int W = off >> 5, S = off & 31;
    const uint32_t v = (S + n <= 32) ? (w[W] >> S) : __funnelshift_r(w[W], w[W + 1], S);
    return n >= 32 ? v : (v & ((1u << n) - 1u));
}

// 4 * field(w, off, n): the byte offset of a 4-byte table entry, in two ops
__device__ __forceinline__ uint32_t field4(const uint32_t* w, int off, int n) {
    const int W = off >> 5, S = off & 31;
    const uint32_t mask = ((1u << n) - 1u) << 2;
    if (S + n <= 32) return (S >= 2 ? (w[W] >> (S - 2)) : (w[W] << (2 - S))) & mask;
    return (__funnelshift_r(w[W], w[W + 1], S) << 2) & mask;
}

// 2^x with the hardware approximation (a few ulp in fp32; -inf gives +0):
// the softmax weights only, never the logits
__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(x));
    return r;
}

template <typename T>
__device__ __forceinline__ T lds_at(const void* base, uint32_t byte_off) {
    return *reinterpret_cast<const T*>(reinterpret_cast<const unsigned char*>(base) + byte_off);
}

// the bit offset of key k-step kk in thread c's run of 32 coordinates
// (fractional rates: k-steps 2, 3, 6, 7 are second-group)
template <int KB, int KB2>
__device__ __forceinline__ constexpr int key_off(int kk) {
    return (kk >> 2) * 8 * (KB + KB2) + ((kk & 3) == 0 ? 0 : (kk & 3) == 1 ? 4 * KB : (kk & 3) == 2 ? 8 * KB : 8 * KB + 4 * KB2);
}
// the bit offset of value m-tile mt in thread g's run of 16 coordinates
template <int VB, int VB2>
__device__ __forceinline__ constexpr int val_off(int mt) {
    return mt < 4 ? 2 * VB * mt : 8 * VB + 2 * VB2 * (mt - 4);
}

template <int KB, int VB, int G, int KB2 = KB, int VB2 = VB>
__global__ void __launch_bounds__(kMmaWarps * 32, (G > 4 ? 2 : 4)) decode_mma_kernel(const __grid_constant__ DecodeParams p) {
    using T = MmaTile<KB, VB, KB2, VB2>;
    constexpr int NT = (G + 3) / 4;   // n-tiles of 4 heads (x hi/lo)
    constexpr bool K2 = KB2 != KB, V2 = VB2 != VB;  // two channel groups
    constexpr int KL = 1 << (2 * KB);  // key pair-table entries
    constexpr int VL = 1 << (2 * VB);  // value pair-table entries
    constexpr int KL2 = K2 ? 1 << (2 * KB2) : 1, VL2 = V2 ? 1 << (2 * VB2) : 1;
    constexpr bool KLO = KB >= 3;      // second (lo) key table for 8+ centroids
    constexpr int D = 128;

    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* stages = smem;
    uint16_t* ps = reinterpret_cast<uint16_t*>(smem + kMmaWarps * kMmaStages * T::BYTES);  // [warps][NT][8][16]
    __shared__ uint32_t klut[KL];
    __shared__ uint32_t klo[KLO ? KL : 1];
    __shared__ uint32_t vlut[VL];
    __shared__ uint32_t klut2[KL2];
    __shared__ uint32_t klo2[(KLO && K2) ? KL2 : 1];
    __shared__ uint32_t vlut2[VL2];
    __shared__ __align__(8) uint2 slut4[16];  // 4 sign bits -> (+-1, +-1), (+-1, +-1) as fp16
    __shared__ __align__(8) uint64_t s_bar[kMmaStages];  // one per stage of the CTA ring
    __shared__ uint32_t s_cnt[kMmaStages];                // warps done with a stage, cumulative

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int split = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;

    for (int i = threadIdx.x; i < KL; i += blockDim.x) klut[i] = p.klut[i];
    if constexpr (KLO)
        for (int i = threadIdx.x; i < KL; i += blockDim.x) klo[i] = p.klut_lo[i];
    for (int i = threadIdx.x; i < VL; i += blockDim.x) vlut[i] = p.vlut[i];
    if constexpr (K2) {
        for (int i = threadIdx.x; i < KL2; i += blockDim.x) klut2[i] = p.klut2[i];
        if constexpr (KLO)
            for (int i = threadIdx.x; i < KL2; i += blockDim.x) klo2[i] = p.klut2_lo[i];
    }
    if constexpr (V2)
        for (int i = threadIdx.x; i < VL2; i += blockDim.x) vlut2[i] = p.vlut2[i];
    const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(&s_bar[0]);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int sb = 0; sb < kMmaStages; ++sb) {
            mbar_init(bar0 + 8 * sb, 1);
            s_cnt[sb] = 0u;
        }
        mbar_init_fence();
    }
    if (threadIdx.x < 16) {
        const uint32_t pos = 0x3C00u, neg = 0xBC00u, e = threadIdx.x;
        slut4[e].x = ((e & 1) ? pos : neg) | (((e & 2) ? pos : neg) << 16);
        slut4[e].y = ((e & 4) ? pos : neg) | (((e & 8) ? pos : neg) << 16);
    }

    // a length outside [0, min(capacity, max_seq_len)] is clamped into it
    const int L = max(0, (int)min((int64_t)p.seq_lens[b], min(p.capacity, (int64_t)p.max_seq_len)));
    const int t0 = split * p.chunk;
    const int t1 = min(t0 + p.chunk, L);
    const int ntiles = t1 > t0 ? (t1 - t0 + 15) >> 4 : 0;
    const int nmine = ntiles > warp ? (ntiles - warp + kMmaWarps - 1) / kMmaWarps : 0;
    const int64_t rowbase = ((int64_t)b * p.hkv + kv) * p.capacity;

    // ---- CTA ring: stage sb holds one group of kMmaWarps consecutive tiles (64
    // tokens, warp w's tile at position w), plane by plane: the region of plane
    // X starts at kMmaWarps * T::OFF_X, so each plane of a group is one bulk
    // copy. Group i goes to stage i % kMmaStages; the last warp done with a
    // group (a cumulative counter per stage) refills its stage with group
    // i + kMmaStages. ----
    constexpr int SB = kMmaWarps * T::BYTES;
    const uint32_t stages_s = (uint32_t)__cvta_generic_to_shared(stages);
    const int ngroups = (ntiles + kMmaWarps - 1) / kMmaWarps;
    auto issue_group = [&](int gi) {  // one thread
        const int sb = gi % kMmaStages;
        const int ntg = min(kMmaWarps, ntiles - kMmaWarps * gi);  // tiles in the group
        const int64_t slot = rowbase + t0 + 16 * kMmaWarps * gi;
        const uint32_t dst = stages_s + sb * SB, bar = bar0 + 8 * sb;
        const uint32_t ntok = 16u * (uint32_t)ntg;
        fence_proxy_async_smem();  // the warps' reads of this stage come first
        mbar_arrive_expect_tx(bar, (uint32_t)ntg * T::BYTES);
        bulk_g2s(dst + kMmaWarps * T::OFF_KC, p.kcodes + slot * T::KS, ntok * T::KS, bar);
        bulk_g2s(dst + kMmaWarps * T::OFF_SG, p.ksigns + slot * 16, ntok * 16, bar);
        bulk_g2s(dst + kMmaWarps * T::OFF_KN, p.knorm + slot, ntok * 2, bar);
        bulk_g2s(dst + kMmaWarps * T::OFF_KR, p.krnorm + slot, ntok * 2, bar);
        bulk_g2s(dst + kMmaWarps * T::OFF_VC, p.vcodes + slot * T::VS, ntok * T::VS, bar);
        bulk_g2s(dst + kMmaWarps * T::OFF_VN, p.vnorm + slot, ntok * 2, bar);
    };
    // Launched as a programmatic dependent of the query prep, which writes the
    // B operands and, in a decode step, appends the new token of each batch
    // row at append_pos[b]: griddepcontrol.wait returns once that launch has
    // completed. A split whose tiles do not hold the appended slot reads
    // nothing the prep writes into the cache, so its first copies go out
    // before the wait and overlap the prep.
    bool early = true;
    if (p.append_pos != nullptr) {
        const int ap = p.append_pos[b];
        early = !(ap >= t0 && ap < t0 + 16 * ntiles);
    }
    if (early && threadIdx.x == 0)
        for (int gi = 0; gi < kMmaStages && gi < ngroups; ++gi) issue_group(gi);
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    if (!early && threadIdx.x == 0)
        for (int gi = 0; gi < kMmaStages && gi < ngroups; ++gi) issue_group(gi);

    // ---- B fragments (static for the CTA), written by the query prep in the
    // order this thread reads them: 16 words of q' and 16 of kappa u ----
    uint32_t bk[NT][8][2], bs[NT][8][2];
    int qrow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hb = nt * 4 + (g >> 1);  // head of B column n = g
        const int lo = g & 1;
        const bool ok = hb < G;
        uint4 wk[4], ws[4];
        if (ok) {
            const int row = b * p.hq + (p.use_table ? (int)p.head_table[kv * G + hb] : kv * G + hb);
            const uint4* fk = reinterpret_cast<const uint4*>(p.frag + (int64_t)row * kFragWords + (lo * 4 + c) * 16);
            const uint4* fs = fk + (2 * 4 * 16) / 4;  // ks = 1
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                wk[j] = __ldg(fk + j);
                ws[j] = __ldg(fs + j);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) wk[j] = ws[j] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // words 4j .. 4j+3 = (kk, r) = (2j, 0), (2j, 1), (2j+1, 0), (2j+1, 1)
            bk[nt][2 * j][0] = wk[j].x; bk[nt][2 * j][1] = wk[j].y;
            bk[nt][2 * j + 1][0] = wk[j].z; bk[nt][2 * j + 1][1] = wk[j].w;
            bs[nt][2 * j][0] = ws[j].x; bs[nt][2 * j][1] = ws[j].y;
            bs[nt][2 * j + 1][0] = ws[j].z; bs[nt][2 * j + 1][1] = ws[j].w;
        }
        const int hc = nt * 4 + c;  // head whose logits this thread owns
        qrow[nt] = hc < G ? b * p.hq + (p.use_table ? (int)p.head_table[kv * G + hc] : kv * G + hc) : -1;
    }

    float M[NT], Zp[NT], acc[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        M[nt] = -INFINITY;
        Zp[nt] = 0.0f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[nt][mt][r] = 0.0f;
    }

    __syncthreads();  // lookup tables filled
    const float inv_lk = p.inv_lam_k, inv_lv = p.inv_lam_v;
    uint16_t* wps = ps + warp * NT * 8 * 16;

    int i = 0;
    for (; i < nmine; ++i) {
        // warp-uniform outcome of the bounded wait on this tile's buffer
        const bool landed = mbar_wait_bounded(bar0 + 8 * (i % kMmaStages), (i / kMmaStages) & 1, kWaitLimitNs,
                                              p.err, kErrScanWait);
        if (!__all_sync(TQ_FULL_MASK, landed)) break;
        // this warp's tile inside the stage: plane X at kMmaWarps * OFF_X + warp * (size of X)
        const unsigned char* st = stages + (i % kMmaStages) * SB;
        const unsigned char* p_kc = st + kMmaWarps * T::OFF_KC + warp * T::KC;
        const unsigned char* p_sg = st + kMmaWarps * T::OFF_SG + warp * T::SG;
        const unsigned char* p_kn = st + kMmaWarps * T::OFF_KN + warp * T::NB;
        const unsigned char* p_kr = st + kMmaWarps * T::OFF_KR + warp * T::NB;
        const unsigned char* p_vc = st + kMmaWarps * T::OFF_VC + warp * T::VC;
        const unsigned char* p_vn = st + kMmaWarps * T::OFF_VN + warp * T::NB;
        const int tok0 = t0 + 16 * (warp + kMmaWarps * i);

        // ---- keys and signs: D[token][2h+s] ----
        // thread c's 32 coordinates: 16 (KB + KB2) bits from bit 16 c (KB + KB2)
        constexpr int KWN = (KB + KB2 + 1) / 2;  // words holding them
        uint32_t kw0[KWN + 1], kw1[KWN + 1];
        if constexpr (!K2) {
            const uint32_t* r0 = reinterpret_cast<const uint32_t*>(p_kc + g * T::KS) + KB * c;
            const uint32_t* r1 = reinterpret_cast<const uint32_t*>(p_kc + (g + 8) * T::KS) + KB * c;
#pragma unroll
            for (int w = 0; w < KB; ++w) {
                kw0[w] = r0[w];
                kw1[w] = r1[w];
            }
        } else {
            // an odd KB + KB2 starts odd c's run half way into a word
            constexpr int TW = T::KS / 4;  // words per token
            const int wb = (c * (KB + KB2)) >> 1, sh = ((c * (KB + KB2)) & 1) * 16;
            const uint32_t* r0 = reinterpret_cast<const uint32_t*>(p_kc + g * T::KS) + wb;
            const uint32_t* r1 = reinterpret_cast<const uint32_t*>(p_kc + (g + 8) * T::KS) + wb;
            uint32_t x0[KWN + 1], x1[KWN + 1];
#pragma unroll
            for (int w = 0; w <= KWN; ++w) {
                x0[w] = wb + w < TW ? r0[w] : 0u;
                x1[w] = wb + w < TW ? r1[w] : 0u;
            }
#pragma unroll
            for (int w = 0; w < KWN; ++w) {
                kw0[w] = __funnelshift_r(x0[w], x0[w + 1], sh);
                kw1[w] = __funnelshift_r(x1[w], x1[w + 1], sh);
            }
        }
        kw0[KWN] = 0u;
        kw1[KWN] = 0u;
        const uint32_t sw0 = reinterpret_cast<const uint32_t*>(p_sg + g * 16)[c];
        const uint32_t sw1 = reinterpret_cast<const uint32_t*>(p_sg + (g + 8) * 16)[c];
        // two accumulator chains per product (even and odd kk) so that
        // consecutive MMAs do not wait on each other
        float dk[2][NT][4], ds[2][NT][4];
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    dk[e][nt][r] = 0.0f;
                    ds[e][nt][r] = 0.0f;
                }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const bool first = !K2 || (kk & 3) < 2;
            const int kw = first ? KB : KB2, ko = key_off<KB, KB2>(kk);
            const uint32_t* tab = first ? klut : klut2;
            const uint32_t* tlo = first ? klo : klo2;
            const uint32_t f0 = field4(kw0, ko, 2 * kw), f1 = field4(kw1, ko, 2 * kw);
            const uint32_t f2 = field4(kw0, ko + 2 * kw, 2 * kw);
            const uint32_t f3 = field4(kw1, ko + 2 * kw, 2 * kw);
            const uint32_t a0 = lds_at<uint32_t>(tab, f0), a1 = lds_at<uint32_t>(tab, f1);
            const uint32_t a2 = lds_at<uint32_t>(tab, f2), a3 = lds_at<uint32_t>(tab, f3);
            if constexpr (KLO) {
                const uint32_t l0 = lds_at<uint32_t>(tlo, f0), l1 = lds_at<uint32_t>(tlo, f1);
                const uint32_t l2 = lds_at<uint32_t>(tlo, f2), l3 = lds_at<uint32_t>(tlo, f3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma16816(dk[kk & 1][nt], l0, l1, l2, l3, bk[nt][kk][0], bk[nt][kk][1]);
            }
            // four sign bits 4kk..4kk+3 -> registers for slots (0,1) and (2,3)
            const uint2 sg0 = lds_at<uint2>(slut4, kk == 0 ? (sw0 << 3) & 0x78u : (sw0 >> (4 * kk - 3)) & 0x78u);
            const uint2 sg1 = lds_at<uint2>(slut4, kk == 0 ? (sw1 << 3) & 0x78u : (sw1 >> (4 * kk - 3)) & 0x78u);
            const uint32_t s0 = sg0.x, s1 = sg1.x, s2 = sg0.y, s3 = sg1.y;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                mma16816(dk[kk & 1][nt], a0, a1, a2, a3, bk[nt][kk][0], bk[nt][kk][1]);
                mma16816(ds[kk & 1][nt], s0, s1, s2, s3, bs[nt][kk][0], bs[nt][kk][1]);
            }
        }

        const uint16_t* kn = reinterpret_cast<const uint16_t*>(p_kn);
        const uint16_t* kr = reinterpret_cast<const uint16_t*>(p_kr);
        const uint16_t* vn = reinterpret_cast<const uint16_t*>(p_vn);
        const bool v0 = tok0 + g < t1, v1 = tok0 + g + 8 < t1;
        const float kn0 = f16_bits_to_f32(kn[g]), kn1 = f16_bits_to_f32(kn[g + 8]);
        const float kg0 = f16_bits_to_f32(kr[g]), kg1 = f16_bits_to_f32(kr[g + 8]);
        const float vn0 = f16_bits_to_f32(vn[g]), vn1 = f16_bits_to_f32(vn[g + 8]);

#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const bool hv = qrow[nt] >= 0;
            // column 2h holds the hi split of head h, 2h+1 the lo split
            const float k0 = (dk[0][nt][0] + dk[1][nt][0]) + (dk[0][nt][1] + dk[1][nt][1]);
            const float k1 = (dk[0][nt][2] + dk[1][nt][2]) + (dk[0][nt][3] + dk[1][nt][3]);
            const float s0_ = (ds[0][nt][0] + ds[1][nt][0]) + (ds[0][nt][1] + ds[1][nt][1]);
            const float s1_ = (ds[0][nt][2] + ds[1][nt][2]) + (ds[0][nt][3] + ds[1][nt][3]);
            const float l0 = kn0 * fmaf(kg0, s0_, k0 * inv_lk);
            const float l1 = kn1 * fmaf(kg1, s1_, k1 * inv_lk);
            if (p.logits != nullptr && hv) {
                if (v0) p.logits[(int64_t)qrow[nt] * p.max_seq_len + tok0 + g] = l0;
                if (v1) p.logits[(int64_t)qrow[nt] * p.max_seq_len + tok0 + g + 8] = l1;
            }
            const float s0 = (v0 && hv) ? l0 * p.scale_log2 : -INFINITY;
            const float s1 = (v1 && hv) ? l1 * p.scale_log2 : -INFINITY;
            float m = fmaxf(s0, s1);
            m = fmaxf(m, __shfl_xor_sync(TQ_FULL_MASK, m, 4));
            m = fmaxf(m, __shfl_xor_sync(TQ_FULL_MASK, m, 8));
            m = fmaxf(m, __shfl_xor_sync(TQ_FULL_MASK, m, 16));
            const float mn = fmaxf(M[nt], m);
            const float corr = (mn == -INFINITY) ? 1.0f : ex2(M[nt] - mn);
            const float p0 = (s0 == -INFINITY) ? 0.0f : ex2(s0 - mn);
            const float p1 = (s1 == -INFINITY) ? 0.0f : ex2(s1 - mn);
            Zp[nt] = fmaf(Zp[nt], corr, p0 + p1);
            M[nt] = mn;
            // the running max of a head rarely moves after the first tiles:
            // rescale only when it moved for some head of the warp
            if (__any_sync(TQ_FULL_MASK, corr != 1.0f)) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[nt][mt][r] *= corr;
            }
            const float w0 = v0 ? p0 * vn0 : 0.0f, w1 = v1 ? p1 * vn1 : 0.0f;
            uint16_t* row_hi = wps + (nt * 8 + 2 * c) * 16;
            uint16_t* row_lo = row_hi + 16;
            row_hi[g] = (uint16_t)split_half(w0, 0);
            row_lo[g] = (uint16_t)split_half(w0, 1);
            row_hi[g + 8] = (uint16_t)split_half(w1, 0);
            row_lo[g + 8] = (uint16_t)split_half(w1, 1);
        }
        __syncwarp();

        // ---- values: D[coord][2h+s] += A[coord][token] B[token][2h+s] ----
        uint32_t bv[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t* prow = reinterpret_cast<const uint32_t*>(wps + (nt * 8 + g) * 16);
            bv[nt][0] = prow[2 * c];      // tokens 4c, 4c+1
            bv[nt][1] = prow[2 * c + 1];  // tokens 4c+2, 4c+3
        }
        // each thread: tokens 4c..4c+3, coordinates 16g..16g+15 (8 (VB + VB2)
        // bits from bit 8 (VB + VB2) g)
        uint32_t vf[4][3];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t* vr = reinterpret_cast<const uint32_t*>(p_vc + (4 * c + j) * T::VS);
            const int bit0 = 8 * (VB + VB2) * g;
            const int w = bit0 >> 5, sh = bit0 & 31;
            const uint32_t x0 = vr[w];
            const uint32_t x1 = (w + 1 < T::VS / 4) ? vr[w + 1] : 0u;
            const uint32_t x2 = (w + 2 < T::VS / 4) ? vr[w + 2] : 0u;
            vf[j][0] = __funnelshift_r(x0, x1, sh);
            vf[j][1] = __funnelshift_r(x1, x2, sh);
            vf[j][2] = 0u;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t x[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                x[j] = (!V2 || mt < 4) ? lds_at<uint32_t>(vlut, field4(vf[j], val_off<VB, VB2>(mt), 2 * VB))
                                       : lds_at<uint32_t>(vlut2, field4(vf[j], val_off<VB, VB2>(mt), 2 * VB2));
            const uint32_t a0 = prmt(x[0], x[1], 0x5410u);
            const uint32_t a1 = prmt(x[0], x[1], 0x7632u);
            const uint32_t a2 = prmt(x[2], x[3], 0x5410u);
            const uint32_t a3 = prmt(x[2], x[3], 0x7632u);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(acc[nt][mt], a0, a1, a2, a3, bv[nt][0], bv[nt][1]);
        }
        __syncwarp();
        if (lane == 0) {  // done with this stage; the last warp of the group refills it
            const int sb = i % kMmaStages;
            const uint32_t arrivals = (uint32_t)min(kMmaWarps, ntiles - kMmaWarps * i);
            __threadfence_block();
            const uint32_t before = atomicAdd(&s_cnt[sb], 1u);
            // cumulative count: every earlier group of this stage was complete (kMmaWarps arrivals)
            if (before == (uint32_t)(kMmaWarps * (i / kMmaStages)) + arrivals - 1u && i + kMmaStages < ngroups)
                issue_group(i + kMmaStages);
        }
    }
    if (i < nmine) {
        // a copy did not land in time (the error word says so and this
        // split's output is not valid): wait, bounded, for the copies still
        // in flight before the buffers are reused below
        for (int j = i; j < nmine && j < i + kMmaStages; ++j)
            mbar_wait_bounded(bar0 + 8 * (j % kMmaStages), (j / kMmaStages) & 1, kWaitLimitNs, p.err, kErrScanWait);
    }
    __syncthreads();

    // the merge kernel may be scheduled now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    // ---- merge the warps of the CTA and write this split's partials ----
    float* s_acc = reinterpret_cast<float*>(smem);  // [warps][G][D]
    float* s_mz = s_acc + kMmaWarps * G * D;        // [warps][G][2]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float z = Zp[nt];
        z += __shfl_xor_sync(TQ_FULL_MASK, z, 4);
        z += __shfl_xor_sync(TQ_FULL_MASK, z, 8);
        z += __shfl_xor_sync(TQ_FULL_MASK, z, 16);
        const int h = nt * 4 + c;
        if (h < G) {
            float* dst = s_acc + (warp * G + h) * D;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                dst[16 * g + 2 * mt] = (acc[nt][mt][0] + acc[nt][mt][1]) * inv_lv;
                dst[16 * g + 2 * mt + 1] = (acc[nt][mt][2] + acc[nt][mt][3]) * inv_lv;
            }
            if (g == 0) {
                s_mz[(warp * G + h) * 2] = M[nt];
                s_mz[(warp * G + h) * 2 + 1] = z;
            }
        }
    }
    __syncthreads();
    const int ci = threadIdx.x;  // coordinate 0..127
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float mstar = -INFINITY;
#pragma unroll
        for (int w = 0; w < kMmaWarps; ++w) mstar = fmaxf(mstar, s_mz[(w * G + h) * 2]);
        float z = 0.0f, a = 0.0f;
#pragma unroll
        for (int w = 0; w < kMmaWarps; ++w) {
            const float mw = s_mz[(w * G + h) * 2];
            const float wt = (mw == -INFINITY) ? 0.0f : ex2(mw - mstar);
            z = fmaf(s_mz[(w * G + h) * 2 + 1], wt, z);
            a = fmaf(s_acc[(w * G + h) * D + ci], wt, a);
        }
        const int row = b * p.hq + (p.use_table ? (int)p.head_table[kv * G + h] : kv * G + h);
        float* out = p.partial + ((int64_t)row * p.n_splits + split) * (D + kPartPad);
        out[ci] = a;
        if (ci == 0) {
            out[D] = mstar;
            out[D + 1] = z;
        }
    }
}

template <int KB, int VB, int G, int KB2 = KB, int VB2 = VB>
size_t decode_mma_smem();

// Launches the scan as a programmatic dependent of the launch before it on
// the stream: its CTAs may become resident and set up while that launch runs,
// and wait for it (griddepcontrol.wait) before reading anything.
template <int KB, int VB, int G, int KB2 = KB, int VB2 = VB>
cudaError_t launch_decode_mma_t(const DecodeParams& p, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.n_splits, (unsigned)p.hkv, (unsigned)p.batch);
    cfg.blockDim = dim3(kMmaWarps * 32);
    cfg.dynamicSmemBytes = decode_mma_smem<KB, VB, G, KB2, VB2>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_mma_kernel<KB, VB, G, KB2, VB2>, p);
}

template <int KB, int VB, int G, int KB2, int VB2>
size_t decode_mma_smem() {
    using T = MmaTile<KB, VB, KB2, VB2>;
    constexpr int NT = (G + 3) / 4;
    size_t pipe = (size_t)kMmaWarps * kMmaStages * T::BYTES + 2 * kMmaWarps * NT * 8 * 16;
    size_t merge = (size_t)kMmaWarps * G * 128 * 4 + kMmaWarps * G * 2 * 4;
    return pipe > merge ? pipe : merge;
}

}  // namespace tqk

namespace tqk {

// Instantiations for one G: every single-width (KB, VB) in 1..4, and the
// fractional-rate caches with both keys and values split into two groups
// (KB2 = KB - 1, VB2 = VB - 1).
template <int G, int KB, int KB2>
cudaError_t decode_mma_v(const DecodeParams& p, int vb, cudaStream_t s) {
    constexpr bool two = KB2 != KB;
    switch (vb) {
        case 1:
            if constexpr (!two) return launch_decode_mma_t<KB, 1, G>(p, s);
            break;
        case 2: return launch_decode_mma_t<KB, 2, G, KB2, two ? 1 : 2>(p, s);
        case 3: return launch_decode_mma_t<KB, 3, G, KB2, two ? 2 : 3>(p, s);
        case 4: return launch_decode_mma_t<KB, 4, G, KB2, two ? 3 : 4>(p, s);
    }
    return cudaErrorInvalidValue;
}

template <int G>
cudaError_t dispatch_decode_mma(const DecodeParams& p, int kbits, int vbits, bool two, cudaStream_t s) {
    if (!two) {
        switch (kbits) {
            case 1: return decode_mma_v<G, 1, 1>(p, vbits, s);
            case 2: return decode_mma_v<G, 2, 2>(p, vbits, s);
            case 3: return decode_mma_v<G, 3, 3>(p, vbits, s);
            case 4: return decode_mma_v<G, 4, 4>(p, vbits, s);
        }
    } else {
        switch (kbits) {
            case 2: return decode_mma_v<G, 2, 1>(p, vbits, s);
            case 3: return decode_mma_v<G, 3, 2>(p, vbits, s);
            case 4: return decode_mma_v<G, 4, 3>(p, vbits, s);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace tqk
