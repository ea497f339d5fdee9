// Quantize-on-append for d = m = 128, bf16 input, on the 5th-generation
// tensor cores (tcgen05) with the accumulators in tensor memory.
//
// The steps are those of the A2A TurboQuant explainer ("Stage 1": random
// rotation, then a Lloyd-Max scalar quantizer per coordinate; "Stage 2": a
// 1-bit sign sketch of the residual) and of the Qiita TurboQuant article
// ("Rotate, then quantize"; "One more stage so attention does not break"):
//   n = ||x||, y = Pi x / n, idx_i = #{j : y_i >= t_j}, and for keys
//   r = y - c[idx], gamma = ||r||, z_j = [(S r)_j >= 0].
//
// Both rotations are one dense contraction Y = X W^T over a tile of 128
// vectors (M = 128, N = 128 output coordinates, K = 128):
//  * dense QR: W = Pi split into three bf16 limbs (about 24 bits), three
//    accumulating passes;
//  * randomized Hadamard: W = H diag(s), every entry +-1 and exact in bf16,
//    one pass; the 1/sqrt(d) scale is applied to the accumulator.
// The input is exact in bf16, so every product is exact and the fp32
// accumulation is the only rounding (the guard band below covers it).
// For keys the sign sketch is a second contraction Z = R S^T (N = 128 sign
// rows), R split into bf16 hi/lo halves (16 bits) against S (exact in bf16).
//
// Warp-specialised, persistent, one CTA per SM (it holds all 512 TMEM
// columns):
//  * TMA warp: tiled tensor copies of the 128-vector input tiles (two boxes
//    of 64 coordinates x 128 rows with the 128-byte swizzle, the K-major
//    layout the MMA reads) into a ring of shared-memory buffers;
//  * MMA warp: the rotation MMAs of a tile into one of NB TMEM accumulators
//    (four for values, two for keys), and (keys) the sign-sketch MMAs with
//    A = R read from TMEM;
//  * epilogue warps: thread = vector (its TMEM lane), each of the NP warps of
//    a lane quarter takes 128 / NP coordinates. Phase 1: the norm from the
//    staged input, then per 16 coordinates the rotated values from TMEM,
//    codes by sign-bit arithmetic (below), the guard test, the residual, and
//    (keys) R hi/lo written into R's own 128 columns once the previous tile's
//    sign-sketch MMAs have read them. Phase 2 (keys): the signs of S r from
//    TMEM.
// The epilogue runs phase 1 of tile i+1 before phase 2 of tile i, so the
// sign-sketch MMAs of tile i overlap it.
//
// Codes from sign bits: with the symmetric codebook (boundaries -t_H' ..
// -t_1, 0, t_1 .. t_H', centroids c), a coordinate with s = [y < 0] and
// thermometer g_j = [|y| >= t_j] has code (1 - s, k XOR s...) where k =
// sum_j g_j is written in binary as bit b = XOR of g_j over the j divisible
// by 2^b. Each g_j is the inverted sign bit of dv_j = |y| - t_j, and every
// such XOR has an odd number of terms, so every code bit is the inverted sign
// bit of (y XOR the dv_j of its terms). The bits are shifted into the packed
// words with funnel shifts (one instruction per bit) from the last stream bit
// down, and the words are inverted once at the end.
//
// Coordinates whose |y| lies within `guard` of a boundary are re-decided
// from an fp64 dot product (warp-cooperative), as in the other quantize
// kernels.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "pipeline.cuh"
#include "tcgen05.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kQuVec = 128;        // vectors per tile (MMA M, TMEM lanes)
constexpr int kQuD = 128;          // coordinates (MMA N and K)
constexpr uint32_t kQuTileBytes = kQuVec * kQuD * 2;  // 32 KB of bf16
constexpr uint32_t kQuBBytes = kQuD * kQuD * 2;       // one 128 x 128 bf16 operand

// epilogue warps per TMEM lane quarter (each takes 128 / kQuParts coordinates)
constexpr int kQuParts = 4;

struct QuantUmmaParams {
    CUtensorMap tmap;     // the input: 2-D bf16 [n][128] (row stride x_stride), box 64 x 128, 128-byte swizzle
    QuantParams q;
    const void* w_umma;   // rotation operand(s), 128 x 128 bf16 each, K-major with the 128-byte swizzle
    const void* s_umma;   // S, 128 x 128 bf16, the same layout (keys)
};

template <int NP>
struct QuCfg {
    static constexpr int kEpi = 4 * NP;             // epilogue warps
    static constexpr int kWarps = kEpi + 2;         // + TMA warp + MMA warp
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kCpt = kQuD / NP;          // coordinates per epilogue thread
    static constexpr int kNch = kCpt / 32;          // 32-coordinate chunks per thread
};

// input tile buffers: as many as fit beside the operands (2 to 4)
__host__ __device__ constexpr int qu_xbufs(int nlimb, bool prod) {
    const int fixed = nlimb * 32 + (prod ? 32 : 0) + 6;  // KB: operands, partials, slack
    const int n = (227 - fixed) / 32;
    return n > 4 ? 4 : n;
}

// bytes of dynamic shared memory: rotation limbs, S, input buffers, norm and
// gamma partials
template <int NP>
__host__ __device__ constexpr size_t qu_smem_bytes(int nlimb, bool prod) {
    return (size_t)nlimb * kQuBBytes + (prod ? kQuBBytes : 0) + (size_t)qu_xbufs(nlimb, prod) * kQuTileBytes +
           (size_t)4 * NP * kQuVec * sizeof(float) + 1024;  // + 1024: alignment slack
}

__device__ __forceinline__ uint32_t shf_in(uint32_t acc, uint32_t src) {
    // (acc << 1) | (src >> 31): shift the sign bit of src into the word
    return __funnelshift_l(src, acc, 1);
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// fp32 bits XOR
__device__ __forceinline__ uint32_t fx(float a) { return __float_as_uint(a); }

// CB2 != CB: a fractional-rate cache (two channel groups): coordinate i
// takes CB code bits and the first codebook when i % 16 < 8, CB2 bits and
// the second codebook otherwise, codes packed in coordinate order with their
// own widths. Inside a 32-coordinate chunk every coordinate's group and bit
// offset are compile-time constants.
template <int CB, int CB2, bool PROD, bool RHT, int NP>
__global__ void __launch_bounds__(QuCfg<NP>::kThreads, 1)
    quantize_umma_kernel(const __grid_constant__ QuantUmmaParams P) {
    using C = QuCfg<NP>;
    constexpr int NL = RHT ? 1 : 3;        // bf16 limbs of W
    constexpr bool TWO = CB2 != CB;
    constexpr int L = 1 << CB, L2 = 1 << CB2;                  // cells
    constexpr int HX = L / 2, HX2 = L2 / 2;                    // first non-negative cell
    constexpr int NPB = HX - 1, NPB2 = HX2 - 1;                // positive boundaries t_1 .. t_NPB
    constexpr int CHB = 16 * (CB + CB2);                       // packed bits of a 32-coordinate chunk
    static_assert(!TWO || CB2 == CB - 1, "the second group is one bit narrower");
    constexpr int kQuXBufs = qu_xbufs(NL, PROD);
    // TMEM: rotation accumulators at columns 128 b (b < NB1); keys also R
    // (hi/lo halves) at 256 and the S r accumulator at 384
    constexpr int NB1 = PROD ? 2 : 4;
    constexpr uint32_t kColR = 256, kColZ = 384;
    static_assert(kQuXBufs >= 2, "two input buffers at least");
    const QuantParams& p = P.q;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned start (the swizzle atoms), derived from smem_raw so
    // that the compiler keeps the shared address space (plain shared loads)
    unsigned char* smem = smem_raw + ((1024u - ((uint32_t)__cvta_generic_to_shared(smem_raw) & 1023u)) & 1023u);
    unsigned char* sB1 = smem;                                  // NL x [128 x 128] rotation operand
    unsigned char* sB2 = sB1 + (size_t)NL * kQuBBytes;          // S (keys)
    unsigned char* sX = sB2 + (PROD ? kQuBBytes : 0);           // input tiles
    // norm and gamma partials of the NP warps of a lane quarter, [2][NP][128]
    // each (double-buffered by tile parity: a warp can only refill a buffer
    // after every warp of its quarter arrived on the next exchange)
    float* s_nrm = reinterpret_cast<float*>(sX + (size_t)kQuXBufs * kQuTileBytes);
    float* s_gam = s_nrm + 2 * NP * kQuVec;

    __shared__ __align__(8) uint64_t s_bfull;
    __shared__ __align__(8) uint64_t s_xfull[kQuXBufs], s_xfree[kQuXBufs];
    __shared__ __align__(8) uint64_t s_a1full[NB1], s_tfree[NB1];   // rotation accumulator full / read
    __shared__ __align__(8) uint64_t s_rfull, s_a2full, s_a2free;     // keys: R written, S r done / read
    __shared__ __align__(8) uint64_t s_xn[4], s_xg[4];  // partial-sum exchanges, one per lane quarter
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ float s_sgn[RHT ? kQuD : 1];  // RHT signs, for the fp64 re-decisions

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntiles = (p.n + kQuVec - 1) / kQuVec;
    const int64_t nmine = (int)blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    const uint32_t bfull = (uint32_t)__cvta_generic_to_shared(&s_bfull);
    const uint32_t xfull0 = (uint32_t)__cvta_generic_to_shared(&s_xfull[0]);
    const uint32_t xfree0 = (uint32_t)__cvta_generic_to_shared(&s_xfree[0]);
    const uint32_t a1full0 = (uint32_t)__cvta_generic_to_shared(&s_a1full[0]);
    const uint32_t tfree0 = (uint32_t)__cvta_generic_to_shared(&s_tfree[0]);
    const uint32_t rfull = (uint32_t)__cvta_generic_to_shared(&s_rfull);
    const uint32_t a2full = (uint32_t)__cvta_generic_to_shared(&s_a2full);
    const uint32_t a2free = (uint32_t)__cvta_generic_to_shared(&s_a2free);
    const uint32_t xn0 = (uint32_t)__cvta_generic_to_shared(&s_xn[0]);
    const uint32_t xg0 = (uint32_t)__cvta_generic_to_shared(&s_xg[0]);
    if (tid == 0) {
        for (int q = 0; q < 4; ++q) {
            mbar_init(xn0 + 8 * q, NP);
            mbar_init(xg0 + 8 * q, NP);
        }
        mbar_init(bfull, 1);
        for (int b = 0; b < kQuXBufs; ++b) {
            mbar_init(xfull0 + 8 * b, 1);
            mbar_init(xfree0 + 8 * b, C::kEpi + 1);  // the epilogue warps and the rotation MMAs' commit
        }
        for (int b = 0; b < NB1; ++b) {
            mbar_init(a1full0 + 8 * b, 1);
            mbar_init(tfree0 + 8 * b, C::kEpi);
        }
        mbar_init(rfull, C::kEpi);
        mbar_init(a2full, 1);
        mbar_init(a2free, C::kEpi);
        s_abort = 0;
        mbar_init_fence();
    }
    if constexpr (RHT)
        if (tid < kQuD) s_sgn[tid] = p.sgn[tid];
    if (warp == 1) {
        tmem_alloc((uint32_t)__cvta_generic_to_shared(&s_tmem), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;

    if (warp == 0) {
        // ======================= TMA =======================
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(&P.tmap) : "memory");
            // the static operands: W limbs and S, once per CTA
            mbar_arrive_expect_tx(bfull, (uint32_t)(NL + (PROD ? 1 : 0)) * kQuBBytes);
            const uint32_t b1 = (uint32_t)__cvta_generic_to_shared(sB1);
            constexpr uint32_t CH = 16384;  // bytes per bulk copy
            for (uint32_t o = 0; o < NL * kQuBBytes; o += CH)
                bulk_g2s(b1 + o, reinterpret_cast<const unsigned char*>(P.w_umma) + o, CH, bfull);
            if constexpr (PROD)
                for (uint32_t o = 0; o < kQuBBytes; o += CH)
                    bulk_g2s((uint32_t)__cvta_generic_to_shared(sB2) + o,
                             reinterpret_cast<const unsigned char*>(P.s_umma) + o, CH, bfull);
            int64_t issued = 0;
            for (int64_t it = 0; it < nmine; ++it) {
                const int xb = (int)(it % kQuXBufs);
                if (it >= kQuXBufs &&
                    !mbar_wait_bounded(xfree0 + 8 * xb, (uint32_t)(((it / kQuXBufs) - 1) & 1), kWaitLimitNs, p.err,
                                       kErrQuantWait)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const int64_t tile = blockIdx.x + it * gridDim.x;
                const uint32_t dst = (uint32_t)__cvta_generic_to_shared(sX + (size_t)xb * kQuTileBytes);
                mbar_arrive_expect_tx(xfull0 + 8 * xb, kQuTileBytes);
                // coordinates 0..63 and 64..127: two 16 KB swizzled halves
                tma_load_2d(dst, &P.tmap, 0, (int)(tile * kQuVec), xfull0 + 8 * xb);
                tma_load_2d(dst + kQuTileBytes / 2, &P.tmap, 64, (int)(tile * kQuVec), xfull0 + 8 * xb);
                issued = it + 1;
            }
            // every copy issued lands (bounded) before the CTA's shared memory is released
            for (int64_t it = issued > kQuXBufs ? issued - kQuXBufs : 0; it < issued; ++it)
                mbar_wait_bounded(xfull0 + 8 * (int)(it % kQuXBufs), (uint32_t)((it / kQuXBufs) & 1), kWaitLimitNs,
                                  p.err, kErrQuantWait);
            mbar_wait_bounded(bfull, 0, kWaitLimitNs, p.err, kErrQuantWait);
        }
    } else if (warp == 1) {
        // ======================= MMA =======================
        if (lane == 0) {
            bool ok = mbar_wait_bounded(bfull, 0, kWaitLimitNs, p.err, kErrQuantWait);
            const uint32_t idesc = umma_idesc_bf16(kQuVec, kQuD);
            // A = input tile, two 128-byte-swizzled halves of 64 coordinates:
            // element (r, k) at (k/64)*16384 + r*128 + (((k%64)/8) ^ (r%8))*16
            // + (k%8)*2 (SBO 1024 between 8-row atoms); a K = 16 step moves the
            // start 32 bytes along the row
            const uint32_t x0 = (uint32_t)__cvta_generic_to_shared(sX);
            // B = W / S in the same swizzled K-major layout (two 16 KB halves of
            // 64 coordinates per 128 x 128 operand)
            const uint32_t b1s = (uint32_t)__cvta_generic_to_shared(sB1);
            const uint32_t b2s = (uint32_t)__cvta_generic_to_shared(sB2);
            int64_t last_commit = -1;  // tiles whose last MMA was committed
            auto rot = [&](int64_t it) -> bool {
                const int xb = (int)(it % kQuXBufs), tb = (int)(it % NB1);
                if (!mbar_wait_bounded(xfull0 + 8 * xb, (uint32_t)((it / kQuXBufs) & 1), kWaitLimitNs, p.err,
                                       kErrQuantWait))
                    return false;
                // the epilogue has read this accumulator's previous tile
                if (it >= NB1 && !mbar_wait_bounded(tfree0 + 8 * tb, (uint32_t)(((it / NB1) - 1) & 1), kWaitLimitNs,
                                                    p.err, kErrQuantWait))
                    return false;
                tc_fence_after_sync();
                const uint32_t xa = x0 + xb * kQuTileBytes;
                const uint32_t acc = tmem + (uint32_t)(128 * tb);
#pragma unroll
                for (int l = 0; l < NL; ++l)
#pragma unroll
                    for (int s = 0; s < kQuD / 16; ++s)
                        umma_f16(acc, umma_desc_sw128(xa + (s >> 2) * (kQuTileBytes / 2) + (s & 3) * 32, 1024),
                                 umma_desc_sw128(b1s + l * kQuBBytes + (s >> 2) * (kQuBBytes / 2) + (s & 3) * 32, 1024),
                                 idesc, l > 0 || s > 0);
                umma_commit(a1full0 + 8 * tb);
                umma_commit(xfree0 + 8 * xb);
                return true;
            };
            auto sgn = [&](int64_t it) -> bool {
                // R of this tile written; the S r accumulator read by the previous tile's epilogue
                if (!mbar_wait_bounded(rfull, (uint32_t)(it & 1), kWaitLimitNs, p.err, kErrQuantWait)) return false;
                if (it >= 1 && !mbar_wait_bounded(a2free, (uint32_t)((it - 1) & 1), kWaitLimitNs, p.err, kErrQuantWait))
                    return false;
                tc_fence_after_sync();
                // R of coordinates 16g .. 16g+15: hi halves in columns 16g .. 16g+7,
                // lo halves in 16g+8 .. 16g+15 (two per column)
                const uint32_t racc = tmem + kColR;
                const uint32_t zacc = tmem + kColZ;
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const uint64_t bd = umma_desc_sw128(b2s + (g >> 2) * (kQuBBytes / 2) + (g & 3) * 32, 1024);
                    umma_f16_ta(zacc, racc + 16u * g, bd, idesc, g > 0);
                    umma_f16_ta(zacc, racc + 16u * g + 8u, bd, idesc, true);
                }
                umma_commit(a2full);
                return true;
            };
            for (int64_t it = 0; ok && it < nmine && it < NB1; ++it) ok = rot(it);
            for (int64_t it = 0; ok && it < nmine; ++it) {
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                if constexpr (PROD) {
                    if (!(ok = sgn(it))) break;
                }
                last_commit = it;
                if (it + NB1 < nmine && !(ok = rot(it + NB1))) break;
            }
            if (!ok) *abort_flag = 1;
            // the MMAs in flight complete (bounded) before TMEM is released: the
            // last commit covers every MMA issued before it
            if (nmine > 0) {
                if constexpr (PROD) {
                    if (last_commit >= 0)
                        mbar_wait_bounded(a2full, (uint32_t)(last_commit & 1), kWaitLimitNs, p.err, kErrQuantWait);
                } else {
                    const int64_t lt = nmine - 1;
                    mbar_wait_bounded(a1full0 + 8 * (int)(lt % NB1), (uint32_t)((lt / NB1) & 1), kWaitLimitNs, p.err,
                                      kErrQuantWait);
                }
            }
        }
    } else {
        // ======================= epilogue =======================
        const int ew = warp - 2;             // 0 .. 4 NP - 1
        const int qd = warp & 3;             // TMEM lane quarter this warp may access
        const int h = ew >> 2;               // coordinate part
        const int r = 32 * qd + lane;        // vector row in the tile (TMEM lane)
        const int cbase = C::kCpt * h;       // first coordinate of this thread
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * qd) << 16);
        // the NP warps of this quarter swap partial sums through shared
        // memory and an mbarrier (one arrival per warp, bounded wait)
        auto exchange = [&](uint32_t bar, float* buf, float val, int64_t it, bool& ok) -> float {
            float* b = buf + (int)(it & 1) * NP * kQuVec;
            b[h * kQuVec + r] = val;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
            if (!mbar_wait_bounded(bar, (uint32_t)(it & 1), kWaitLimitNs, p.err, kErrQuantWait)) ok = false;
            float t = 0.0f;
#pragma unroll
            for (int k = 0; k < NP; ++k) t += b[k * kQuVec + r];
            return t;
        };

        // positive boundaries (fp32) of each group's codebook
        float tp[NPB > 0 ? NPB : 1], tp2[NPB2 > 0 ? NPB2 : 1];
#pragma unroll
        for (int j = 0; j < NPB; ++j) tp[j] = p.cb.t[HX + j];
#pragma unroll
        for (int j = 0; j < NPB2; ++j) tp2[j] = TWO ? p.cb2.t[HX2 + j] : 0.0f;
        // stream bit of code bit 0 of coordinate j (0 .. 31) of a chunk: each
        // block of 16 holds 8 codes of CB bits, then 8 of CB2 bits
        auto bit_of = [](int j) {
            const int jl = j & 15;
            return (j >> 4) * 8 * (CB + CB2) + (jl < 8 ? CB * jl : 8 * CB + CB2 * (jl - 8));
        };

        auto slot_of = [&](int64_t v) -> int64_t {
            if (v >= p.n) return -1;
            int64_t s;
            if (p.dst_slot) {
                s = p.dst_slot[v];
            } else if (p.append_pos) {
                const int32_t pos = p.append_pos[v / p.heads];
                s = (pos >= 0 && pos < p.capacity) ? v * p.capacity + pos : -1;
            } else {
                s = p.slot0 + v;
            }
            return (s >= p.total_slots) ? -1 : s;
        };
        // staged input element (row `row` of buffer xb, coordinate k) as fp32,
        // for the rare fp64 paths: the tile stays staged until phase 1 ends,
        // so that a re-decision costs a shared-memory read, not a trip to HBM
        // (a slow warp would hold back every warp waiting on its barriers)
        auto xel = [&](int xb, int row, int k) -> float {
            const uint16_t b = *reinterpret_cast<const uint16_t*>(
                sX + (size_t)xb * kQuTileBytes + (k >> 6) * (kQuTileBytes / 2) + row * 128 +
                ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2);
            return __uint_as_float((uint32_t)b << 16);
        };

        // ---------------- phase 1: norm, codes, residual ----------------
        auto phase1 = [&](int64_t it) -> bool {
            const int xb = (int)(it % kQuXBufs), tb = (int)(it % NB1);
            const int64_t tile = blockIdx.x + it * gridDim.x;
            const int64_t v = tile * kQuVec + r;
            const bool valid = v < p.n;
            // a failed wait still takes part in both exchanges (so no partner
            // waits for an arrival that never comes), then reports failure
            bool ok = mbar_wait_bounded(xfull0 + 8 * xb, (uint32_t)((it / kQuXBufs) & 1), kWaitLimitNs, p.err,
                                        kErrQuantWait);
            // partial sum of squares over this thread's coordinates (row r of
            // the swizzled halves: chunk j of 8 coordinates at chunk j ^ (r % 8))
            const unsigned char* xrow = sX + (size_t)xb * kQuTileBytes + r * 128;
            float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < C::kCpt / 8; ++j) {
                const int k8 = cbase / 8 + j;  // chunk of 8 coordinates, 0..15
                const uint4 w = *reinterpret_cast<const uint4*>(xrow + (k8 >> 3) * (kQuTileBytes / 2) +
                                                                (((k8 & 7) ^ (r & 7)) << 4));
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 xv = make_float2(__uint_as_float(ww[e] << 16), __uint_as_float(ww[e] & 0xFFFF0000u));
                    ss2 = __ffma2_rn(xv, xv, ss2);
                }
            }
            const float ss = exchange(xn0 + 8 * qd, s_nrm, ss2.x + ss2.y, it, ok);
            float n32 = sqrtf(ss);
            bool wide = !(ss > 1.0e-30f && ss < 1.0e30f);  // squares under/overflow: the norm in fp64
            uint16_t n16 = f16_bits_sat(n32);
            bool nclose = false;
            if (!wide && n32 > 0.0f && n32 < 65504.0f) {
                const float dn = __half2float(__float2half_rd(n32));
                const float up = __half2float(__float2half_ru(n32));
                nclose = dn != up && fabsf(n32 - 0.5f * (dn + up)) <= 1.0e-6f * n32;
            }
            // rare: the norm in fp64, one vector at a time by the whole warp
            unsigned nb = __ballot_sync(TQ_FULL_MASK, valid && (wide || nclose));
            while (nb) {
                const int src = __ffs(nb) - 1;
                nb &= nb - 1;
                double s = 0.0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const double xv = (double)xel(xb, 32 * qd + src, 4 * lane + k);
                    s = fma(xv, xv, s);
                }
                s = warp_sum(s);
                if (lane == src) {
                    const double nd = sqrt(s);
                    if (wide) n32 = (float)nd;
                    n16 = __half_as_ushort(__double2half(fmin(nd, 65504.0)));
                }
            }
            const float inv_n = n32 > 0.0f ? 1.0f / n32 : 0.0f;
            const float sc = RHT ? p.inv_sqrt_d * inv_n : inv_n;
            const int64_t slot = valid ? slot_of(v) : -1;

            if (ok && !mbar_wait_bounded(a1full0 + 8 * tb, (uint32_t)((it / NB1) & 1), kWaitLimitNs, p.err,
                                         kErrQuantWait))
                ok = false;
            ok = __all_sync(TQ_FULL_MASK, ok);
            tc_fence_after_sync();
            const uint32_t acc = lane_addr + (uint32_t)(128 * tb);
            // keys: R goes to its own columns once the previous tile's S r
            // product has read them (waited for just before the first store)
            bool rfree = !PROD || it == 0;
            float gam2 = 0.0f;
#pragma unroll 1
            for (int ch = 0; ch < (ok ? C::kNch : 0); ++ch) {
                const int c0 = cbase + 32 * ch;  // first coordinate of the chunk
                // The chunk's packed stream (CHB bits) is built as CHB / 8 byte
                // chains, each taking its 8 bits from the highest down (short
                // dependency chains). The two 16-coordinate groups are done one
                // after the other (the upper first), each ending with its
                // re-decisions and, for keys, its R hi/lo halves written over
                // its own 16 columns (hi pairs in the first 8, lo in the last 8).
                constexpr int NBY = CHB / 8;
                uint32_t by[NBY];
#pragma unroll
                for (int q = 0; q < NBY; ++q) by[q] = 0u;
#pragma unroll
                for (int grp = 1; grp >= 0; --grp) {
                    float raw[16];
                    tmem_ld16(acc + (uint32_t)(c0 + 16 * grp), raw);
                    tmem_ld_wait();
                    uint32_t hv[PROD ? 16 : 1];
                    float2 g2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
                    float gm[4] = {INFINITY, INFINITY, INFINITY, INFINITY};  // distance partials
                    float r_odd = 0.0f;  // the residual of coordinate j + 1 while j is formed
#pragma unroll
                    for (int jl = 15; jl >= 0; --jl) {
                        const int j = 16 * grp + jl;  // coordinate in the chunk
                        // its group (folds to a constant in the unrolled loop)
                        const bool g1 = !TWO || jl < 8;
                        const int W = g1 ? CB : CB2, NB = g1 ? NPB : NPB2, H = g1 ? HX : HX2;
                        const float* tpw = g1 ? tp : tp2;
                        const float* cw = g1 ? p.cb.c : p.cb2.c;
                        const float yv = raw[jl] * sc;
                        const float ay = fabsf(yv);
                        float dv[NPB > 0 ? NPB : 1];
#pragma unroll
                        for (int b = 0; b < NPB; ++b)
                            if (b < NB) dv[b] = ay - tpw[b];
                        // code bits W-1 (sign) .. 0, most significant first
#pragma unroll
                        for (int b = CB - 1; b >= 0; --b) {
                            if (b >= W) continue;
                            uint32_t t = fx(yv);
                            if (b < W - 1) {
#pragma unroll
                                for (int q = 1; q <= NPB; ++q)
                                    if (q <= NB && (q % (1 << b)) == 0) t ^= fx(dv[q - 1]);
                            }
                            const int bit = bit_of(j) + b;  // stream bit in the chunk
                            by[bit >> 3] = shf_in(by[bit >> 3], t);
                        }
                        // distance to the nearest boundary (|y| itself: the boundary at 0)
                        float& g = gm[jl & 3];
                        if (NB == 0) {
                            g = fminf(g, ay);
                        } else {
                            g = min3f(g, ay, fabsf(dv[0]));
#pragma unroll
                            for (int b = 1; b < NPB; b += 2) {
                                if (b >= NB) continue;
                                g = (b + 1 < NB) ? min3f(g, fabsf(dv[b]), fabsf(dv[b + 1])) : fminf(g, fabsf(dv[b]));
                            }
                        }
                        if constexpr (PROD) {
                            // residual: |y| - c(cell) with the sign of y
                            float cpos = cw[H];
#pragma unroll
                            for (int b = 0; b < NPB; ++b)
                                if (b < NB) cpos = dv[b] >= 0.0f ? cw[H + 1 + b] : cpos;
                            const float rj = __uint_as_float(fx(ay - cpos) ^ (fx(yv) & 0x80000000u));
                            if (jl & 1) {
                                r_odd = rj;
                            } else {
                                const float2 rv = make_float2(rj, r_odd);
                                g2[(jl >> 1) & 1] = __ffma2_rn(rv, rv, g2[(jl >> 1) & 1]);
                                const float2 hi = make_float2(__uint_as_float(fx(rj) & 0xFFFF0000u),
                                                              __uint_as_float(fx(r_odd) & 0xFFFF0000u));
                                const float2 lo = __ffma2_rn(hi, make_float2(-1.0f, -1.0f), rv);  // r - hi, exact
                                hv[jl / 2] = __byte_perm(fx(rj), fx(r_odd), 0x7632u);
                                const __nv_bfloat162 lb = __floats2bfloat162_rn(lo.x, lo.y);
                                hv[8 + jl / 2] = *reinterpret_cast<const uint32_t*>(&lb);
                            }
                        }
                    }
                    float gsum = (g2[0].x + g2[0].y) + (g2[1].x + g2[1].y);
                    const float gmin = fminf(fminf(gm[0], gm[1]), fminf(gm[2], gm[3]));

                    // ---- rare: fp64 re-decision of coordinates near a boundary ----
                    unsigned need = __ballot_sync(TQ_FULL_MASK, valid && !(gmin >= p.guard));
                    // which coordinates of the group, from its columns one at a
                    // time (they still hold y)
                    uint32_t myflags = 0u;
                    if (need) {
                        float yy[16];
                        tmem_ld16(acc + (uint32_t)(c0 + 16 * grp), yy);
                        tmem_ld_wait();
#pragma unroll
                        for (int jl = 0; jl < 16; ++jl) {
                            const bool g1 = !TWO || jl < 8;
                            const float ay = fabsf(yy[jl] * sc);
                            float dm = ay;
#pragma unroll
                            for (int b = 0; b < NPB; ++b)
                                if (b < (g1 ? NPB : NPB2)) dm = fminf(dm, fabsf(ay - (g1 ? tp[b] : tp2[b])));
                            if (!(dm >= p.guard)) myflags |= 1u << jl;
                        }
                    }
                    while (need) {
                        const int src = __ffs(need) - 1;
                        need &= need - 1;
                        uint32_t fm = __shfl_sync(TQ_FULL_MASK, myflags, src);
                        const int row = 32 * qd + src;
                        while (fm) {
                            const int jl = __ffs(fm) - 1;
                            fm &= fm - 1;
                            const int j = 16 * grp + jl;
                            const int i = c0 + j;  // output coordinate
                            double part = 0.0, s2 = 0.0;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int e = 4 * lane + k;
                                const double xv = (double)xel(xb, row, e);
                                s2 = fma(xv, xv, s2);
                                if constexpr (RHT) {
                                    const double t = (double)s_sgn[e] * xv;
                                    part += (__popc(i & e) & 1) ? -t : t;
                                } else {
                                    part = fma(p.pi64[(size_t)i * kQuD + e], xv, part);
                                }
                            }
                            part = warp_sum(part);
                            const double nrow = sqrt(warp_sum(s2));
                            double y64 = 0.0;
                            if (nrow > 0.0) y64 = RHT ? part / (sqrt((double)kQuD) * nrow) : part / nrow;
                            if (lane == src) {
                                const bool g1 = !TWO || jl < 8;
                                const Codebook& bk = g1 ? p.cb : p.cb2;
                                const int W = g1 ? CB : CB2;
                                int k = 0;
#pragma unroll
                                for (int t = 0; t < L - 1; ++t)
                                    if (t < (g1 ? L : L2) - 1) k += (y64 >= bk.t64[t]) ? 1 : 0;
                                // the code bits in the byte chains (held inverted)
                                const int sb = bit_of(j), q0 = sb >> 3, o = sb & 7;
                                const uint32_t wm = (1u << W) - 1u;
                                const uint32_t inv = ~(uint32_t)k & wm;
#pragma unroll
                                for (int q = 0; q < NBY; ++q) {
                                    if (q == q0) by[q] = (by[q] & ~(wm << o)) | (inv << o);
                                    if (q == q0 + 1 && o + W > 8) by[q] = (by[q] & ~(wm >> (8 - o))) | (inv >> (8 - o));
                                }
                                if constexpr (PROD) {
                                    // the new residual into its hi/lo halves; gamma^2
                                    // corrected by the change of this coordinate's square
                                    const float nv = (float)(y64 - (double)bk.c[k]);
                                    const int hw = jl >> 1, sh16 = 16 * (jl & 1);
                                    uint32_t hiw = 0u, low = 0u;
#pragma unroll
                                    for (int jj = 0; jj < 8; ++jj)
                                        if (jj == hw) {
                                            hiw = hv[jj];
                                            low = hv[8 + jj];
                                        }
                                    const float old = __uint_as_float(((hiw >> sh16) & 0xFFFFu) << 16) +
                                                      __uint_as_float(((low >> sh16) & 0xFFFFu) << 16);
                                    gsum += nv * nv - old * old;
                                    const float nhi = __uint_as_float(fx(nv) & 0xFFFF0000u);
                                    const uint32_t lob = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(nv - nhi));
                                    hiw = (hiw & ~(0xFFFFu << sh16)) | ((fx(nv) >> 16) << sh16);
                                    low = (low & ~(0xFFFFu << sh16)) | (lob << sh16);
#pragma unroll
                                    for (int jj = 0; jj < 8; ++jj)
                                        if (jj == hw) {
                                            hv[jj] = hiw;
                                            hv[8 + jj] = low;
                                        }
                                }
                            }
                        }
                    }
                    if constexpr (PROD) {
                        gam2 += gsum;
                        if (!rfree) {
                            if (!mbar_wait_bounded(a2full, (uint32_t)((it - 1) & 1), kWaitLimitNs, p.err,
                                                   kErrQuantWait))
                                ok = false;
                            ok = __all_sync(TQ_FULL_MASK, ok);
                            tc_fence_after_sync();
                            rfree = true;
                        }
                        if (ok) tmem_st16(lane_addr + kColR + (uint32_t)(c0 + 16 * grp), hv);
                    }
                }
                // the appended bits were the inverted code bits
                if (slot >= 0) {
                    unsigned char* rowp = p.codes + slot * (int64_t)p.code_stride + (c0 / 32) * NBY;
                    if constexpr (NBY % 4 == 0) {
                        uint32_t* dst = reinterpret_cast<uint32_t*>(rowp);
#pragma unroll
                        for (int w = 0; w < NBY / 4; ++w)
                            dst[w] = ~((by[4 * w] & 0xFFu) | ((by[4 * w + 1] & 0xFFu) << 8) |
                                       ((by[4 * w + 2] & 0xFFu) << 16) | (by[4 * w + 3] << 24));
                    } else {  // an odd CB + CB2: 2-byte units (the chunk starts on an even byte)
                        uint16_t* dst = reinterpret_cast<uint16_t*>(rowp);
#pragma unroll
                        for (int w = 0; w < NBY / 2; ++w)
                            dst[w] = (uint16_t)~((by[2 * w] & 0xFFu) | ((by[2 * w + 1] & 0xFFu) << 8));
                    }
                }
            }
            if constexpr (PROD) tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0 && ok) {
                mbar_arrive(tfree0 + 8 * tb);  // the rotation accumulator was read
                mbar_arrive(xfree0 + 8 * xb);  // the staged input was read (norm and re-decisions)
                if constexpr (PROD) mbar_arrive(rfull);
            }
            if constexpr (PROD) {
                const float g2 = exchange(xg0 + 8 * qd, s_gam, gam2, it, ok);
                if (ok && h == 0 && slot >= 0) p.rnorm[slot] = f16_bits_sat(sqrtf(g2));
            }
            if (ok && h == 0 && slot >= 0) p.norm[slot] = n16;
            return ok;
        };

        // ---------------- phase 2 (keys): the signs of S r ----------------
        auto phase2 = [&](int64_t it) -> bool {
            const int64_t tile = blockIdx.x + it * gridDim.x;
            const int64_t v = tile * kQuVec + r;
            if (!mbar_wait_bounded(a2full, (uint32_t)(it & 1), kWaitLimitNs, p.err, kErrQuantWait)) return false;
            tc_fence_after_sync();
            const int64_t slot = v < p.n ? slot_of(v) : -1;
            const uint32_t zacc = lane_addr + kColZ;
#pragma unroll 1
            for (int ch = 0; ch < C::kNch; ++ch) {
                const int c0 = cbase + 32 * ch;
                uint32_t raw[32];
                tmem_ld32(zacc + (uint32_t)c0, raw);
                tmem_ld_wait();
                // bit j set: (S r)_j < 0 (sign bit); z_j = [(S r)_j >= 0]; four byte chains
                uint32_t bq[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int j = 31; j >= 0; --j) bq[j >> 3] = shf_in(bq[j >> 3], raw[j]);
                const uint32_t w = (bq[0] & 0xFFu) | ((bq[1] & 0xFFu) << 8) | ((bq[2] & 0xFFu) << 16) | (bq[3] << 24);
                if (slot >= 0) reinterpret_cast<uint32_t*>(p.signs + slot * (int64_t)p.sign_stride)[c0 / 32] = ~w;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(a2free);  // the S r accumulator was read
            return true;
        };

        bool ok = true;
        if (nmine > 0) ok = phase1(0);
        for (int64_t it = 0; ok && it < nmine; ++it) {
            if (it + 1 < nmine) ok = phase1(it + 1);
            if (!ok) break;
            if constexpr (PROD) ok = phase2(it);
            if (*abort_flag) ok = false;
        }
        if (!ok) *abort_flag = 1;
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the driver's tensor-map encoder, looked up once
inline EncodeTiled qu_encode_fn() {
    static EncodeTiled fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiled>(f);
        return (EncodeTiled) nullptr;
    }();
    return fn;
}

// the launch's parameters: the input as a 2-D bf16 tensor map (boxes of 64
// coordinates x 128 rows, 128-byte swizzle) and the operands
inline cudaError_t qu_params(const QuantParams& p, const void* w_umma, const void* s_umma, QuantUmmaParams* P) {
    EncodeTiled enc = qu_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    P->q = p;
    P->w_umma = w_umma;
    P->s_umma = s_umma;
    const cuuint64_t dims[2] = {(cuuint64_t)kQuD, (cuuint64_t)p.n};
    const cuuint64_t strides[1] = {(cuuint64_t)p.x_stride * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)kQuVec};
    const cuuint32_t estr[2] = {1u, 1u};
    if (enc(&P->tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

// the shapes every instantiation takes (bf16 input, d = 128, keys m = 128,
// 16-byte aligned rows)
inline bool qu_shape_ok(const QuantParams& p, int dtype) {
    return dtype == 1 && p.d == 128 && (p.m == 0 || p.m == 128) && p.n > 0 && p.n < (1ll << 31) - kQuVec &&
           ((uintptr_t)p.x % 16) == 0 && (p.x_stride * 2) % 16 == 0 && qu_encode_fn() != nullptr;
}

template <int CB, int CB2, bool PROD, bool RHT, int NP>
cudaError_t go_qu(const QuantUmmaParams& P, cudaStream_t s) {
    auto kern = quantize_umma_kernel<CB, CB2, PROD, RHT, NP>;
    constexpr size_t smem = qu_smem_bytes<NP>(RHT ? 1 : 3, PROD);
    static_assert(smem <= 227 * 1024 - 1024, "shared memory above the per-CTA limit");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles = (P.q.n + kQuVec - 1) / kQuVec;
    const int blocks = (int)(tiles < sms ? tiles : sms);
    kern<<<blocks, QuCfg<NP>::kThreads, smem, s>>>(P);
    return cudaGetLastError();
}

}  // namespace tqk
