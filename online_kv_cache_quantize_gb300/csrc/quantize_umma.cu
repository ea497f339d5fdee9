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
//  * TMA warp: tiled tensor copies of the 128-vector input tiles (16 boxes of
//    8 coordinates x 128 rows, so the tile lands in the no-swizzle K-major
//    core-matrix layout the MMA reads) into a ring of shared-memory buffers;
//  * MMA warp: the rotation MMAs of a tile into one of two TMEM buffers, and
//    (keys) the sign-sketch MMAs with A = R read from TMEM;
//  * epilogue warps: thread = vector (its TMEM lane), each of the NP warps of
//    a lane quarter takes 128 / NP coordinates. Phase 1: the norm from the
//    staged input, then per 32 coordinates the rotated values from TMEM,
//    codes by sign-bit arithmetic (below), the guard test, the residual, and
//    R hi/lo written back over the columns just read. Phase 2 (keys): the
//    signs of S r from TMEM.
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
#include <cuda.h>

#include "common.cuh"
#include "pipeline.cuh"
#include "tcgen05.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kQuVec = 128;        // vectors per tile (MMA M, TMEM lanes)
constexpr int kQuD = 128;          // coordinates (MMA N and K)
constexpr int kQuXBufs = 2;        // input tile buffers
constexpr uint32_t kQuTileBytes = kQuVec * kQuD * 2;  // 32 KB of bf16
constexpr uint32_t kQuBBytes = kQuD * kQuD * 2;       // one 128 x 128 bf16 operand

// epilogue warps per TMEM lane quarter (each takes 128 / kQuParts coordinates)
constexpr int kQuParts = 2;

struct QuantUmmaParams {
    CUtensorMap tmap;     // the input: 2-D bf16 [n][128] (row stride x_stride), box 8 x 128
    QuantParams q;
    const void* w_umma;   // rotation operand(s), 128 x 128 bf16 each, core-matrix layout
    const void* s_umma;   // S, 128 x 128 bf16, core-matrix layout (keys)
};

template <int NP>
struct QuCfg {
    static constexpr int kEpi = 4 * NP;             // epilogue warps
    static constexpr int kWarps = kEpi + 2;         // + TMA warp + MMA warp
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kCpt = kQuD / NP;          // coordinates per epilogue thread
    static constexpr int kNch = kCpt / 32;          // 32-coordinate chunks per thread
};

// bytes of dynamic shared memory: rotation limbs, S, input buffers, norm and
// gamma partials
template <int NP>
__host__ __device__ constexpr size_t qu_smem_bytes(int nlimb, bool prod) {
    return (size_t)nlimb * kQuBBytes + (prod ? kQuBBytes : 0) + (size_t)kQuXBufs * kQuTileBytes +
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

template <int CB, bool PROD, bool RHT, int NP>
__global__ void __launch_bounds__(QuCfg<NP>::kThreads, 1)
    quantize_umma_kernel(const __grid_constant__ QuantUmmaParams P) {
    using C = QuCfg<NP>;
    constexpr int NL = RHT ? 1 : 3;        // bf16 limbs of W
    constexpr int L = 1 << CB;             // cells
    constexpr int HX = L / 2;              // index of the first non-negative cell
    constexpr int NPB = HX - 1;            // positive boundaries t_1 .. t_NPB
    constexpr int WPC = CB;                // packed code words per 32-coordinate chunk
    const QuantParams& p = P.q;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
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
    __shared__ __align__(8) uint64_t s_a1full[2], s_rfull[2], s_a2full[2], s_tfree[2];
    __shared__ __align__(8) uint64_t s_xn[4], s_xg[4];  // partial-sum exchanges, one per lane quarter
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntiles = (p.n + kQuVec - 1) / kQuVec;
    const int64_t nmine = (int)blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    const uint32_t bfull = (uint32_t)__cvta_generic_to_shared(&s_bfull);
    const uint32_t xfull0 = (uint32_t)__cvta_generic_to_shared(&s_xfull[0]);
    const uint32_t xfree0 = (uint32_t)__cvta_generic_to_shared(&s_xfree[0]);
    const uint32_t a1full0 = (uint32_t)__cvta_generic_to_shared(&s_a1full[0]);
    const uint32_t rfull0 = (uint32_t)__cvta_generic_to_shared(&s_rfull[0]);
    const uint32_t a2full0 = (uint32_t)__cvta_generic_to_shared(&s_a2full[0]);
    const uint32_t tfree0 = (uint32_t)__cvta_generic_to_shared(&s_tfree[0]);
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
        for (int b = 0; b < 2; ++b) {
            mbar_init(a1full0 + 8 * b, 1);
            mbar_init(rfull0 + 8 * b, C::kEpi);
            mbar_init(a2full0 + 8 * b, 1);
            mbar_init(tfree0 + 8 * b, C::kEpi);
        }
        s_abort = 0;
        mbar_init_fence();
    }
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
#pragma unroll 1
                for (int j = 0; j < kQuD / 8; ++j)
                    tma_load_2d(dst + j * (kQuVec * 16), &P.tmap, 8 * j, (int)(tile * kQuVec), xfull0 + 8 * xb);
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
            // A = input tile: element (r, k) at (k/8)*2048 + (r/8)*128 + (r%8)*16 + (k%8)*2
            // (LBO 2048 along K, SBO 128 along M); a K = 16 step is 4096 bytes on
            const uint32_t x0 = (uint32_t)__cvta_generic_to_shared(sX);
            // B = W / S: element (n, k) at (n/8)*2048 + (k/8)*128 + (n%8)*16 + (k%8)*2
            const uint64_t db1 = umma_desc((uint32_t)__cvta_generic_to_shared(sB1), 128, 2048);
            const uint64_t db2 = umma_desc((uint32_t)__cvta_generic_to_shared(sB2), 128, 2048);
            int64_t last_commit = -1;  // tiles whose last MMA was committed
            auto rot = [&](int64_t it) -> bool {
                const int xb = (int)(it % kQuXBufs), tb = (int)(it & 1);
                if (!mbar_wait_bounded(xfull0 + 8 * xb, (uint32_t)((it / kQuXBufs) & 1), kWaitLimitNs, p.err,
                                       kErrQuantWait))
                    return false;
                // the TMEM buffer's previous tile is done with it: its sign
                // MMAs read R from it (keys), or its epilogue read it (values)
                if (it >= 2) {
                    const uint32_t par = (uint32_t)(((it - 2) >> 1) & 1);
                    if (!mbar_wait_bounded(PROD ? a2full0 + 8 * tb : tfree0 + 8 * tb, par, kWaitLimitNs, p.err,
                                           kErrQuantWait))
                        return false;
                }
                tc_fence_after_sync();
                const uint64_t da = umma_desc(x0 + xb * kQuTileBytes, 2048, 128);
                const uint32_t acc = tmem + (uint32_t)(256 * tb);
#pragma unroll
                for (int l = 0; l < NL; ++l)
#pragma unroll
                    for (int s = 0; s < kQuD / 16; ++s)
                        umma_f16(acc, da + (uint64_t)(s * (4096 >> 4)),
                                 db1 + (uint64_t)((l * kQuBBytes + s * 256) >> 4), idesc, l > 0 || s > 0);
                umma_commit(a1full0 + 8 * tb);
                umma_commit(xfree0 + 8 * xb);
                return true;
            };
            auto sgn = [&](int64_t it) -> bool {
                const int tb = (int)(it & 1);
                if (!mbar_wait_bounded(rfull0 + 8 * tb, (uint32_t)((it >> 1) & 1), kWaitLimitNs, p.err,
                                       kErrQuantWait))
                    return false;
                tc_fence_after_sync();
                // R of coordinates 32q .. 32q+31: hi halves in columns 32q .. 32q+15,
                // lo halves in 32q+16 .. 32q+31 (two per column)
                const uint32_t racc = tmem + (uint32_t)(256 * tb);
                const uint32_t zacc = racc + 128u;
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint64_t bd = db2 + (uint64_t)(((32 * q + 16 * e) / 8 * 128) >> 4);
                        umma_f16_ta(zacc, racc + 32u * q + 8u * e, bd, idesc, q > 0 || e > 0);
                        umma_f16_ta(zacc, racc + 32u * q + 16u + 8u * e, bd, idesc, true);
                    }
                umma_commit(a2full0 + 8 * tb);
                return true;
            };
            if (ok && nmine > 0) ok = rot(0);
            if (ok && nmine > 1) ok = rot(1);
            for (int64_t it = 0; ok && it < nmine; ++it) {
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                if constexpr (PROD) {
                    if (!(ok = sgn(it))) break;
                }
                last_commit = it;
                if (it + 2 < nmine && !(ok = rot(it + 2))) break;
            }
            if (!ok) *abort_flag = 1;
            // the MMAs in flight complete (bounded) before TMEM is released
            if (nmine > 0) {
                const int64_t lt = nmine - 1;
                if constexpr (PROD) {
                    if (last_commit >= 0)
                        mbar_wait_bounded(a2full0 + 8 * (int)(last_commit & 1), (uint32_t)((last_commit >> 1) & 1),
                                          kWaitLimitNs, p.err, kErrQuantWait);
                } else {
                    mbar_wait_bounded(a1full0 + 8 * (int)(lt & 1), (uint32_t)((lt >> 1) & 1), kWaitLimitNs, p.err,
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

        // positive boundaries (fp32) and the centroid magnitudes for keys
        float tp[NPB > 0 ? NPB : 1];
#pragma unroll
        for (int j = 0; j < NPB; ++j) tp[j] = p.cb.t[HX + j];

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
        auto xel = [&](int xb, int row, int k) -> float {  // staged input element as fp32
            const uint16_t b = *reinterpret_cast<const uint16_t*>(sX + (size_t)xb * kQuTileBytes + (k >> 3) * 2048 +
                                                                   (row >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
            return __uint_as_float((uint32_t)b << 16);
        };

        // ---------------- phase 1: norm, codes, residual ----------------
        auto phase1 = [&](int64_t it) -> bool {
            const int xb = (int)(it % kQuXBufs), tb = (int)(it & 1);
            const int64_t tile = blockIdx.x + it * gridDim.x;
            const int64_t v = tile * kQuVec + r;
            const bool valid = v < p.n;
            // a failed wait still takes part in both exchanges (so no partner
            // waits for an arrival that never comes), then reports failure
            bool ok = mbar_wait_bounded(xfull0 + 8 * xb, (uint32_t)((it / kQuXBufs) & 1), kWaitLimitNs, p.err,
                                        kErrQuantWait);
            // partial sum of squares over this thread's coordinates
            const unsigned char* xrow = sX + (size_t)xb * kQuTileBytes + (r >> 3) * 128 + (r & 7) * 16;
            float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < C::kCpt / 8; ++j) {
                const uint4 w = *reinterpret_cast<const uint4*>(xrow + (cbase / 8 + j) * 2048);
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
            if (valid && (wide || nclose)) {  // rare: this thread's vector in fp64
                double s = 0.0;
                for (int k = 0; k < kQuD; ++k) {
                    const double xv = (double)xel(xb, r, k);
                    s = fma(xv, xv, s);
                }
                const double nd = sqrt(s);
                if (wide) n32 = (float)nd;
                n16 = __half_as_ushort(__double2half(fmin(nd, 65504.0)));
            }
            const float inv_n = n32 > 0.0f ? 1.0f / n32 : 0.0f;
            const float sc = RHT ? p.inv_sqrt_d * inv_n : inv_n;
            const int64_t slot = valid ? slot_of(v) : -1;

            if (ok && !mbar_wait_bounded(a1full0 + 8 * tb, (uint32_t)((it >> 1) & 1), kWaitLimitNs, p.err,
                                         kErrQuantWait))
                ok = false;
            ok = __all_sync(TQ_FULL_MASK, ok);
            tc_fence_after_sync();
            const uint32_t acc = lane_addr + (uint32_t)(256 * tb);
            float gam2 = 0.0f;
#pragma unroll 1
            for (int ch = 0; ch < (ok ? C::kNch : 0); ++ch) {
                const int c0 = cbase + 32 * ch;  // first coordinate of the chunk
                uint32_t raw[32];
                tmem_ld32(acc + (uint32_t)c0, raw);
                tmem_ld_wait();
                float rr[32];
                uint32_t wd[WPC];
#pragma unroll
                for (int w = 0; w < WPC; ++w) wd[w] = 0u;
                float gmin = INFINITY;
                // the stream bits of the chunk, appended from the last one down
#pragma unroll
                for (int j = 31; j >= 0; --j) {
                    const float yv = __uint_as_float(raw[j]) * sc;
                    const float ay = fabsf(yv);
                    float dv[NPB > 0 ? NPB : 1];
#pragma unroll
                    for (int b = 0; b < NPB; ++b) dv[b] = ay - tp[b];
                    // code bits CB-1 (sign) .. 0, most significant first
#pragma unroll
                    for (int b = CB - 1; b >= 0; --b) {
                        uint32_t t = fx(yv);
                        if (b < CB - 1) {
#pragma unroll
                            for (int q = 1; q <= NPB; ++q)
                                if ((q % (1 << b)) == 0) t ^= fx(dv[q - 1]);
                        }
                        const int bit = CB * j + b;       // stream bit in the chunk
                        const int w = bit >> 5;
                        wd[w] = shf_in(wd[w], t);
                    }
                    // distance to the nearest boundary
                    float dm = ay;
#pragma unroll
                    for (int b = 0; b < NPB; b += 2) dm = (b + 1 < NPB) ? min3f(dm, fabsf(dv[b]), fabsf(dv[b + 1]))
                                                                        : fminf(dm, fabsf(dv[b]));
                    gmin = fminf(gmin, dm);
                    if constexpr (PROD) {
                        // residual: |y| - c(cell) with the sign of y
                        float cpos = p.cb.c[HX];
#pragma unroll
                        for (int b = 0; b < NPB; ++b) cpos = dv[b] >= 0.0f ? p.cb.c[HX + 1 + b] : cpos;
                        rr[j] = __uint_as_float(fx(ay - cpos) ^ (fx(yv) & 0x80000000u));
                    }
                }
                // the appended bits were the inverted code bits; a word of the
                // chunk stream is complete once 32 bits went in (chunk streams
                // are CB whole words)
#pragma unroll
                for (int w = 0; w < WPC; ++w) wd[w] = ~wd[w];

                // ---- rare: fp64 re-decision of coordinates near a boundary ----
                unsigned need = __ballot_sync(TQ_FULL_MASK, valid && !(gmin >= p.guard));
                if (need) tmem_ld32(acc + (uint32_t)c0, raw);  // y again (the columns still hold it)
                if (need) tmem_ld_wait();
                while (need) {
                    const int src = __ffs(need) - 1;
                    need &= need - 1;
                    uint32_t fm = 0u;
                    if (lane == src) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float ay = fabsf(__uint_as_float(raw[j]) * sc);
                            float dm = ay;
#pragma unroll
                            for (int b = 0; b < NPB; ++b) dm = fminf(dm, fabsf(ay - tp[b]));
                            if (!(dm >= p.guard)) fm |= 1u << j;
                        }
                    }
                    fm = __shfl_sync(TQ_FULL_MASK, fm, src);
                    const int row = 32 * qd + src;
                    while (fm) {
                        const int j = __ffs(fm) - 1;
                        fm &= fm - 1;
                        const int i = c0 + j;  // output coordinate
                        double part = 0.0, s2 = 0.0;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int e = 4 * lane + k;
                            const double xv = (double)xel(xb, row, e);
                            s2 = fma(xv, xv, s2);
                            if constexpr (RHT) {
                                const double t = (double)p.sgn[e] * xv;
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
                            int k = 0;
#pragma unroll
                            for (int t = 0; t < L - 1; ++t) k += (y64 >= p.cb.t64[t]) ? 1 : 0;
                            const int bit = CB * j;
                            const int w = bit >> 5, sh = bit & 31;
                            const uint32_t m0 = ((1u << CB) - 1u) << sh;
#pragma unroll
                            for (int ww = 0; ww < WPC; ++ww) {
                                if (ww == w) wd[ww] = (wd[ww] & ~m0) | ((uint32_t)k << sh);
                                if (ww == w + 1 && sh + CB > 32) {
                                    const uint32_t m1 = ((1u << CB) - 1u) >> (32 - sh);
                                    wd[ww] = (wd[ww] & ~m1) | ((uint32_t)k >> (32 - sh));
                                }
                            }
                            if constexpr (PROD) {
                                const float nv = (float)(y64 - (double)p.cb.c[k]);
#pragma unroll
                                for (int jj = 0; jj < 32; ++jj)
                                    if (jj == j) rr[jj] = nv;
                            }
                        }
                    }
                }
                // ---- store this chunk's codes ----
                if (slot >= 0) {
                    uint32_t* dst = reinterpret_cast<uint32_t*>(p.codes + slot * (int64_t)p.code_stride) + c0 / 32 * CB;
#pragma unroll
                    for (int w = 0; w < WPC; ++w) dst[w] = wd[w];
                }
                if constexpr (PROD) {
                    // gamma and R as bf16 hi (truncated) / lo (rounded) halves,
                    // written over the 32 columns just read
                    uint32_t hv[32];
                    float2 g2 = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float2 rv = make_float2(rr[j], rr[j + 1]);
                        g2 = __ffma2_rn(rv, rv, g2);
                        const float h0 = __uint_as_float(fx(rr[j]) & 0xFFFF0000u);
                        const float h1 = __uint_as_float(fx(rr[j + 1]) & 0xFFFF0000u);
                        const float2 lo = __ffma2_rn(make_float2(h0, h1), make_float2(-1.0f, -1.0f), rv);  // r - hi, exact
                        hv[j / 2] = __byte_perm(fx(rr[j]), fx(rr[j + 1]), 0x7632u);
                        const __nv_bfloat162 lb = __floats2bfloat162_rn(lo.x, lo.y);
                        hv[16 + j / 2] = *reinterpret_cast<const uint32_t*>(&lb);
                    }
                    gam2 += g2.x + g2.y;
                    tmem_st32(acc + (uint32_t)c0, hv);
                }
            }
            if constexpr (PROD) tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0 && ok) {
                mbar_arrive(xfree0 + 8 * xb);  // the input tile was read (norm and re-decisions)
                mbar_arrive(PROD ? rfull0 + 8 * tb : tfree0 + 8 * tb);
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
            const int tb = (int)(it & 1);
            const int64_t tile = blockIdx.x + it * gridDim.x;
            const int64_t v = tile * kQuVec + r;
            if (!mbar_wait_bounded(a2full0 + 8 * tb, (uint32_t)((it >> 1) & 1), kWaitLimitNs, p.err, kErrQuantWait))
                return false;
            tc_fence_after_sync();
            const int64_t slot = v < p.n ? slot_of(v) : -1;
            const uint32_t zacc = lane_addr + (uint32_t)(256 * tb + 128);
#pragma unroll 1
            for (int ch = 0; ch < C::kNch; ++ch) {
                const int c0 = cbase + 32 * ch;
                uint32_t raw[32];
                tmem_ld32(zacc + (uint32_t)c0, raw);
                tmem_ld_wait();
                uint32_t w = 0u;
#pragma unroll
                for (int j = 31; j >= 0; --j) w = shf_in(w, raw[j]);
                // bit j set: (S r)_j < 0 (sign bit); z_j = [(S r)_j >= 0]
                if (slot >= 0) reinterpret_cast<uint32_t*>(p.signs + slot * (int64_t)p.sign_stride)[c0 / 32] = ~w;
            }
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

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
    }
    return fn;
}

template <int CB, bool PROD, bool RHT, int NP>
cudaError_t go_qu(const QuantUmmaParams& P, cudaStream_t s) {
    auto kern = quantize_umma_kernel<CB, PROD, RHT, NP>;
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

}  // namespace

bool quantize_umma_supported(const QuantParams& p, int dtype, int code_bits) {
    return dtype == 1 && p.d == 128 && (p.m == 0 || p.m == 128) && p.code_bits2 == 0 && code_bits >= 1 &&
           code_bits <= (p.m == 128 ? 3 : 4) && p.n > 0 && p.n < (1ll << 31) - kQuVec && ((uintptr_t)p.x % 16) == 0 &&
           (p.x_stride * 2) % 16 == 0 && encode_fn() != nullptr;
}

cudaError_t launch_quantize_umma(const QuantParams& p, const void* w_umma, const void* s_umma, int rht, int prod,
                                 int code_bits, cudaStream_t s) {
    if (p.n <= 0) return cudaSuccess;
    EncodeTiled enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    QuantUmmaParams P;
    P.q = p;
    P.w_umma = w_umma;
    P.s_umma = s_umma;
    const cuuint64_t dims[2] = {(cuuint64_t)kQuD, (cuuint64_t)p.n};
    const cuuint64_t strides[1] = {(cuuint64_t)p.x_stride * 2};
    const cuuint32_t box[2] = {8u, (cuuint32_t)kQuVec};
    const cuuint32_t estr[2] = {1u, 1u};
    if (enc(&P.tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    constexpr int NP = kQuParts;
    // keys (PROD) have 1..3 code bits (2..4 bits with the sign bit), values 1..4
#define TQ_QU_MSE(CBV) \
    if (code_bits == CBV && !prod) return rht ? go_qu<CBV, false, true, NP>(P, s) : go_qu<CBV, false, false, NP>(P, s);
#define TQ_QU_PROD(CBV) \
    if (code_bits == CBV && prod) return rht ? go_qu<CBV, true, true, NP>(P, s) : go_qu<CBV, true, false, NP>(P, s);
    TQ_QU_MSE(1)
    TQ_QU_MSE(2)
    TQ_QU_MSE(3)
    TQ_QU_MSE(4)
    TQ_QU_PROD(1)
    TQ_QU_PROD(2)
    TQ_QU_PROD(3)
#undef TQ_QU_MSE
#undef TQ_QU_PROD
    return cudaErrorNotSupported;
}

}  // namespace tqk
