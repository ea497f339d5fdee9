// Quantize-on-append for d = m = 128 with the two dense contractions on the
// tensor cores (mma.sync m16n8k16, bf16 x bf16 -> f32).
//
// Follows the same steps as quantize.cuh (A2A TurboQuant explainer, "Stage 1"
// and "Stage 2"; Qiita TurboQuant article, "Rotate, then quantize" and "One
// more stage so attention does not break"): n = ||x||, y = Pi x / n, Lloyd-Max
// codes, and for keys r = y - c[idx], gamma = ||r||, z = [S r >= 0].
//
// A warp quantizes a tile of 16 vectors. In the "quad layout" used throughout,
// thread (g, c) = (lane / 4, lane % 4) owns coordinates 32c .. 32c+31 of tile
// rows g and g+8, so its codes fill whole 32-bit words of the packed stream
// and its 32 sign bits are one word: no cross-lane packing.
//  * dense rotation: Y = X Pi^T on the tensor cores, Pi^T split into three
//    bf16 limbs (about 24 bits), X exact in bf16 or split into three limbs
//    when it is fp32; the host stores the B operand in fragment order with the
//    output columns permuted so that the accumulators land in the quad layout
//    and the K order permuted so that each thread builds its A fragments in
//    registers from its own coordinates (k-step kk takes 32c + 4kk .. +3);
//  * RHT: the Walsh-Hadamard butterflies run in registers in the quad layout
//    (strides 1..16 inside a thread, 32 and 64 across the quad);
//  * S r: R split into bf16 hi/lo (16 bits) against S, which is exact in bf16.
// Codes are decided from the fp32 y by comparing |y| with the positive
// boundaries (the codebook is symmetric), and any coordinate within `guard`
// of a boundary is re-decided from an fp64 dot product, as in quantize.cuh.
#pragma once

#include "common.cuh"
#include "pipeline.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kQmWarps = 4;  // warps per CTA
constexpr int kQmSmemLimit = 227 * 1024;

template <typename XT, bool RHT>
constexpr int qm_warps() { return kQmWarps; }

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16_zfill(uint32_t smem_addr, const void* gptr, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr), "l"(gptr), "r"(valid ? 16 : 0));
}

// packed fp32 pairs (one instruction for two lanes of a register pair);
// each lane rounds exactly as the scalar operation would
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
// (a + b, a - b) for both lanes of the pairs, bit-identical to the scalar forms
__device__ __forceinline__ void butterfly2(float& a0, float& a1, float& b0, float& b1) {
    const float2 a = f2(a0, a1), b = f2(b0, b1);
    const float2 s = __fadd2_rn(a, b);
    const float2 d = __ffma2_rn(b, f2(-1.0f, -1.0f), a);  // a - b, one rounding
    a0 = s.x;
    a1 = s.y;
    b0 = d.x;
    b1 = d.y;
}

// two floats -> bf16 pair (lo half = a), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Raw staging tile of 16 input rows: element i of row r at byte
// r * RSB + (i + SK * (i / 32)) * sizeof(XT). The per-32-element skew puts
// the four blocks of a quad in different banks.
template <typename XT>
struct QmStage {
    static constexpr int ESZ = sizeof(XT);
    static constexpr int SK = 16 / ESZ;                    // 16-byte skew per block
    static constexpr int RSB = (128 + 4 * SK) * ESZ;       // 320 (bf16) / 576 (fp32)
    static constexpr int BYTES = 16 * RSB;
    __device__ static int off(int r, int i) { return r * RSB + (i + SK * (i >> 5)) * ESZ; }
};

template <typename XT>
__device__ __forceinline__ float stage_at(const unsigned char* t, int r, int i) {
    if constexpr (sizeof(XT) == 4) return *reinterpret_cast<const float*>(t + QmStage<XT>::off(r, i));
    else return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(t + QmStage<XT>::off(r, i))) << 16);
}

template <typename XT>
struct QmSmem {
    static constexpr int WARP_BYTES = 2 * QmStage<XT>::BYTES;  // double-buffered staging
};

// Cell of one coordinate against a symmetric codebook of CBX bits (the
// positive boundaries only, see below): returns the code, sets dmin (the
// distance of |y| to the nearest boundary) and, for keys, cpos = the centroid
// magnitude of the cell.
template <int CBX, bool PROD>
__device__ __forceinline__ int qm_cell(const Codebook& cbk, float yv, float& dmin, float& cpos) {
    constexpr int LX = 1 << CBX, HX = LX / 2;
    const float av = fabsf(yv);
    int k = 0;
    dmin = av;
    cpos = cbk.c[HX];
#pragma unroll
    for (int t = HX; t < LX - 1; ++t) {
        const bool ge = av >= cbk.t[t];
        k += ge ? 1 : 0;
        if (PROD) cpos = ge ? cbk.c[t + 1] : cpos;
        dmin = fminf(dmin, fabsf(av - cbk.t[t]));
    }
    return yv >= 0.0f ? HX + k : HX - 1 - k;
}

// bit offset of coordinate j (0..31) in a thread's run of codes: CB bits each,
// or (fractional rates, CB2 != CB) CB bits when j % 16 < 8 and CB2 otherwise
template <int CB, int CB2>
__device__ __forceinline__ constexpr int qm_bit(int j) {
    return CB2 == CB ? CB * j
                     : (j >> 4) * 8 * (CB + CB2) + ((j & 15) < 8 ? (j & 7) * CB : 8 * CB + (j & 7) * CB2);
}

template <typename XT, int CB, bool PROD, bool RHT, int CB2 = CB>
__global__ void __launch_bounds__(kQmWarps * 32, 3) quantize_mma_kernel(const __grid_constant__ QuantParams p) {
    constexpr int D = 128;
    constexpr int L = 1 << CB;
    constexpr bool TWO = CB2 != CB;  // two channel groups (fractional rate)
    constexpr int NLX = (!RHT && sizeof(XT) == 4) ? 3 : 1;  // limbs of X for the dense GEMM
    constexpr int NW = qm_warps<XT, RHT>();
    using S = QmSmem<XT>;
    using ST = QmStage<XT>;
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int B1_BYTES = RHT ? 0 : 3 * 8 * 16 * 32 * 8;
    constexpr int B2_BYTES = PROD ? 8 * 16 * 32 * 8 : 0;
    const uint2* b1 = reinterpret_cast<const uint2*>(smem);
    const uint2* b2 = reinterpret_cast<const uint2*>(smem + B1_BYTES);
    __shared__ float s_cent[kMaxLevels];
    __shared__ float s_cent2[TWO ? kMaxLevels : 1];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    unsigned char* xs_base = smem + B1_BYTES + B2_BYTES + warp * S::WARP_BYTES;  // 2 raw staging tiles
    const uint32_t xs_s = (uint32_t)__cvta_generic_to_shared(xs_base);

    // ---- CTA set-up: the B fragments by bulk copies on an mbarrier that each
    // warp waits on only before its first tensor-core product (so the load
    // overlaps the first tile's norm, rotation and bucketize), and the
    // centroids into shared memory ----
    __shared__ __align__(8) uint64_t s_fbar;
    const uint32_t fbar = (uint32_t)__cvta_generic_to_shared(&s_fbar);
    constexpr int FRAG_BYTES = B1_BYTES + B2_BYTES;
    if (threadIdx.x == 0) {
        mbar_init(fbar, 1);
        mbar_init_fence();
        if constexpr (FRAG_BYTES > 0) {
            const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(smem);
            mbar_arrive_expect_tx(fbar, FRAG_BYTES);
            constexpr int CH = 16384;
            for (int o = 0; o < B1_BYTES; o += CH)
                bulk_g2s(s0 + o, reinterpret_cast<const unsigned char*>(p.pi_frag) + o, CH, fbar);
            for (int o = 0; o < B2_BYTES; o += CH)
                bulk_g2s(s0 + B1_BYTES + o, reinterpret_cast<const unsigned char*>(p.s_frag) + o, CH, fbar);
        }
    }
    if (threadIdx.x < kMaxLevels) s_cent[threadIdx.x] = p.cb.c[threadIdx.x];
    if constexpr (TWO)
        if (threadIdx.x < kMaxLevels) s_cent2[threadIdx.x] = p.cb2.c[threadIdx.x];
    bool frag_ready = FRAG_BYTES == 0, failed = false;
    // warp-uniform: true once the fragments are in shared memory
    auto frags = [&]() -> bool {
        if (!frag_ready) {
            const bool ok = mbar_wait_bounded(fbar, 0, kWaitLimitNs, p.err, kErrQuantWait);
            frag_ready = __all_sync(TQ_FULL_MASK, ok);
        }
        return frag_ready;
    };
    // RHT signs of this thread's coordinates 32c .. 32c+31 as one mask (bit j
    // set: coordinate 32c + j is negated), applied by flipping float sign bits
    uint32_t sgm = 0u;
    if constexpr (RHT) {
#pragma unroll
        for (int j = 0; j < 32; ++j) sgm |= (p.sgn[32 * c + j] < 0.0f ? 1u : 0u) << j;
    }

    const int64_t ntiles = (p.n + 15) / 16;
    const int64_t tstep = (int64_t)gridDim.x * NW;
    // stage 16 input rows of `tile` into buffer `buf` with cp.async (zero-filled past n)
    auto stage = [&](int64_t tile, int buf) {
        constexpr int EPC = 16 / ST::ESZ;  // elements per 16-byte chunk
        constexpr int CPR = D / EPC;       // chunks per row
#pragma unroll
        for (int q = lane; q < 16 * CPR; q += 32) {
            const int r = q / CPR, ch = q % CPR;
            const int64_t v = tile * 16 + r;
            const bool ok = v < p.n;
            const XT* src = reinterpret_cast<const XT*>(p.x) + (ok ? v : 0) * p.x_stride + ch * EPC;
            cp_async16_zfill(xs_s + buf * ST::BYTES + ST::off(r, ch * EPC), src, ok);
        }
    };
    int64_t tile = (int64_t)blockIdx.x * NW + warp;
    if (tile < ntiles) stage(tile, 0);
    asm volatile("cp.async.commit_group;\n" ::);  // group: first tile
    __syncthreads();  // centroids and the barrier's initialisation, for every warp
    for (int it = 0; tile < ntiles && !failed; tile += tstep, ++it) {
        const int64_t v0 = tile * 16;
        unsigned char* xs = xs_base + (it & 1) * ST::BYTES;
        if (tile + tstep < ntiles) stage(tile + tstep, (it + 1) & 1);  // prefetch the next tile
        asm volatile("cp.async.commit_group;\n" ::);
        asm volatile("cp.async.wait_group 1;\n" ::);
        __syncwarp();

        // ---- quad layout: x of rows g, g+8, coordinates 32c..32c+31 ----
        float y[2][32];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const uint4* src = reinterpret_cast<const uint4*>(xs + ST::off(g + 8 * rr, 32 * c));
            if constexpr (sizeof(XT) == 4) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 t = src[k];
                    y[rr][4 * k] = __uint_as_float(t.x);
                    y[rr][4 * k + 1] = __uint_as_float(t.y);
                    y[rr][4 * k + 2] = __uint_as_float(t.z);
                    y[rr][4 * k + 3] = __uint_as_float(t.w);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 t = src[k];
                    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        y[rr][8 * k + 2 * e] = bf16_lo(w[e]);
                        y[rr][8 * k + 2 * e + 1] = bf16_hi(w[e]);
                    }
                }
            }
        }
        // norms (quad reduction), with a rescaled retry when squares under/overflow
        float n32[2], inv_n[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float2 s2v = f2(0.0f, 0.0f);  // even and odd coordinates, packed
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float2 v = f2(y[rr][j], y[rr][j + 1]);
                s2v = __ffma2_rn(v, v, s2v);
            }
            float ss = s2v.x + s2v.y;
            ss += __shfl_xor_sync(TQ_FULL_MASK, ss, 1);
            ss += __shfl_xor_sync(TQ_FULL_MASK, ss, 2);
            n32[rr] = sqrtf(ss);
            const bool odd = !(ss > 1.0e-30f && ss < 1.0e30f);
            if (__any_sync(TQ_FULL_MASK, odd)) {
                float amax = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(y[rr][j]));
                amax = fmaxf(amax, __shfl_xor_sync(TQ_FULL_MASK, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(TQ_FULL_MASK, amax, 2));
                float s2 = 0.0f;
                const float ia = amax > 0.0f ? 1.0f / amax : 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j) s2 = fmaf(y[rr][j] * ia, y[rr][j] * ia, s2);
                s2 += __shfl_xor_sync(TQ_FULL_MASK, s2, 1);
                s2 += __shfl_xor_sync(TQ_FULL_MASK, s2, 2);
                if (odd) n32[rr] = amax * sqrtf(s2);
            }
            inv_n[rr] = n32[rr] > 0.0f ? 1.0f / n32[rr] : 0.0f;
        }

        // ---- rotation ----
        if constexpr (RHT) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    y[rr][j] = __int_as_float(__float_as_int(y[rr][j]) ^ (int)((sgm << (31 - j)) & 0x80000000u));
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int j = 0; j < 32; j += 2) {  // stride 1: within a pair
                    const float a = y[rr][j], b = y[rr][j + 1];
                    y[rr][j] = a + b;
                    y[rr][j + 1] = a - b;
                }
#pragma unroll
            for (int h = 2; h < 32; h <<= 1)  // strides 2..16: two butterflies per packed pair
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                    for (int j = 0; j < 32; j += 2)
                        if ((j & h) == 0) butterfly2(y[rr][j], y[rr][j + 1], y[rr][j + h], y[rr][j + h + 1]);
#pragma unroll
            for (int hb = 1; hb < 4; hb <<= 1) {
                const float sgn_self = (c & hb) ? -1.0f : 1.0f;  // upper half: o - y
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float o0 = __shfl_xor_sync(TQ_FULL_MASK, y[rr][j], hb);
                        const float o1 = __shfl_xor_sync(TQ_FULL_MASK, y[rr][j + 1], hb);
                        const float2 r = __ffma2_rn(f2(sgn_self, sgn_self), f2(y[rr][j], y[rr][j + 1]), f2(o0, o1));
                        y[rr][j] = r.x;
                        y[rr][j + 1] = r.y;
                    }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const float sc = p.inv_sqrt_d * inv_n[rr];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float2 r = __fmul2_rn(f2(y[rr][j], y[rr][j + 1]), f2(sc, sc));
                    y[rr][j] = r.x;
                    y[rr][j + 1] = r.y;
                }
            }
        } else {
            if (!frags()) {  // the fragments never landed (the error word says so)
                failed = true;
                break;
            }
            // two passes of 8 n-tiles (output coordinates 32c + 0..15, then
            // 32c + 16..31) keep the live accumulators at 32 registers; the
            // first pass's results wait in `first` while y still feeds pass 2
            float first[8][4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float acc[8][4];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    // A fragments from this thread's own coordinates 32c + 4kk .. +3
                    // of rows g (slots 0, 2) and g + 8 (slots 1, 3), as bf16 limbs
                    uint32_t a[NLX][4];
#pragma unroll
                    for (int sl = 0; sl < 4; ++sl) {
                        const float v0 = y[sl & 1][4 * kk + (sl & 2)], v1 = y[sl & 1][4 * kk + (sl & 2) + 1];
                        const uint32_t h1 = pack_bf16(v0, v1);
                        a[0][sl] = h1;
                        if constexpr (NLX == 3) {
                            const float r0 = v0 - bf16_lo(h1), r1 = v1 - bf16_hi(h1);
                            const uint32_t h2 = pack_bf16(r0, r1);
                            a[1][sl] = h2;
                            a[2][sl] = pack_bf16(r0 - bf16_lo(h2), r1 - bf16_hi(h2));
                        }
                    }
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        const int ng = 8 * half + nt;
                        const uint2 f1 = b1[((0 * 8 + kk) * 16 + ng) * 32 + lane];
                        const uint2 f2 = b1[((1 * 8 + kk) * 16 + ng) * 32 + lane];
                        const uint2 f3 = b1[((2 * 8 + kk) * 16 + ng) * 32 + lane];
                        mma16816_bf16(acc[nt], a[0][0], a[0][1], a[0][2], a[0][3], f1.x, f1.y);
                        mma16816_bf16(acc[nt], a[0][0], a[0][1], a[0][2], a[0][3], f2.x, f2.y);
                        mma16816_bf16(acc[nt], a[0][0], a[0][1], a[0][2], a[0][3], f3.x, f3.y);
                        if constexpr (NLX == 3) {
                            mma16816_bf16(acc[nt], a[1][0], a[1][1], a[1][2], a[1][3], f1.x, f1.y);
                            mma16816_bf16(acc[nt], a[1][0], a[1][1], a[1][2], a[1][3], f2.x, f2.y);
                            mma16816_bf16(acc[nt], a[2][0], a[2][1], a[2][2], a[2][3], f1.x, f1.y);
                        }
                    }
                }
                if (half == 0) {
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) first[nt][e] = acc[nt][e];
                } else {
                    // accumulator (row g / g+8, column 2c+e of n-tile nt) = coordinate 32c + 2nt + e
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        y[0][2 * nt] = first[nt][0] * inv_n[0];
                        y[0][2 * nt + 1] = first[nt][1] * inv_n[0];
                        y[1][2 * nt] = first[nt][2] * inv_n[1];
                        y[1][2 * nt + 1] = first[nt][3] * inv_n[1];
                        y[0][16 + 2 * nt] = acc[nt][0] * inv_n[0];
                        y[0][16 + 2 * nt + 1] = acc[nt][1] * inv_n[0];
                        y[1][16 + 2 * nt] = acc[nt][2] * inv_n[1];
                        y[1][16 + 2 * nt + 1] = acc[nt][3] * inv_n[1];
                    }
                }
            }
        }

        // ---- bucketize with guard band; for keys y becomes the residual ----
        // idx = #{t_j <= y}: with the symmetric codebook (t_{H-1} = 0, positive
        // boundaries t_H..t_{L-2}) and k = #{positive t <= |y|},
        // idx = H + k for y >= 0 and H - 1 - k for y < 0 (exact ties are inside
        // the guard band and decided in fp64 below).
        uint32_t idxw[2][4];
        uint32_t flag[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            flag[rr] = 0u;
#pragma unroll
            for (int w = 0; w < 4; ++w) idxw[rr][w] = 0u;
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float yv = y[rr][j];
                const bool sec = TWO && (j & 15) >= 8;  // second channel group
                const int w = sec ? CB2 : CB;
                float dmin, cpos;
                const int idx = sec ? qm_cell<CB2, PROD>(p.cb2, yv, dmin, cpos) : qm_cell<CB, PROD>(p.cb, yv, dmin, cpos);
                if (!(dmin >= p.guard)) flag[rr] |= 1u << j;
                if (PROD) y[rr][j] = yv >= 0.0f ? yv - cpos : yv + cpos;
                const int bit = qm_bit<CB, CB2>(j);
                idxw[rr][bit >> 5] |= (uint32_t)idx << (bit & 31);
                if ((bit & 31) + w > 32) idxw[rr][(bit >> 5) + 1] |= (uint32_t)idx >> (32 - (bit & 31));
            }
        }
        if (v0 + g >= p.n) flag[0] = 0u;
        if (v0 + g + 8 >= p.n) flag[1] = 0u;

        // fp16 norms; near an fp16 rounding midpoint they are re-rounded from fp64
        uint16_t n16[2];
        bool nclose[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            n16[rr] = f16_bits_sat(n32[rr]);
            nclose[rr] = false;
            if (n32[rr] > 0.0f && n32[rr] < 65504.0f) {
                const float dn = __half2float(__float2half_rd(n32[rr]));
                const float up = __half2float(__float2half_ru(n32[rr]));
                nclose[rr] = dn != up && fabsf(n32[rr] - 0.5f * (dn + up)) <= 1.0e-6f * n32[rr];
            }
        }

        // ---- fp64 re-decision of flagged coordinates (warp-cooperative, rare) ----
        if (__any_sync(TQ_FULL_MASK, (flag[0] | flag[1]) != 0u || nclose[0] || nclose[1])) {
            // warp-uniform condition: the quad sums below shuffle over the full warp
            if (__any_sync(TQ_FULL_MASK, nclose[0] || nclose[1])) {
#pragma unroll 1
                for (int rr = 0; rr < 2; ++rr) {
                    double s = 0.0;
#pragma unroll 8
                    for (int j = 0; j < 32; ++j) {
                        const double xv = (double)stage_at<XT>(xs, g + 8 * rr, 32 * c + j);
                        s = fma(xv, xv, s);
                    }
                    s += __shfl_xor_sync(TQ_FULL_MASK, s, 1);
                    s += __shfl_xor_sync(TQ_FULL_MASK, s, 2);
                    if (nclose[rr]) n16[rr] = __half_as_ushort(__double2half(fmin(sqrt(s), 65504.0)));
                }
            }
            while (true) {
                const unsigned bal = __ballot_sync(TQ_FULL_MASK, (flag[0] | flag[1]) != 0u);
                if (!bal) break;
                const int src = __ffs(bal) - 1;
                const int rr_src = __shfl_sync(TQ_FULL_MASK, flag[0] ? 0 : 1, src);
                const int j_src = __shfl_sync(TQ_FULL_MASK, __ffs(flag[0] ? flag[0] : flag[1]) - 1, src);
                const int row = (src >> 2) + 8 * rr_src;
                const int i = 32 * (src & 3) + j_src;
                double part = 0.0, s2 = 0.0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int e = 4 * lane + k;
                    const double xv = (double)stage_at<XT>(xs, row, e);
                    s2 = fma(xv, xv, s2);
                    if constexpr (RHT) {
                        const double t = (double)p.sgn[e] * xv;
                        part += (__popc(i & e) & 1) ? -t : t;
                    } else {
                        part = fma(p.pi64[(size_t)i * D + e], xv, part);
                    }
                }
                part = warp_sum(part);
                const double nrow = sqrt(warp_sum(s2));
                double y64 = 0.0;
                if (nrow > 0.0) y64 = RHT ? part / (sqrt((double)D) * nrow) : part / nrow;
                if (lane == src) {
                    const bool sec = TWO && (j_src & 15) >= 8;
                    int k = 0;
                    if (sec) {
#pragma unroll
                        for (int t = 0; t < (1 << CB2) - 1; ++t) k += (y64 >= p.cb2.t64[t]) ? 1 : 0;
                    } else {
#pragma unroll
                        for (int t = 0; t < L - 1; ++t) k += (y64 >= p.cb.t64[t]) ? 1 : 0;
                    }
                    const float nv = PROD ? (float)y64 - (sec ? s_cent2[k] : s_cent[k]) : (float)y64;
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        if (rr != rr_src) continue;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (j != j_src) continue;
                            y[rr][j] = nv;
                            const int w = (TWO && (j & 15) >= 8) ? CB2 : CB;
                            const int bit = qm_bit<CB, CB2>(j);
                            const uint32_t m0 = ((1u << w) - 1u) << (bit & 31);
                            idxw[rr][bit >> 5] = (idxw[rr][bit >> 5] & ~m0) | ((uint32_t)k << (bit & 31));
                            if ((bit & 31) + w > 32) {
                                const int sh = 32 - (bit & 31);
                                const uint32_t m1 = ((1u << w) - 1u) >> sh;
                                idxw[rr][(bit >> 5) + 1] = (idxw[rr][(bit >> 5) + 1] & ~m1) | ((uint32_t)k >> sh);
                            }
                        }
                        flag[rr] &= ~(1u << j_src);
                    }
                }
            }
        }

        // ---- slots of rows g and g+8 ----
        int64_t slot[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int64_t v = v0 + g + 8 * rr;
            int64_t s = -1;
            if (v < p.n) {
                if (p.dst_slot) {
                    s = p.dst_slot[v];
                } else if (p.append_pos) {
                    const int32_t pos = p.append_pos[v / p.heads];
                    s = (pos >= 0 && pos < p.capacity) ? v * p.capacity + pos : -1;
                } else {
                    s = p.slot0 + v;
                }
                if (s >= p.total_slots) s = -1;
            }
            slot[rr] = s;
        }
        // ---- store codes and norms ----
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            if (slot[rr] < 0) continue;
            if constexpr (TWO) {
                // this thread's 16 (CB + CB2) bits are CB + CB2 half-words from
                // half-word c (CB + CB2) of the slot (half-word aligned for odd c)
                uint16_t* d16 = reinterpret_cast<uint16_t*>(p.codes + slot[rr] * (int64_t)p.code_stride) + c * (CB + CB2);
#pragma unroll
                for (int h = 0; h < CB + CB2; ++h) d16[h] = (uint16_t)(idxw[rr][h >> 1] >> (16 * (h & 1)));
                if (c == 0) p.norm[slot[rr]] = n16[rr];
                continue;
            }
            uint32_t* dst = reinterpret_cast<uint32_t*>(p.codes + slot[rr] * (int64_t)p.code_stride) + CB * c;
            if constexpr (CB == 2) {
                *reinterpret_cast<uint2*>(dst) = make_uint2(idxw[rr][0], idxw[rr][1]);
            } else if constexpr (CB == 4) {
                *reinterpret_cast<uint4*>(dst) = make_uint4(idxw[rr][0], idxw[rr][1], idxw[rr][2], idxw[rr][3]);
            } else {
#pragma unroll
                for (int w = 0; w < CB; ++w) dst[w] = idxw[rr][w];
            }
            if (c == 0) p.norm[slot[rr]] = n16[rr];
        }

        if constexpr (PROD) {
            // gamma = ||r|| (y holds r); the S r GEMM takes R as bf16 hi/lo A
            // fragments straight from this thread's coordinates
            float gam[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                float2 g2v = f2(0.0f, 0.0f);  // even and odd coordinates, packed
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float2 v = f2(y[rr][j], y[rr][j + 1]);
                    g2v = __ffma2_rn(v, v, g2v);
                }
                float g2 = g2v.x + g2v.y;
                g2 += __shfl_xor_sync(TQ_FULL_MASK, g2, 1);
                g2 += __shfl_xor_sync(TQ_FULL_MASK, g2, 2);
                gam[rr] = sqrtf(g2);
            }
            if (!frags()) {
                failed = true;
                break;
            }
            // R as bf16 hi/lo A fragments for all 8 k-steps (64 registers; y is
            // dead afterwards), then two passes of 8 n-tiles (16 sign bits
            // each) so that only 32 accumulators are live at a time
            uint32_t fr[8][2][4];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
#pragma unroll
                for (int sl = 0; sl < 4; ++sl) {
                    const float v0 = y[sl & 1][4 * kk + (sl & 2)], v1 = y[sl & 1][4 * kk + (sl & 2) + 1];
                    const uint32_t h = pack_bf16(v0, v1);
                    fr[kk][0][sl] = h;
                    fr[kk][1][sl] = pack_bf16(v0 - bf16_lo(h), v1 - bf16_hi(h));
                }
            uint32_t sw[2] = {0u, 0u};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float z[8][4];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) z[nt][e] = 0.0f;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        const uint2 f = b2[(kk * 16 + 8 * half + nt) * 32 + lane];
                        mma16816_bf16(z[nt], fr[kk][0][0], fr[kk][0][1], fr[kk][0][2], fr[kk][0][3], f.x, f.y);
                        mma16816_bf16(z[nt], fr[kk][1][0], fr[kk][1][1], fr[kk][1][2], fr[kk][1][3], f.x, f.y);
                    }
                }
                // accumulator (row g / g+8, column 2c+e of n-tile nt) = sign bit 2nt + e of the thread's word
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const int bit = 2 * (8 * half + nt);
                    sw[0] |= (z[nt][0] >= 0.0f ? 1u : 0u) << bit;
                    sw[0] |= (z[nt][1] >= 0.0f ? 1u : 0u) << (bit + 1);
                    sw[1] |= (z[nt][2] >= 0.0f ? 1u : 0u) << bit;
                    sw[1] |= (z[nt][3] >= 0.0f ? 1u : 0u) << (bit + 1);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                if (slot[rr] < 0) continue;
                reinterpret_cast<uint32_t*>(p.signs + slot[rr] * (int64_t)p.sign_stride)[c] = sw[rr];
                if (c == 0) p.rnorm[slot[rr]] = f16_bits_sat(gam[rr]);
            }
        }
        __syncwarp();
    }
    asm volatile("cp.async.wait_group 0;\n" ::);
    // a warp with no tile (or that gave up) still lets the fragment copies land
    // before the CTA's shared memory is released
    if (!frag_ready) mbar_wait_bounded(fbar, 0, kWaitLimitNs, p.err, kErrQuantWait);
}

template <typename XT, int CB, bool PROD, bool RHT>
constexpr size_t quantize_mma_smem() {
    return (RHT ? 0 : 3 * 8 * 16 * 32 * 8) + (PROD ? 8 * 16 * 32 * 8 : 0) +
           (size_t)qm_warps<XT, RHT>() * QmSmem<XT>::WARP_BYTES;
}

// One launch: a persistent grid of at most (SMs x resident CTAs) CTAs, each
// warp taking tiles of 16 vectors.
template <typename XT, int CB, bool PROD, bool RHT, int CB2 = CB>
cudaError_t launch_quantize_mma_t(const QuantParams& p, cudaStream_t s) {
    if (p.n <= 0) return cudaSuccess;
    auto kern = quantize_mma_kernel<XT, CB, PROD, RHT, CB2>;
    constexpr int NW = qm_warps<XT, RHT>();
    constexpr size_t smem = quantize_mma_smem<XT, CB, PROD, RHT>();
    static_assert(smem + 2 * kMaxLevels * sizeof(float) <= kQmSmemLimit, "shared memory above the per-CTA limit");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t tiles = (p.n + 15) / 16;
    int64_t blocks = (tiles + NW - 1) / NW;
    if (blocks > (int64_t)sms * per_sm) blocks = (int64_t)sms * per_sm;
    kern<<<(unsigned)blocks, NW * 32, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tqk
