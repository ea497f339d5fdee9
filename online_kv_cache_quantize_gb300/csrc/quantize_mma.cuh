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
//    output columns permuted so that the accumulators land in the quad layout;
//  * RHT: the Walsh-Hadamard butterflies run in registers in the quad layout
//    (strides 1..16 inside a thread, 32 and 64 across the quad);
//  * S r: R split into bf16 hi/lo (16 bits) against S, which is exact in bf16.
// Codes are decided from the fp32 y, and any coordinate within `guard` of a
// boundary is re-decided from an fp64 dot product, as in quantize.cuh.
#pragma once

#include "common.cuh"
#include "tq_launch.h"

namespace tqk {

constexpr int kQmWarps = 4;
constexpr int kQmRowWords = 68;  // 128 bf16 + 8 pad = 272 B per smem row (conflict-free quads)

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bf16_bits(float v) { return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// bf16 pair (lo half = a, hi half = b)
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) { return bf16_bits(a) | (bf16_bits(b) << 16); }

// fp32 staging tile: coordinate i of row r at r*144 + i + 4*(i/32); the skew
// puts the four 32-coordinate blocks of a quad in different banks
__device__ __forceinline__ int xpos(int r, int i) { return r * 144 + i + ((i >> 5) << 2); }

template <int NLIMB_X>
struct QmSmem {
    // per warp: fp32 copy of the tile (for norms, RHT and the fp64 path) and
    // bf16 operand tiles (X limbs for the dense GEMM, then R hi/lo)
    static constexpr int XF_BYTES = 16 * 144 * 4;                     // fp32 rows, see xpos()
    static constexpr int AT = NLIMB_X > 2 ? NLIMB_X : 2;              // operand tiles
    static constexpr int AT_BYTES = AT * 16 * kQmRowWords * 4;
    static constexpr int WARP_BYTES = XF_BYTES + AT_BYTES;
};

template <typename XT, int CB, bool PROD, bool RHT>
__global__ void __launch_bounds__(kQmWarps * 32) quantize_mma_kernel(const __grid_constant__ QuantParams p) {
    constexpr int D = 128;
    constexpr int L = 1 << CB;
    constexpr int NLX = (!RHT && sizeof(XT) == 4) ? 3 : 1;  // limbs of X for the dense GEMM
    using S = QmSmem<NLX>;
    extern __shared__ __align__(16) unsigned char smem[];
    const uint2* b1 = reinterpret_cast<const uint2*>(smem);                      // dense: 3 limbs
    const int b1_bytes = RHT ? 0 : 3 * 8 * 16 * 32 * 8;
    const uint2* b2 = reinterpret_cast<const uint2*>(smem + b1_bytes);           // PROD: S fragments
    const int b2_bytes = PROD ? 8 * 16 * 32 * 8 : 0;
    unsigned char* wbase = smem + b1_bytes + b2_bytes;
    __shared__ float s_cent[kMaxLevels];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    unsigned char* wsm = wbase + warp * S::WARP_BYTES;
    float* xf = reinterpret_cast<float*>(wsm);                     // [16][144], see xpos()
    uint32_t* at = reinterpret_cast<uint32_t*>(wsm + S::XF_BYTES);  // [AT][16][68]

    // ---- CTA set-up: B fragments and centroids into shared memory ----
    {
        const uint4* src1 = reinterpret_cast<const uint4*>(p.pi_frag);
        uint4* dst1 = reinterpret_cast<uint4*>(smem);
        for (int i = threadIdx.x; i < b1_bytes / 16; i += blockDim.x) dst1[i] = src1[i];
        const uint4* src2 = reinterpret_cast<const uint4*>(p.s_frag);
        uint4* dst2 = reinterpret_cast<uint4*>(smem + b1_bytes);
        for (int i = threadIdx.x; i < b2_bytes / 16; i += blockDim.x) dst2[i] = src2[i];
        if (threadIdx.x < kMaxLevels) s_cent[threadIdx.x] = p.cb.c[threadIdx.x];
    }
    float sg[32];
    if constexpr (RHT) {
#pragma unroll
        for (int j = 0; j < 32; ++j) sg[j] = p.sgn[32 * c + j];
    }
    __syncthreads();

    const int64_t ntiles = (p.n + 15) / 16;
    for (int64_t tile = (int64_t)blockIdx.x * kQmWarps + warp; tile < ntiles; tile += (int64_t)gridDim.x * kQmWarps) {
        const int64_t v0 = tile * 16;
        // ---- stage X (16 rows) as fp32 in shared memory ----
        {
            constexpr int EPC = 16 / sizeof(XT);  // elements per 16-byte chunk
            constexpr int CPR = D / EPC;          // chunks per row
            for (int q = lane; q < 16 * CPR; q += 32) {
                const int r = q / CPR, ch = q % CPR;
                const int64_t v = v0 + r;
                float* dst = xf + xpos(r, ch * EPC);
                if (v < p.n) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(reinterpret_cast<const XT*>(p.x) + v * p.x_stride + ch * EPC);
                    if constexpr (sizeof(XT) == 4) {
                        *reinterpret_cast<uint4*>(dst) = raw;
                    } else {
                        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            dst[2 * k] = __uint_as_float(w[k] << 16);
                            dst[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
                        }
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < EPC; ++k) dst[k] = 0.0f;
                }
            }
        }
        __syncwarp();

        // ---- quad layout: x of rows g, g+8, coordinates 32c..32c+31 ----
        float y[2][32];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const float4* src = reinterpret_cast<const float4*>(xf + xpos(g + 8 * rr, 32 * c));
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 t = src[k];
                y[rr][4 * k] = t.x;
                y[rr][4 * k + 1] = t.y;
                y[rr][4 * k + 2] = t.z;
                y[rr][4 * k + 3] = t.w;
            }
        }
        // norms (quad reduction), with a rescaled retry when squares under/overflow
        float n32[2], inv_n[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float ss = 0.0f;
#pragma unroll
            for (int j = 0; j < 32; ++j) ss = fmaf(y[rr][j], y[rr][j], ss);
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
                for (int j = 0; j < 32; ++j) y[rr][j] *= sg[j];
#pragma unroll
            for (int h = 1; h < 32; h <<= 1)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if ((j & h) == 0) {
                            const float a = y[rr][j], b = y[rr][j + h];
                            y[rr][j] = a + b;
                            y[rr][j + h] = a - b;
                        }
#pragma unroll
            for (int hb = 1; hb < 4; hb <<= 1) {
                const bool upper = (c & hb) != 0;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float o = __shfl_xor_sync(TQ_FULL_MASK, y[rr][j], hb);
                        y[rr][j] = upper ? (o - y[rr][j]) : (y[rr][j] + o);
                    }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const float sc = p.inv_sqrt_d * inv_n[rr];
#pragma unroll
                for (int j = 0; j < 32; ++j) y[rr][j] *= sc;
            }
        } else {
            // X limbs -> bf16 operand tiles (natural coordinate order)
            for (int q = lane; q < 16 * 64; q += 32) {
                const int r = q >> 6, w = q & 63;
                const float a = xf[xpos(r, 2 * w)], b = xf[xpos(r, 2 * w + 1)];
                if constexpr (NLX == 1) {
                    at[r * kQmRowWords + w] = pack_bf16(a, b);
                } else {
                    const float a1 = __bfloat162float(__float2bfloat16_rn(a)), b1v = __bfloat162float(__float2bfloat16_rn(b));
                    const float a2 = __bfloat162float(__float2bfloat16_rn(a - a1));
                    const float b2v = __bfloat162float(__float2bfloat16_rn(b - b1v));
                    at[r * kQmRowWords + w] = pack_bf16(a1, b1v);
                    at[16 * kQmRowWords + r * kQmRowWords + w] = pack_bf16(a2, b2v);
                    at[32 * kQmRowWords + r * kQmRowWords + w] = pack_bf16(a - a1 - a2, b - b1v - b2v);
                }
            }
            __syncwarp();
            float acc[16][4];
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
#pragma unroll 1
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t a[NLX][4];
#pragma unroll
                for (int l = 0; l < NLX; ++l) {
                    const uint32_t* t = at + l * 16 * kQmRowWords;
                    a[l][0] = t[g * kQmRowWords + 8 * kk + c];
                    a[l][1] = t[(g + 8) * kQmRowWords + 8 * kk + c];
                    a[l][2] = t[g * kQmRowWords + 8 * kk + 4 + c];
                    a[l][3] = t[(g + 8) * kQmRowWords + 8 * kk + 4 + c];
                }
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    const uint2 f1 = b1[((0 * 8 + kk) * 16 + nt) * 32 + lane];
                    const uint2 f2 = b1[((1 * 8 + kk) * 16 + nt) * 32 + lane];
                    const uint2 f3 = b1[((2 * 8 + kk) * 16 + nt) * 32 + lane];
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
            // accumulator (row g / g+8, column 2c+e of n-tile nt) = coordinate 32c + 2nt + e
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                y[0][2 * nt] = acc[nt][0] * inv_n[0];
                y[0][2 * nt + 1] = acc[nt][1] * inv_n[0];
                y[1][2 * nt] = acc[nt][2] * inv_n[1];
                y[1][2 * nt + 1] = acc[nt][3] * inv_n[1];
            }
        }

        // ---- bucketize with guard band ----
        uint32_t idxw[2][4];  // packed codes: 32 coordinates x CB bits = CB words per row
        uint32_t flag[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            flag[rr] = 0u;
#pragma unroll
            for (int w = 0; w < 4; ++w) idxw[rr][w] = 0u;
        }
        const bool rowok0 = v0 + g < p.n, rowok1 = v0 + g + 8 < p.n;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                int k = 0;
                float dmin = 3.0e38f;
#pragma unroll
                for (int t = 0; t < L - 1; ++t) {
                    k += (y[rr][j] >= p.cb.t[t]) ? 1 : 0;
                    dmin = fminf(dmin, fabsf(y[rr][j] - p.cb.t[t]));
                }
                if (!(dmin >= p.guard)) flag[rr] |= 1u << j;
                const int bit = CB * j;
                idxw[rr][bit >> 5] |= (uint32_t)k << (bit & 31);
                if ((bit & 31) + CB > 32) idxw[rr][(bit >> 5) + 1] |= (uint32_t)k >> (32 - (bit & 31));
            }
        }
        if (!rowok0) flag[0] = 0u;
        if (!rowok1) flag[1] = 0u;

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

        // ---- fp64 re-decision of flagged coordinates (warp-cooperative) ----
        if (__any_sync(TQ_FULL_MASK, (flag[0] | flag[1]) != 0u || nclose[0] || nclose[1])) {
            // fp64 norms of the 16 rows: lane l sums coordinates 4l..4l+3 of each row
            double n64[2] = {0.0, 0.0};
#pragma unroll 1
            for (int r = 0; r < 16; ++r) {
                double s = 0.0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const double xv = (double)xf[xpos(r, 4 * lane + k)];
                    s = fma(xv, xv, s);
                }
                s = warp_sum(s);
                if (r == g) n64[0] = sqrt(s);
                if (r == g + 8) n64[1] = sqrt(s);
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
                if (nclose[rr]) n16[rr] = __half_as_ushort(__double2half(fmin(n64[rr], 65504.0)));
            while (true) {
                const unsigned bal = __ballot_sync(TQ_FULL_MASK, (flag[0] | flag[1]) != 0u);
                if (!bal) break;
                const int src = __ffs(bal) - 1;
                const int rr_src = __shfl_sync(TQ_FULL_MASK, flag[0] ? 0 : 1, src);
                const int j_src = __shfl_sync(TQ_FULL_MASK, __ffs(flag[0] ? flag[0] : flag[1]) - 1, src);
                const int row = (src >> 2) + 8 * rr_src;
                const int i = 32 * (src & 3) + j_src;
                double part = 0.0;
                if constexpr (RHT) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int e = 4 * lane + k;
                        const double t = (double)p.sgn[e] * (double)xf[xpos(row, e)];
                        part += (__popc(i & e) & 1) ? -t : t;
                    }
                } else {
                    const double* prow = p.pi64 + (size_t)i * D;
#pragma unroll
                    for (int k = 0; k < 4; ++k) part = fma(prow[4 * lane + k], (double)xf[xpos(row, 4 * lane + k)], part);
                }
                part = warp_sum(part);
                double nrow = 0.0;
                {
                    double s = 0.0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const double xv = (double)xf[xpos(row, 4 * lane + k)];
                        s = fma(xv, xv, s);
                    }
                    nrow = sqrt(warp_sum(s));
                }
                double y64 = 0.0;
                if (nrow > 0.0) y64 = RHT ? part / (sqrt((double)D) * nrow) : part / nrow;
                if (lane == src) {
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        if (rr != rr_src) continue;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (j != j_src) continue;
                            int k = 0;
#pragma unroll
                            for (int t = 0; t < L - 1; ++t) k += (y64 >= p.cb.t64[t]) ? 1 : 0;
                            y[rr][j] = (float)y64;
                            const int bit = CB * j;
                            const uint32_t m0 = ((1u << CB) - 1u) << (bit & 31);
                            idxw[rr][bit >> 5] = (idxw[rr][bit >> 5] & ~m0) | ((uint32_t)k << (bit & 31));
                            if ((bit & 31) + CB > 32) {
                                const int sh = 32 - (bit & 31);
                                const uint32_t m1 = ((1u << CB) - 1u) >> sh;
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
            uint32_t* dst = reinterpret_cast<uint32_t*>(p.codes + slot[rr] * (int64_t)p.code_stride) + CB * c;
#pragma unroll
            for (int w = 0; w < CB; ++w) dst[w] = idxw[rr][w];
            if (c == 0) p.norm[slot[rr]] = n16[rr];
        }

        if constexpr (PROD) {
            // residual, gamma, and R as bf16 hi/lo tiles for the S r GEMM
            float gam[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                float g2 = 0.0f;
                uint32_t* th = at + (g + 8 * rr) * kQmRowWords + 16 * c;
                uint32_t* tl = th + 16 * kQmRowWords;
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const int bit0 = CB * j, bit1 = CB * (j + 1);
                    const uint32_t k0 = ((bit0 & 31) + CB <= 32 ? (idxw[rr][bit0 >> 5] >> (bit0 & 31))
                                                                 : __funnelshift_r(idxw[rr][bit0 >> 5], idxw[rr][(bit0 >> 5) + 1], bit0 & 31)) & (L - 1);
                    const uint32_t k1 = ((bit1 & 31) + CB <= 32 ? (idxw[rr][bit1 >> 5] >> (bit1 & 31))
                                                                 : __funnelshift_r(idxw[rr][bit1 >> 5], idxw[rr][(bit1 >> 5) + 1], bit1 & 31)) & (L - 1);
                    const float r0 = y[rr][j] - s_cent[k0], r1 = y[rr][j + 1] - s_cent[k1];
                    g2 = fmaf(r0, r0, fmaf(r1, r1, g2));
                    const float h0 = __bfloat162float(__float2bfloat16_rn(r0));
                    const float h1 = __bfloat162float(__float2bfloat16_rn(r1));
                    th[j >> 1] = pack_bf16(h0, h1);
                    tl[j >> 1] = pack_bf16(r0 - h0, r1 - h1);
                }
                g2 += __shfl_xor_sync(TQ_FULL_MASK, g2, 1);
                g2 += __shfl_xor_sync(TQ_FULL_MASK, g2, 2);
                gam[rr] = sqrtf(g2);
            }
            __syncwarp();
            float z[16][4];
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) z[nt][e] = 0.0f;
#pragma unroll 1
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t a[2][4];
#pragma unroll
                for (int l = 0; l < 2; ++l) {
                    const uint32_t* t = at + l * 16 * kQmRowWords;
                    a[l][0] = t[g * kQmRowWords + 8 * kk + c];
                    a[l][1] = t[(g + 8) * kQmRowWords + 8 * kk + c];
                    a[l][2] = t[g * kQmRowWords + 8 * kk + 4 + c];
                    a[l][3] = t[(g + 8) * kQmRowWords + 8 * kk + 4 + c];
                }
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    const uint2 f = b2[(kk * 16 + nt) * 32 + lane];
                    mma16816_bf16(z[nt], a[0][0], a[0][1], a[0][2], a[0][3], f.x, f.y);
                    mma16816_bf16(z[nt], a[1][0], a[1][1], a[1][2], a[1][3], f.x, f.y);
                }
            }
            uint32_t sw[2] = {0u, 0u};
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                sw[0] |= (z[nt][0] >= 0.0f ? 1u : 0u) << (2 * nt);
                sw[0] |= (z[nt][1] >= 0.0f ? 1u : 0u) << (2 * nt + 1);
                sw[1] |= (z[nt][2] >= 0.0f ? 1u : 0u) << (2 * nt);
                sw[1] |= (z[nt][3] >= 0.0f ? 1u : 0u) << (2 * nt + 1);
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
}

template <typename XT, int CB, bool PROD, bool RHT>
size_t quantize_mma_smem() {
    constexpr int NLX = (!RHT && sizeof(XT) == 4) ? 3 : 1;
    return (RHT ? 0 : 3 * 8 * 16 * 32 * 8) + (PROD ? 8 * 16 * 32 * 8 : 0) + (size_t)kQmWarps * QmSmem<NLX>::WARP_BYTES;
}

}  // namespace tqk
