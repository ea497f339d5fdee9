// Quantize-on-append for a few vectors at a time (the decode step's new
// token of every KV head): one CTA role of 128 threads per vector, thread i
// owns coordinate i (d = 128; keys have m = 128 sign rows).
//
// Same steps as quantize.cuh (A2A TurboQuant explainer, "Stage 1" and
// "Stage 2"; Qiita TurboQuant article, "Rotate, then quantize" and "One more
// stage so attention does not break"): n = ||x||, y = Pi x / n, Lloyd-Max
// codes, and for keys r = y - c[idx], gamma = ||r||, z = [S r >= 0]. Spread
// over 128 threads, every step is a few dependent instructions, so a vector
// costs a few microseconds of latency instead of the serial chain of one
// warp working through a 16-row tile.
//
// Precision as in quantize.cuh: y in fp32 (RHT by butterflies, dense rotation
// as an fp32 dot product), any coordinate within `guard` of a boundary
// re-decided from an fp64 dot product, the fp16 norm re-rounded from fp64
// near a rounding midpoint; S r as an fp32 dot product of each sign row.
#pragma once

#include "common.cuh"
#include "tq_launch.h"

namespace tqk {

// threads of a CTA of the decode step's prep launch (one query row or one
// appended vector per CTA)
constexpr int kStepThreads = 128;

// shared memory of one CTA of that launch, whichever its role
struct StepSmem {
    uint4 s[16 * 128];  // S as bf16, 16-byte unit (q, j) = S[j][8q .. 8q+7] at q * 128 + j
    float x[128];       // the input, fp32
    __align__(16) float y[128];  // butterfly exchange, then the residual r (append) or q' (query)
    float qp[128];      // query: q' = Pi q
    float u[128];       // query: u = S q'
    __align__(16) float part[4][128];  // dense rotation: the four warps' partial sums of Pi x
    float cent[kMaxLevels];
    float cent2[kMaxLevels];  // the second channel group's centroids (two-width caches)
    float red[4];
    double red64[4];
    uint32_t cw[16];    // packed codes: at most 4 bits x 128 coordinates
    int fsel;           // the flagged coordinate being re-decided
};

// barrier 1 over the 128 threads of the CTA
__device__ __forceinline__ void step_sync() { asm volatile("bar.sync 1, 128;\n" ::: "memory"); }

// true in every thread when v is true in any of the 128 threads
__device__ __forceinline__ bool step_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

// sums over the 128 threads in a fixed order (the same value in every thread)
__device__ __forceinline__ float step_sum(float v, StepSmem& s) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) s.red[threadIdx.x >> 5] = v;
    step_sync();
    const float r = (s.red[0] + s.red[1]) + (s.red[2] + s.red[3]);
    step_sync();
    return r;
}
__device__ __forceinline__ double step_sum64(double v, StepSmem& s) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) s.red64[threadIdx.x >> 5] = v;
    step_sync();
    const double r = (s.red64[0] + s.red64[1]) + (s.red64[2] + s.red64[3]);
    step_sync();
    return r;
}
__device__ __forceinline__ float step_max(float v, StepSmem& s) {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) s.red[threadIdx.x >> 5] = v;
    step_sync();
    const float r = fmaxf(fmaxf(s.red[0], s.red[1]), fmaxf(s.red[2], s.red[3]));
    step_sync();
    return r;
}

// Starts the copy of S (m = d = 128, bf16, unit layout above) into s.s:
// sixteen 16-byte cp.async per thread, one commit group. The caller waits
// (cp.async.wait_group 0) and then synchronises before reading s.s.
__device__ __forceinline__ void stage_s(const uint16_t* s16, StepSmem& s) {
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(s.s);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const int unit = u * kStepThreads + (int)threadIdx.x;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst + 16 * unit),
                     "l"(reinterpret_cast<const uint4*>(s16) + unit)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// (S v)_j for j = threadIdx.x: row j of the staged S (exact bf16 -> fp32)
// against v in shared memory, as four interleaved partial sums (coordinates
// 2q and 2q + 1 of each quarter of a 16-byte unit), added at the end
__device__ __forceinline__ float s_row_dot(const StepSmem& s, const float* v) {
    const int j = threadIdx.x;
    float z0 = 0.0f, z1 = 0.0f, z2 = 0.0f, z3 = 0.0f;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const uint4 sr = s.s[q * kStepThreads + j];
        const float4 r0 = *reinterpret_cast<const float4*>(v + 8 * q);
        const float4 r1 = *reinterpret_cast<const float4*>(v + 8 * q + 4);
        z0 = fmaf(__uint_as_float(sr.x << 16), r0.x, z0);
        z0 = fmaf(__uint_as_float(sr.x & 0xffff0000u), r0.y, z0);
        z1 = fmaf(__uint_as_float(sr.y << 16), r0.z, z1);
        z1 = fmaf(__uint_as_float(sr.y & 0xffff0000u), r0.w, z1);
        z2 = fmaf(__uint_as_float(sr.z << 16), r1.x, z2);
        z2 = fmaf(__uint_as_float(sr.z & 0xffff0000u), r1.y, z2);
        z3 = fmaf(__uint_as_float(sr.w << 16), r1.z, z3);
        z3 = fmaf(__uint_as_float(sr.w & 0xffff0000u), r1.w, z3);
    }
    return (z0 + z1) + (z2 + z3);
}

// (H t)_i for i = threadIdx.x over the 128 threads of the CTA (t is thread
// i's element, H the Sylvester Walsh-Hadamard matrix): strides 1..16 across
// the lanes of a warp, 32 and 64 as one 4-point transform over the four warps
// through s.y. The caller writes s.y again only after a later barrier.
__device__ __forceinline__ float wht128(float t, StepSmem& s) {
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
        const float o = __shfl_xor_sync(TQ_FULL_MASK, t, h);
        t = (lane & h) ? (o - t) : (t + o);
    }
    s.y[i] = t;
    step_sync();
    const float v0 = s.y[lane], v1 = s.y[lane + 32], v2 = s.y[lane + 64], v3 = s.y[lane + 96];
    const float a0 = (warp & 1) ? (v0 - v1) : (v0 + v1);
    const float a1 = (warp & 1) ? (v2 - v3) : (v2 + v3);
    return (warp & 2) ? (a0 - a1) : (a0 + a1);
}

// Quantizes vector v of p into its cache slot. Called by the 128 threads of
// a CTA, all with the same v. xdtype: 0 f32, 1 bf16; cb: code bits per
// coordinate (b - 1 for keys); prod: keys (residual signs); rht: the random-
// sign Walsh-Hadamard rotation, else the dense Pi.
__device__ __forceinline__ void append_vector(const QuantParams& p, int xdtype, int cb, bool prod, bool rht, int64_t v,
                                              StepSmem& s) {
    constexpr int D = 128;
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
    // two channel groups (fractional rates): coordinates with i % 16 >= 8
    // take the second width and codebook
    const bool second = p.code_bits2 != 0 && (i & 15) >= 8;
    const int cbi = second ? p.code_bits2 : cb;
    const Codebook* book = second ? &p.cb2 : &p.cb;
    const int L = 1 << cbi;

    int64_t slot;
    if (p.dst_slot) {
        slot = p.dst_slot[v];
    } else if (p.append_pos) {
        const int32_t pos = p.append_pos[v / p.heads];
        slot = (pos >= 0 && pos < p.capacity) ? v * p.capacity + pos : -1;
    } else {
        slot = p.slot0 + v;
    }
    if (slot < 0 || slot >= p.total_slots) return;  // the same in all 128 threads

    // keys: S (32 KB of bf16) is copied into shared memory now and used last,
    // so the copy hides behind the norm, rotation and bucketize; 16-byte unit
    // (q, j) = S[j][8q .. 8q + 7] sits at unit q * 128 + j in both places, so
    // the copy is contiguous and thread j's reads of its row are conflict-free
    if (prod) stage_s(p.s16, s);
    if (i < kMaxLevels) {
        s.cent[i] = p.cb.c[i];
        s.cent2[i] = p.cb2.c[i];
    }
    if (i < 16) s.cw[i] = 0u;
    const float xi = xdtype == 1 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.x)[v * p.x_stride + i])
                                 : reinterpret_cast<const float*>(p.x)[v * p.x_stride + i];
    s.x[i] = xi;

    // ---- norm, with a rescaled retry when the squares under/overflow ----
    const float ss = step_sum(xi * xi, s);  // its barriers also publish s.x, s.cent and s.cw
    float n32 = sqrtf(ss);
    if (!(ss > 1.0e-30f && ss < 1.0e30f)) {
        const float amax = step_max(fabsf(xi), s);
        const float ia = amax > 0.0f ? 1.0f / amax : 0.0f;
        const float s2 = step_sum((xi * ia) * (xi * ia), s);
        n32 = amax * sqrtf(s2);
    }
    const float inv_n = n32 > 0.0f ? 1.0f / n32 : 0.0f;

    // ---- rotation: y_i = (Pi x)_i / n ----
    float y;
    if (rht) {
        y = wht128(xi * p.sgn[i], s) * (p.inv_sqrt_d * inv_n);
    } else {
        // warp w takes inputs e = 32w .. 32w+31 and lane l outputs 4l .. 4l+3:
        // the lane's 32 row segments of Pi^T are independent 16-byte loads,
        // all in flight at once; the four warps' partial sums meet in s.part
        // (s.x was published by step_sum's barriers)
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) {
            const int e = 32 * warp + kk;
            const float4 t = __ldg(reinterpret_cast<const float4*>(p.pit32 + (size_t)e * D) + lane);
            const float xe = s.x[e];
            acc.x = fmaf(t.x, xe, acc.x);
            acc.y = fmaf(t.y, xe, acc.y);
            acc.z = fmaf(t.z, xe, acc.z);
            acc.w = fmaf(t.w, xe, acc.w);
        }
        *reinterpret_cast<float4*>(&s.part[warp][4 * lane]) = acc;
        step_sync();
        y = ((s.part[0][i] + s.part[1][i]) + (s.part[2][i] + s.part[3][i])) * inv_n;
    }

    // ---- bucketize with the guard band ----
    int k = 0;
    float dmin = 3.0e38f;
#pragma unroll
    for (int t = 0; t < kMaxLevels - 1; ++t) {
        if (t < L - 1) {
            k += (y >= book->t[t]) ? 1 : 0;
            dmin = fminf(dmin, fabsf(y - book->t[t]));
        }
    }
    bool flag = !(dmin >= p.guard);

    // fp16 norm; near an fp16 rounding midpoint it is re-rounded from fp64
    uint16_t n16 = f16_bits_sat(n32);
    bool nclose = false;
    if (n32 > 0.0f && n32 < 65504.0f) {
        const float dn = __half2float(__float2half_rd(n32));
        const float up = __half2float(__float2half_ru(n32));
        nclose = dn != up && fabsf(n32 - 0.5f * (dn + up)) <= 1.0e-6f * n32;
    }

    // ---- fp64 re-decision (rare): the norm from an fp64 sum, and each
    // flagged coordinate's y from an fp64 dot product shared by the 128
    // threads (one term each, then a block sum) -- one thread alone would
    // run 128 dependent fp64 operations, long where the fp64 pipe is narrow ----
    if (step_any(flag || nclose)) {
        const double n64 = sqrt(step_sum64((double)xi * (double)xi, s));
        if (nclose) n16 = __half_as_ushort(__double2half(fmin(n64, 65504.0)));
        while (step_any(flag)) {
            if (i == 0) s.fsel = D;
            step_sync();
            if (flag) atomicMin(&s.fsel, i);
            step_sync();
            const int fi = s.fsel;  // the lowest flagged coordinate; thread i adds term i
            double t;
            if (rht) {
                t = (double)p.sgn[i] * (double)s.x[i];
                if (__popc(fi & i) & 1) t = -t;
            } else {
                t = p.pi64[(size_t)fi * D + i] * (double)s.x[i];
            }
            const double part = step_sum64(t, s);
            if (i == fi) {
                double y64 = 0.0;
                if (n64 > 0.0) y64 = rht ? part / (sqrt((double)D) * n64) : part / n64;
                k = 0;
#pragma unroll
                for (int tt = 0; tt < kMaxLevels - 1; ++tt)
                    if (tt < L - 1) k += (y64 >= book->t64[tt]) ? 1 : 0;
                y = (float)y64;
                flag = false;
            }
        }
    }

    // ---- pack: coordinate i's code at its stream offset (cb * i for one
    // width; with two, each block of 16 coordinates holds 8 codes of each) ----
    const int bit = p.code_bits2 == 0
                        ? cb * i
                        : (i >> 4) * 8 * (cb + p.code_bits2) + (second ? 8 * cb + (i & 7) * p.code_bits2 : (i & 7) * cb);
    atomicOr(&s.cw[bit >> 5], (uint32_t)k << (bit & 31));
    if ((bit & 31) + cbi > 32) atomicOr(&s.cw[(bit >> 5) + 1], (uint32_t)k >> (32 - (bit & 31)));

    float gamma = 0.0f;
    if (prod) {
        // r = y - c[idx], gamma = ||r||, z_j = [(S r)_j >= 0]
        const float r = y - (second ? s.cent2[k] : s.cent[k]);
        gamma = sqrtf(step_sum(r * r, s));
        s.y[i] = r;  // the butterfly reads of s.y finished before step_sum's barriers
        asm volatile("cp.async.wait_group 0;\n" ::: "memory");
        step_sync();  // r and every thread's part of S
        const float z = s_row_dot(s, s.y);  // (S r)_i
        const uint32_t zb = __ballot_sync(TQ_FULL_MASK, z >= 0.0f);  // sign bits 32 warp .. +31
        if (lane == 0) reinterpret_cast<uint32_t*>(p.signs + slot * (int64_t)p.sign_stride)[warp] = zb;
    } else {
        step_sync();  // the packed words are complete
    }
    if (i < (p.code_stride >> 2)) reinterpret_cast<uint32_t*>(p.codes + slot * (int64_t)p.code_stride)[i] = s.cw[i];
    if (i == 0) {
        p.norm[slot] = n16;
        if (prod) p.rnorm[slot] = f16_bits_sat(gamma);
    }
}

}  // namespace tqk
