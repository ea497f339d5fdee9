// Decode attention launches: query preparation (fused with the decode
// step's appends), split-K scan dispatch, merge.
#include <algorithm>

#include "append.cuh"
#include "decode.cuh"

namespace tqk {

// The decode step's work before its scan in one launch: query prep rows
// (decode.cuh) and the appended key and value vectors (append.cuh).

// Query prep of one row (d = m = 128) by the 128 threads of a CTA, thread i
// owning coordinate i: q' = Pi q (random-sign Walsh-Hadamard by butterflies,
// or the dense Pi), u = S q' from S staged in shared memory, and the scan's
// B operands (the same words as write_frag in decode.cuh).
// stage: copy S into shared memory here (false: the caller already has)
__device__ __forceinline__ void prep_row128(const PrepParams& p, int64_t row, StepSmem& s, bool stage = true) {
    constexpr int D = 128;
    const int i = threadIdx.x;
    const bool want_u = p.st32 != nullptr;
    if (want_u && stage) stage_s(p.s16, s);  // lands while q' is formed
    const float qi = p.q_dtype == 1 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.q)[row * D + i])
                                    : reinterpret_cast<const float*>(p.q)[row * D + i];
    float y;
    if (p.rht) {
        y = wht128(qi * p.sgn[i], s) * p.inv_sqrt_d;
    } else {
        // warp w takes inputs e = 32w .. 32w+31, lane l outputs 4l .. 4l+3:
        // each lane's 32 row segments of Pi^T are independent 16-byte loads,
        // issued together (one round of memory latency, not one per
        // dependent batch), then the four warps' partial sums are added
        s.x[i] = qi;
        step_sync();
        const int w = i >> 5, l = i & 31;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const int e = 32 * w + k;
            const float4 t = __ldg(reinterpret_cast<const float4*>(p.pit32 + (size_t)e * D) + l);
            const float xe = s.x[e];
            acc.x = fmaf(t.x, xe, acc.x);
            acc.y = fmaf(t.y, xe, acc.y);
            acc.z = fmaf(t.z, xe, acc.z);
            acc.w = fmaf(t.w, xe, acc.w);
        }
        *reinterpret_cast<float4*>(&s.part[w][4 * l]) = acc;
        step_sync();
        y = (s.part[0][i] + s.part[1][i]) + (s.part[2][i] + s.part[3][i]);
    }
    s.qp[i] = y;
    if (p.qprime) p.qprime[row * D + i] = y;
    if (want_u) {
        asm volatile("cp.async.wait_group 0;\n" ::: "memory");
        step_sync();  // q' and all of S
        const float u = s_row_dot(s, s.qp);
        if (p.u) p.u[row * D + i] = u;
        s.u[i] = u;
    }
    if (p.frag) {
        step_sync();
        write_frag(p, row, s.qp, want_u ? s.u : nullptr, i);
        write_frag(p, row, s.qp, want_u ? s.u : nullptr, i + kStepThreads);
    }
}

__global__ void __launch_bounds__(kStepThreads) step_prep_kernel(const __grid_constant__ StepPrepParams p) {
    // the scan that follows on the stream may be scheduled now: it waits for
    // this grid to complete before it reads anything written here
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    __shared__ StepSmem s;
    int64_t b = blockIdx.x;
    if (b < p.pp.rows) {
        prep_row128(p.pp, b, s);
        return;
    }
    b -= p.pp.rows;
    if (b < p.k.n) {
        append_vector(p.k, p.k_dtype, p.k_cb, true, p.k_rht != 0, b, s);
        return;
    }
    b -= p.k.n;
    if (b < p.v.n) append_vector(p.v, p.v_dtype, p.v_cb, false, p.v_rht != 0, b, s);
}

cudaError_t launch_step_prep(const StepPrepParams& p, cudaStream_t s) {
    const int64_t ctas = p.pp.rows + p.k.n + p.v.n;
    if (ctas <= 0) return cudaSuccess;
    if (ctas > 0x7fffffff || (p.pp.rows > 0 && (p.pp.d != 128 || (p.pp.st32 && (p.pp.m != 128 || !p.pp.s16)))) ||
        (p.k.n > 0 && (p.k.d != 128 || p.k.m != 128 || !p.k.s16)) ||
        (p.v.n > 0 && p.v.d != 128))
        return cudaErrorInvalidValue;
    step_prep_kernel<<<(unsigned)ctas, kStepThreads, 0, s>>>(p);
    return cudaGetLastError();
}

// Query prep of many rows (the chunked prefill): kPrepRows rows per CTA, S
// staged in shared memory once per CTA instead of read once per row; writes
// q' and u in fp32.
constexpr int kPrepRows = 8;

__global__ void __launch_bounds__(kStepThreads) rows_prep_kernel(const __grid_constant__ PrepParams p) {
    __shared__ StepSmem s;
    if (p.st32 != nullptr) stage_s(p.s16, s);
    const int64_t r0 = (int64_t)blockIdx.x * kPrepRows;
    for (int k = 0; k < kPrepRows && r0 + k < p.rows; ++k) {
        if (k) step_sync();  // the previous row's reads of the shared rows are done
        prep_row128(p, r0 + k, s, false);
    }
}

// Query prep of many rows on the tensor cores (the chunked prefill with the
// random-sign Walsh-Hadamard rotation, d = m = 128): a warp takes 16 rows at a
// time. q' = H diag(s) q / sqrt(d) by butterflies (lane l holding coordinates
// 4l .. 4l + 3 of one row: strides 1 and 2 in the lane, 4 .. 64 by shuffles),
// then u = S q' for the 16 rows as mma.sync m16n8k16 (bf16 x bf16 -> f32)
// with S staged in shared memory: S is exact in bf16 and q' goes in three
// bf16 limbs (hi, mid, lo: 24 significant bits), so every product is exact
// and the fp32 accumulation is the only rounding, as in the row kernel above.
constexpr int kPrepMmaWarps = 4;

__device__ __forceinline__ void mma16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// three bf16 limbs of a pair (the first element in the low half of each word)
__device__ __forceinline__ void bf16_limbs2(float x, float y, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 hf = __bfloat1622float2(h);
    const float rx = x - hf.x, ry = y - hf.y;  // exact
    const __nv_bfloat162 m = __floats2bfloat162_rn(rx, ry);
    const float2 mf = __bfloat1622float2(m);
    const __nv_bfloat162 l = __floats2bfloat162_rn(rx - mf.x, ry - mf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    mid = *reinterpret_cast<const uint32_t*>(&m);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// dynamic shared memory of rows_prep_mma_kernel: S in the unit layout of
// StepSmem::s (32 KB), then each warp's 16 rows of q' (fp32, rows padded to
// 132 floats so that the fragment reads spread over the banks)
constexpr size_t kPrepMmaSmem = 16 * 128 * 16 + (size_t)kPrepMmaWarps * 16 * 132 * 4;

__global__ void __launch_bounds__(kPrepMmaWarps * 32) rows_prep_mma_kernel(const __grid_constant__ PrepParams p) {
    extern __shared__ __align__(16) unsigned char prep_smem[];
    float(*s_q)[16][132] = reinterpret_cast<float(*)[16][132]>(prep_smem + 16 * 128 * 16);
    {
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(prep_smem);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int unit = u * kPrepMmaWarps * 32 + (int)threadIdx.x;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst + 16 * unit),
                         "l"(reinterpret_cast<const uint4*>(p.s16) + unit)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
        asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    }
    __syncthreads();
    const uint32_t* s32 = reinterpret_cast<const uint32_t*>(prep_smem);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const float4 sg = *reinterpret_cast<const float4*>(p.sgn + 4 * lane);
    const int64_t nblk = (p.rows + 15) / 16;
    for (int64_t blk = (int64_t)blockIdx.x * kPrepMmaWarps + warp; blk < nblk;
         blk += (int64_t)gridDim.x * kPrepMmaWarps) {
        const int64_t r0 = blk * 16;
        // ---- q' of the 16 rows ----
#pragma unroll 4
        for (int rr = 0; rr < 16; ++rr) {
            const int64_t row = r0 + rr;
            float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (row < p.rows) {
                if (p.q_dtype == 1) {
                    const uint2 w = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                                   row * 128 + 4 * lane);
                    x = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                                    __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
                } else {
                    x = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.q) + row * 128 + 4 * lane);
                }
            }
            float v[4] = {x.x * sg.x, x.y * sg.y, x.z * sg.z, x.w * sg.w};
            // strides 1 and 2 inside the lane
            float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
            v[0] = a0 + a2; v[1] = a1 + a3; v[2] = a0 - a2; v[3] = a1 - a3;
            // strides 4 .. 64 across the lanes
#pragma unroll
            for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float o = __shfl_xor_sync(TQ_FULL_MASK, v[e], h);
                    v[e] = (lane & h) ? (o - v[e]) : (v[e] + o);
                }
            }
            const float4 y = make_float4(v[0] * p.inv_sqrt_d, v[1] * p.inv_sqrt_d, v[2] * p.inv_sqrt_d,
                                         v[3] * p.inv_sqrt_d);
            if (row < p.rows && p.qprime) *reinterpret_cast<float4*>(p.qprime + row * 128 + 4 * lane) = y;
            *reinterpret_cast<float4*>(&s_q[warp][rr][4 * lane]) = y;
        }
        __syncwarp();
        // ---- u = S q' (16 rows x 128) ----
        float acc[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks) {
            // A: (row g, k 16ks + 2c, +1), (row g + 8, same), (row g, k + 8, + 9), (row g + 8, same)
            const int k0 = 16 * ks + 2 * c;
            const float2 x0 = *reinterpret_cast<const float2*>(&s_q[warp][g][k0]);
            const float2 x1 = *reinterpret_cast<const float2*>(&s_q[warp][g + 8][k0]);
            const float2 x2 = *reinterpret_cast<const float2*>(&s_q[warp][g][k0 + 8]);
            const float2 x3 = *reinterpret_cast<const float2*>(&s_q[warp][g + 8][k0 + 8]);
            uint32_t ah[4], am[4], al[4];
            bf16_limbs2(x0.x, x0.y, ah[0], am[0], al[0]);
            bf16_limbs2(x1.x, x1.y, ah[1], am[1], al[1]);
            bf16_limbs2(x2.x, x2.y, ah[2], am[2], al[2]);
            bf16_limbs2(x3.x, x3.y, ah[3], am[3], al[3]);
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                // B: (k 16ks + 2c, +1) and (k + 8, + 9) of column 8nt + g = row 8nt + g of S;
                // unit (q, j) of the staged S holds S[j][8q .. 8q + 7]
                const uint32_t b0 = s32[((2 * ks) * 128 + 8 * nt + g) * 4 + c];
                const uint32_t b1 = s32[((2 * ks + 1) * 128 + 8 * nt + g) * 4 + c];
                mma16816_bf16(acc[nt], ah, b0, b1);
                mma16816_bf16(acc[nt], am, b0, b1);
                mma16816_bf16(acc[nt], al, b0, b1);
            }
        }
        if (p.u) {
            const int64_t ra = r0 + g, rb = r0 + g + 8;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                if (ra < p.rows)
                    *reinterpret_cast<float2*>(p.u + ra * 128 + 8 * nt + 2 * c) = make_float2(acc[nt][0], acc[nt][1]);
                if (rb < p.rows)
                    *reinterpret_cast<float2*>(p.u + rb * 128 + 8 * nt + 2 * c) = make_float2(acc[nt][2], acc[nt][3]);
            }
        }
        __syncwarp();  // s_q is rewritten by the next block
    }
}

cudaError_t launch_rows_prep(const PrepParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    if (p.d != 128 || p.frag || (p.st32 && (p.m != 128 || !p.s16))) return cudaErrorInvalidValue;
    // the tensor-core kernel reads q and the signs as 16-byte (f32) or 8-byte
    // (bf16) vectors; other alignments take the row kernel
    const bool vec_ok = (reinterpret_cast<uintptr_t>(p.q) % 16) == 0 && (reinterpret_cast<uintptr_t>(p.sgn) % 16) == 0;
    if (p.rht && p.st32 && vec_ok) {
        int dev = 0, sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t nblk = (p.rows + 15) / 16;
        const int64_t ctas = std::min<int64_t>((nblk + kPrepMmaWarps - 1) / kPrepMmaWarps, (int64_t)sms * 3);
        cudaError_t e = cudaFuncSetAttribute(rows_prep_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kPrepMmaSmem);
        if (e != cudaSuccess) return e;
        rows_prep_mma_kernel<<<(unsigned)ctas, kPrepMmaWarps * 32, kPrepMmaSmem, s>>>(p);
        return cudaGetLastError();
    }
    const int64_t ctas = (p.rows + kPrepRows - 1) / kPrepRows;
    if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
    rows_prep_kernel<<<(unsigned)ctas, kStepThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_query_prep(const PrepParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    dim3 grid((unsigned)p.rows), block(kPrepWarps * 32);
    if (p.d <= 64) query_prep_kernel<2><<<grid, block, 0, s>>>(p);
    else if (p.d <= 128) query_prep_kernel<4><<<grid, block, 0, s>>>(p);
    else if (p.d <= 224) query_prep_kernel<7><<<grid, block, 0, s>>>(p);
    else query_prep_kernel<8><<<grid, block, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode_mma_g1(const DecodeParams& p, int kbits, int vbits, bool two, cudaStream_t s);
cudaError_t launch_decode_mma_g2(const DecodeParams& p, int kbits, int vbits, bool two, cudaStream_t s);
cudaError_t launch_decode_mma_g4(const DecodeParams& p, int kbits, int vbits, bool two, cudaStream_t s);
cudaError_t launch_decode_mma_g8(const DecodeParams& p, int kbits, int vbits, bool two, cudaStream_t s);

cudaError_t launch_decode_mma(const DecodeParams& p, int kbits, int vbits, bool two, cudaStream_t s) {
    switch (p.group) {
        case 1: return launch_decode_mma_g1(p, kbits, vbits, two, s);
        case 2: return launch_decode_mma_g2(p, kbits, vbits, two, s);
        case 4: return launch_decode_mma_g4(p, kbits, vbits, two, s);
        case 8: return launch_decode_mma_g8(p, kbits, vbits, two, s);
    }
    return cudaErrorInvalidValue;
}

// Programmatic dependent launch: the merge's CTAs may be scheduled while the
// scan's last CTAs still run (the scan signals launch_dependents once its
// tiles are done); the merge waits for the scan grid to complete before it
// reads a partial (griddepcontrol.wait).
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    const bool bulk = p.d == 128 && p.rht && p.err != nullptr && p.n_splits >= 1 &&
                      p.n_splits <= kCombBulkMaxSplits && (reinterpret_cast<uintptr_t>(p.partial) & 15) == 0;
    if (bulk) {
        const size_t smem = (size_t)p.n_splits * (128 + kPartPad) * sizeof(float);  // <= 48 KB
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)p.rows);
        cfg.blockDim = dim3(kCombBulkThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, combine_bulk_kernel, p);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.rows);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

// The few-splits merge (d = 128), also a programmatic dependent of the scan.
cudaError_t launch_merge_rows(const CombineParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    if (p.d != 128) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((p.rows + kMergeWarps - 1) / kMergeWarps));
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_rows_kernel, p);
}

}  // namespace tqk
