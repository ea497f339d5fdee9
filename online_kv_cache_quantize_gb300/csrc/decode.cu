// Decode attention launches: query preparation (fused with the decode
// step's appends), split-K scan dispatch, merge.
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

cudaError_t launch_rows_prep(const PrepParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    if (p.d != 128 || p.frag || (p.st32 && (p.m != 128 || !p.s16))) return cudaErrorInvalidValue;
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
