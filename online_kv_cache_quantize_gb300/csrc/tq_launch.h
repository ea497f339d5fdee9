// Kernel parameter blocks and launchers of libtq (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tqk {

constexpr int kMaxLevels = 16;  // 2^4 Lloyd-Max cells

// Codebook passed by value in the kernel parameter space: no device buffer.
struct Codebook {
    float c[kMaxLevels];
    float t[kMaxLevels - 1];
    double t64[kMaxLevels - 1];
    int levels;
};

struct QuantParams {
    const void* x;
    int64_t x_stride;
    int64_t n;
    const int64_t* dst_slot;
    const int32_t* append_pos;
    int heads;
    int64_t slot0;
    int64_t total_slots;
    int64_t capacity;
    uint8_t* codes;
    int code_stride;
    uint8_t* signs;
    int sign_stride;
    uint16_t* norm;
    uint16_t* rnorm;
    const float* pit32;   // dense: Pi^T [d][d]
    const double* pi64;   // Pi [d][d] fp64
    const float* sgn;     // RHT signs [d]
    const float* st32;    // S^T [d][m]
    const uint16_t* s16;  // m = d = 128: S as bf16 bits, 16-byte unit (q, j) = S[j][8q .. 8q+7] at q * 128 + j
    const void* pi_frag;  // d = 128 dense: Pi^T limbs in mma fragment order
    const void* s_frag;   // m = d = 128: S in mma fragment order
    int d, m;
    float inv_sqrt_d;
    float guard;          // |y - t_j| below this is re-decided in fp64
    Codebook cb;
    // two channel groups (fractional rates): coordinates with i % 16 >= 8
    // take code_bits2 bits and codebook cb2; 0 = every coordinate as cb
    int code_bits2;
    Codebook cb2;
    uint32_t* err;        // device error word (a wait that ran out sets a bit)
};

// tensor-core quantize for d = m = 128 (x 16-byte aligned rows)
cudaError_t launch_quantize_mma(const QuantParams& p, int dtype, int rht, int prod, int code_bits, cudaStream_t s);
// fractional-rate caches: code_bits for the coordinates with i % 16 < 8,
// p.code_bits2 = code_bits - 1 for the others
cudaError_t launch_quantize_mma2(const QuantParams& p, int dtype, int rht, int prod, int code_bits, cudaStream_t s);

// tcgen05 quantize (d = m = 128, bf16 input with 16-byte aligned rows, one
// code width): w_umma / s_umma are the rotation and S operands, K-major with
// the 128-byte swizzle (tq_rotation::d_w_umma, tq_qjl::d_s_umma)
bool quantize_umma_supported(const QuantParams& p, int dtype, int code_bits);
cudaError_t launch_quantize_umma(const QuantParams& p, const void* w_umma, const void* s_umma, int rht, int prod,
                                 int code_bits, cudaStream_t s);

// dtype: 0 f32, 1 bf16, 2 f16. rht: 0 dense, 1 RHT. prod: 0 MSE, 1 PROD.
cudaError_t launch_quantize(const QuantParams& p, int dtype, int rht, int prod, int code_bits,
                            cudaStream_t s);

// PolarQuant keys (d = 128): the angle codebooks of the 7 levels as the
// cosines and sines of their boundaries t_j: a decision psi >= t_j is the
// sign of b cos t_j - a sin t_j (= rho sin(psi - t_j)) for the pair (a, b),
// in fp32, and in fp64 where the fp32 one is too close to call.
constexpr int kPolarLevels = 7;
struct PolarCodebook {
    float tc[kPolarLevels][15];     // cos t_j
    float ts[kPolarLevels][15];     // sin t_j
    double tc64[kPolarLevels][15];
    double ts64[kPolarLevels][15];
};

struct PolarQuantParams {
    QuantParams q;      // input, slots, codes (the angle stream), norm, rotation, err
    PolarCodebook cb;
    int bits1, bits2;   // level-1 and higher-level code widths
    float guard;        // |b cos t - a sin t| below this is re-decided in fp64
};

cudaError_t launch_polar_quantize(const PolarQuantParams& p, int dtype, int rht, cudaStream_t s);

struct PolarDecodeParams {
    const float* qprime;  // [B*Hq][128] q' = Pi q (written by the query prep)
    int batch, hq, hkv, group;
    const int32_t* seq_lens;
    int16_t head_table[256];  // query heads of KV head kv: head_table[kv * group + j]
    int use_table;            // 0: head kv * group + j
    int64_t capacity;
    const uint8_t* kcodes; int kcode_stride;
    const uint16_t* knorm;
    const uint8_t* vcodes; int vcode_stride;
    const uint16_t* vnorm;
    int vbits;
    float vc[kMaxLevels];     // value centroids
    float c1cos[kMaxLevels], c1sin[kMaxLevels];  // level-1 centroid angles
    float ccos[kPolarLevels - 1][kMaxLevels];    // levels 2 .. 7
    float csin[kPolarLevels - 1][kMaxLevels];
    float scale_log2;     // softmax scale * log2(e)
    int n_splits, chunk;  // chunk: tokens per split
    float* partial;       // [B*Hq][n_splits][128 + kPartPad]: a, then M and Z
    float* logits;        // optional [B*Hq][max_seq_len]
    int max_seq_len;
};

// (bits1, bits2) in {(2,2), (3,2), (4,2), (4,3), (3,3), (4,4)}, group in {1, 2, 4, 8}
bool polar_decode_supported(int bits1, int bits2);
cudaError_t launch_polar_decode(const PolarDecodeParams& p, int bits1, int bits2, cudaStream_t s);

struct PrepParams {
    const void* q;        // [rows][d]
    int q_dtype;          // 0 f32, 1 bf16
    int64_t rows;
    int d, m;
    const float* pit32;   // dense Pi^T [d][d]
    const float* sgn;     // RHT signs
    int rht;
    float inv_sqrt_d;
    const float* st32;    // S^T [d][m] or NULL (no u)
    const uint16_t* s16;  // m = d = 128: S as bf16 in the append kernel's unit layout (the decode prep)
    float* qprime;        // [rows][d] or NULL
    float* u;             // [rows][m] or NULL
    // d = m = 128 decode: the scan's B operands of every query row, fp16
    // hi/lo splits of q' and of qjl_scale * u in fragment order (kFragWords
    // words per row; see decode_mma.cuh), or NULL
    uint32_t* frag;
    float qjl_scale;
};

constexpr int kFragWords = 256;

// floats per split partial row of the decode scan: a[0..d), M at d, Z at d + 1,
// padded so every row starts on a 16-byte boundary
constexpr int kPartPad = 4;

cudaError_t launch_query_prep(const PrepParams& p, cudaStream_t s);
// d = 128 rows in fp32 (q' and u; m = 128 with S in its unit layout): several
// rows per CTA sharing one copy of S
cudaError_t launch_rows_prep(const PrepParams& p, cudaStream_t s);

// One launch for the work a decode step does before its scan: the query prep
// of pp.rows query rows (d = 128) and the quantize-on-append of k.n key and
// v.n value vectors (d = m = 128), one CTA per query row or vector. Any part
// may be empty. The scan launched right after it on the same stream may
// start early (programmatic dependent launch) and waits for it to finish.
struct StepPrepParams {
    PrepParams pp;
    QuantParams k, v;
    int k_dtype, v_dtype;  // 0 f32, 1 bf16
    int k_cb, v_cb;        // code bits per coordinate (keys b - 1)
    int k_rht, v_rht;
};

cudaError_t launch_step_prep(const StepPrepParams& p, cudaStream_t s);

struct DecodeParams {
    const uint32_t* frag; // [B*Hq][kFragWords] B operands written by the query prep
    int batch, hq, hkv, d, m, group;
    const int32_t* seq_lens;
    // decode step: the slot its prep launch appends in each batch row (the
    // scan waits for that launch before copying the tile holding it); NULL
    // when the prep appends nothing
    const int32_t* append_pos;
    const int16_t* heads_of_kv;  // nullptr -> kv*G + j; else HOST-built table in params
    int16_t head_table[256];     // heads_of_kv table by value: [hkv][G]
    int use_table;
    int64_t capacity;
    const uint8_t* kcodes; int kcode_stride;
    const uint8_t* ksigns; int ksign_stride;
    const uint16_t* knorm;
    const uint16_t* krnorm;
    const uint8_t* vcodes; int vcode_stride;
    const uint16_t* vnorm;
    float kc[kMaxLevels];
    float vc[kMaxLevels];
    float qjl_scale;      // sqrt(pi/2)/m
    float scale_log2;     // softmax scale * log2(e)
    int n_splits;
    int chunk;            // tokens per split
    float* partial;       // [B*Hq][n_splits][d + kPartPad]: a, then M and Z
    float* logits;        // optional [B*Hq][max_seq_len]
    int max_seq_len;
    // tensor-core scan: 2-coordinate fp16 pair tables of lam * centroid
    uint32_t klut[256];
    uint32_t klut_lo[256];  // residual table lam*c - fp16(lam*c), used for 3-4 bit key codes
    uint32_t vlut[256];
    // fractional-rate caches: the second channel group's tables (same lam)
    uint32_t klut2[64];
    uint32_t klut2_lo[64];
    uint32_t vlut2[64];
    float inv_lam_k, inv_lam_v;
    uint32_t* err;          // device error word (a wait that ran out sets a bit)
};

// two: keys and values are both fractional-rate caches (code bits kbits /
// kbits - 1 and vbits / vbits - 1)
cudaError_t launch_decode_mma(const DecodeParams& p, int kbits, int vbits, bool two, cudaStream_t s);

// Chunked prefill: C query tokens x G heads per KV head against the cache,
// causal (query i sees slots 0 .. q_start[b] + i). kPfRows query rows per CTA.
constexpr int kPfRows = 64;
struct PrefillParams {
    const float* qprime;  // [rows][128] q' = Pi q, rows = (b * chunk + i) * hq + h
    const float* u;       // [rows][128] u = S q'
    int batch, chunk, hq, hkv, group;
    const int32_t* q_start;  // [batch] position of the chunk's first token
    int16_t head_table[256];  // query heads of KV head kv: head_table[kv * group + j]
    int use_table;            // 0: head kv * group + j
    int lim_cap;          // visible slots are capped at min(capacity, max_context)
    int64_t capacity;
    const uint8_t* kcodes;
    const uint8_t* ksigns;
    const uint16_t* knorm;
    const uint16_t* krnorm;
    const uint8_t* vcodes;
    const uint16_t* vnorm;
    uint32_t klut[256];
    uint32_t klut_lo[256];
    uint32_t vlut[256];
    uint32_t klut2[64];
    uint32_t klut2_lo[64];
    uint32_t vlut2[64];
    float inv_lam_k, inv_lam_v;
    float qjl_scale;      // sqrt(pi/2)/m
    float scale_log2;     // softmax scale * log2(e)
    int n_splits;
    int split_tokens;     // tokens per split (a multiple of 64)
    float* partial;       // [rows][n_splits][128 + kPartPad]: a, then M and Z
    uint32_t* err;
    // the tcgen05 kernel's stream-K plan: unit u = (batch row, KV head, query
    // block), u = (b * hkv + kv) * qbs + qb, owns tiles [u * unit_tiles,
    // (u + 1) * unit_tiles) of one sequence; CTA c takes tiles [c *
    // tiles_per_cta, (c + 1) * tiles_per_cta) of it, one segment per unit it
    // touches, and writes the unit's rows' partials into slot (c - the unit's
    // first CTA); n_splits = the most CTAs a unit spans
    int qbs;
    int unit_tiles;
    int tiles_per_cta;
};

// two: keys and values are both fractional-rate caches
cudaError_t launch_prefill_mma(const PrefillParams& p, int kbits, int vbits, bool two, cudaStream_t s);
// The tcgen05 version: kPuRows query rows per CTA, split_tokens a multiple
// of kPuTok, one CTA per SM (all of TMEM); keys at 1 or 2 code bits (2 / 1
// for fractional rates), values 1..4.
constexpr int kPuRows = 128;
constexpr int kPuTok = 128;
constexpr int kPuMaxSeg = 8;  // segments (units) one CTA may touch
bool prefill_umma_supported(int kbits, int vbits, bool two);
cudaError_t launch_prefill_umma(const PrefillParams& p, int kbits, int vbits, bool two, cudaStream_t s);

// The library's device error word of the current device (bits kErr* of
// pipeline.cuh), and a kernel that waits on an mbarrier that nothing
// arrives on for at most limit_ns, so that the bounded wait runs out.
cudaError_t device_error_word(uint32_t** out);
cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t s);
// D [128 x n] = A [128 x k] B [n x k]^T (fp16 in, fp32 out) through tcgen05;
// n in {16, 32, 64, 128}, k a multiple of 16 up to 128
// a_tmem != 0: A goes through TMEM (tcgen05.st) and the MMA reads it there
cudaError_t launch_umma_selftest(const void* a, const void* b, float* d, int n, int k, int a_tmem, uint32_t* err,
                                 cudaStream_t s);


struct CombineParams {
    const float* partial;
    int rows;             // B*Hq
    int d, n_splits;
    const float* pi32;    // dense Pi [d][d] (o_j = sum_i Pi_ij a_i)
    const float* sgn;     // RHT signs
    int rht;
    float inv_sqrt_d;
    void* out;
    int out_dtype;        // 0 f32, 1 bf16
    uint32_t* err;        // device error word (null: the merge without bounded waits)
};

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
// the same merge for many rows with few splits each (d = 128): a warp per row
cudaError_t launch_merge_rows(const CombineParams& p, cudaStream_t s);

struct TopkParams {
    const float* qprime;  // [nq][d]
    const float* u;       // [nq][m] or NULL (MSE)
    int nq, d, m;
    const uint8_t* codes; int code_stride;
    const uint8_t* signs; int sign_stride;
    const uint16_t* norm;
    const uint16_t* rnorm;
    int64_t n_db;
    float c[kMaxLevels];
    float qjl_scale;
    int k;
    int n_chunks;
    int64_t chunk_rows;
    float* cand_score;    // [nq][n_chunks][k]
    int32_t* cand_id;     // [nq][n_chunks][k]
    int32_t* ids;
    float* scores;
    // tensor-core scan: lam * centroid fp16 pair tables (hi and the residual
    // lo), 1 / lam, the segment width (padded d and m) and the error word
    uint32_t ktab[256];
    uint32_t ktab_lo[256];
    float inv_lam;
    int ks;
    uint32_t* err;
};

cudaError_t launch_topk(const TopkParams& p, int code_bits, int prod, cudaStream_t s);
// tcgen05 search scan + merge; returns cudaErrorNotSupported when the shape
// does not fit its shared-memory plan (the caller then uses launch_topk)
cudaError_t launch_topk_umma(const TopkParams& p, int code_bits, int prod, int lo, cudaStream_t s);

}  // namespace tqk
