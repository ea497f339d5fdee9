/*
 * tq.h - C ABI of libtq, a GB300 (sm_103a) implementation of the TurboQuant
 * hot path: quantize-on-append of KV head vectors and decode attention scored
 * directly from the packed codes.
 *
 * Sources the operations follow (TurboQuant write-ups):
 *   [Qiita]  Qiita TurboQuant article (the "3-bit KV cache" explainer)
 *   [A2A]    A2A TurboQuant explainer "TurboQuant解説：実装方法とLLMメモリ6倍削減効果"
 *   [DS]     DeepSignal TurboQuant ICLR 2026 article
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" must point to memory of the CUDA device that
 *     is current on the calling thread; "host" pointers are ordinary memory.
 *   - All buffers are owned by the caller. The library allocates device
 *     memory only inside tq_rotation_to_device / tq_qjl_to_device (set-up);
 *     the hot-path calls never allocate: scratch comes from the caller's
 *     workspace argument.
 *   - Hot-path calls are asynchronous on the given stream (NULL = legacy
 *     default stream). Argument errors are found on the host before any
 *     launch and return a status; a launch failure returns TQ_ERR_CUDA;
 *     faults during execution surface at the caller's next synchronisation.
 *   - No call blocks on the device. The one kind of device-side wait (a
 *     kernel waiting for its bulk copies or tensor-core products to land on
 *     an mbarrier) gives up after one second, records the cause in the device
 *     error word and lets the kernel return; tq_device_errors reads it
 *     (TQ_ERR_TIMEOUT).
 *   - tq_last_error() returns a thread-local message for the last failure.
 *   - tq_attn_decode and tq_decode_step keep, per calling thread, the
 *     validated plan of their last call: a call whose argument struct is
 *     byte-for-byte the same (with the same host gqa_map contents, workspace,
 *     current device, and no handle created, uploaded or freed since) skips
 *     the validation and goes straight to its launches. A decode loop that
 *     passes a constant max_seq_len (e.g. the capacity) hits it every step;
 *     device-side values (lengths, positions, the data) may change freely.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tq_stream; /* same type as cudaStream_t */
typedef struct CUevent_st* tq_event;   /* same type as cudaEvent_t  */

typedef enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = 1,  /* null pointer, bad size, mismatched handles   */
    TQ_ERR_UNSUPPORTED = 2,  /* valid but not built: e.g. RHT with d not 2^k  */
    TQ_ERR_ALIGNMENT = 3,    /* a device pointer or stride breaks alignment  */
    TQ_ERR_CAPACITY = 4,     /* a slot range runs past the cache capacity    */
    TQ_ERR_CUDA = 5,         /* a CUDA runtime call failed                   */
    TQ_ERR_TIMEOUT = 6,      /* a device-side wait ran out (tq_device_errors) */
    TQ_ERR_WORKSPACE = 7,    /* workspace missing or smaller than required   */
    TQ_ERR_NO_DEVICE_COPY = 8 /* handle not uploaded with *_to_device        */
} tq_status;

typedef enum { TQ_ROT_DENSE_QR = 0, TQ_ROT_RHT = 1 } tq_rot_kind;
typedef enum { TQ_MSE = 0, TQ_PROD = 1, TQ_POLAR = 2 } tq_mode;
typedef enum { TQ_F32 = 0, TQ_BF16 = 1, TQ_F16 = 2 } tq_dtype;

typedef struct tq_rotation tq_rotation;
typedef struct tq_qjl tq_qjl;

const char* tq_status_string(tq_status s);
const char* tq_last_error(void);

/* sizeof of a public struct by name ("tq_cache", "tq_quant_args",
 * "tq_decode_args", "tq_topk_args"); 0 for an unknown name. Lets bindings
 * check their struct mirrors against this build. */
size_t tq_abi_struct_size(const char* name);

/* ------------------------------------------------------------------------ *
 * Set-up (host).                                                           *
 * ------------------------------------------------------------------------ */

/* The random stream every random draw of the library uses: SplitMix64
 * (Steele, Lea & Flood 2014) in counter form, draw k = mix(seed + (k+1)*gamma).
 * Writes draws start .. start+count-1 to host_out (host, count uint64).
 * The pages only say the random matrices are generated mathematically once
 * and cached ([Qiita] "Rotate, then quantize"; [DS] "QJL"). */
tq_status tq_random_stream(uint64_t seed, uint64_t start, int64_t count, uint64_t* host_out);

/* Data-independent random orthogonal rotation Pi (d x d), y = Pi x.
 * [A2A] "Stage 1: random rotation": QR factorisation of a Gaussian matrix.
 * [Qiita] "What you hit when you try it": Walsh-Hadamard approximation.
 *   kind TQ_ROT_DENSE_QR: G = d*d standard normals (Box-Muller over the
 *     stream, row-major), Householder QR G = QR, Pi = Q diag(sign(diag R)).
 *     3 <= d <= 256.
 *   kind TQ_ROT_RHT: Pi = H diag(s) / sqrt(d), H Sylvester Hadamard
 *     (H_ij = (-1)^popcount(i&j)), s_i = -1 if bit 63 of draw i is set else
 *     +1. d a power of two, 4 <= d <= 256 (else TQ_ERR_UNSUPPORTED).
 * *out receives a host-side handle owned by the caller until
 * tq_free_rotation. No device memory is touched. */
tq_status tq_make_rotation(uint64_t seed, int d, int kind, tq_rotation** out);

/* Copies Pi (fp64, d*d, row-major) to host_out (host, caller-owned). */
tq_status tq_rotation_get(const tq_rotation* rot, double* host_out);

/* *d, *kind receive the handle's size and kind (either may be NULL). */
tq_status tq_rotation_info(const tq_rotation* rot, int* d, int* kind);

/* Uploads the device copies (fp32 Pi and Pi^T, fp64 Pi, RHT signs) to the
 * current device. Allocates device memory (set-up, not hot path). Calling it
 * again is a no-op. Needed before any hot-path call that uses the handle. */
tq_status tq_rotation_to_device(tq_rotation* rot);

/* Frees host and device memory of the handle; NULL is accepted. */
tq_status tq_free_rotation(tq_rotation* rot);

/* QJL projection S (m x d) for the residual sign sketch.
 * [Qiita] "One more stage so attention does not break"; [A2A] "Stage 2".
 * Entries: standard normals (Box-Muller over the stream of `seed`,
 * row-major) rounded to the nearest bfloat16, ties to even, so that the
 * matrix is exact in bf16. 1 <= m <= 256, 3 <= d <= 256. */
tq_status tq_make_qjl(uint64_t seed, int m, int d, tq_qjl** out);
tq_status tq_qjl_get(const tq_qjl* qjl, double* host_out); /* m*d row-major */
tq_status tq_qjl_to_device(tq_qjl* qjl);
tq_status tq_free_qjl(tq_qjl* qjl);

/* Lloyd-Max codebook of the post-rotation law Beta((d-1)/2,(d-1)/2) on
 * [-1, 1] ([A2A] "Stage 1"; [Qiita] "Rotate, then quantize").
 * centroids: host, 2^bits doubles, ascending; boundaries: host, 2^bits - 1
 * doubles, t_j = (c_j + c_{j+1}) / 2. Exactly symmetric; middle boundary 0.
 * 1 <= bits <= 4, 3 <= d <= 4096. Computed once per (d, bits), cached. */
tq_status tq_codebook(int d, int bits, double* centroids, double* boundaries);

/* ------------------------------------------------------------------------ *
 * Packed cache layout (this library's specification; the pages give none). *
 * ------------------------------------------------------------------------ *
 * A cache holds `rows` rows (normally batch*Hkv) of `capacity` slots; slot
 * s = row * capacity + t. Per slot, structure of arrays:
 *   codes[s]: code bytes = ceil(cb * d / 8) rounded up to 16, where
 *             cb = bits (TQ_MSE) or bits - 1 (TQ_PROD). Bit k of coordinate
 *             i's index is stream bit cb*i + k; stream bit p is bit p%8 of
 *             byte p/8 (LSB-first). Padding bits are 0.
 *   signs[s]: (TQ_PROD) sign bytes = ceil(m / 8) rounded up to 16;
 *             bit j (LSB-first) = [(S r)_j >= 0].
 *   norm[s]:  fp16 bits of ||x|| (round to nearest even, saturated 65504).
 *   rnorm[s]: (TQ_PROD) fp16 bits of ||r||, r = Pi x/||x|| - c[idx].
 * All four plane pointers must be 16-byte aligned (norm/rnorm: 2-byte).
 *
 * Fractional bit-rates (bits2 != 0 and != bits; the 2.5 / 3.5 bits per
 * channel the Qiita article's tables quote, read as two channel groups):
 * coordinate i takes `bits` when i % 16 < 8 and `bits2` otherwise, each
 * group with its own Lloyd-Max codebook of the same law; codes are packed in
 * coordinate order with their own widths (coordinate i starts after the bits
 * of coordinates 0 .. i-1), stride tq_code_bytes2 (rounded up to 8 bytes, so
 * the smaller width saves memory). Supported: d = 128 and bits2 = bits - 1
 * (keys 3/2 = 2.5 and 4/3 = 3.5 bits, values likewise). tq_quantize_kv takes
 * them; the decode entry points take them when the key and the value cache
 * are both fractional-rate (one of each kind: TQ_ERR_UNSUPPORTED); the search
 * returns TQ_ERR_UNSUPPORTED. */
typedef struct {
    int mode;         /* TQ_MSE (values) or TQ_PROD (keys)                   */
    int bits;         /* MSE: 1..4 Lloyd-Max bits; PROD: 2..5 = (bits-1) + 1 */
    int d;            /* head dimension                                      */
    int m;            /* PROD: QJL rows; MSE: ignored                        */
    int64_t rows;     /* rows in the cache                                   */
    int64_t capacity; /* slots per row                                       */
    uint8_t* codes;   /* device [rows*capacity][tq_code_bytes]               */
    uint8_t* signs;   /* device [rows*capacity][tq_sign_bytes] (PROD)        */
    uint16_t* norm;   /* device [rows*capacity] fp16 bits                    */
    uint16_t* rnorm;  /* device [rows*capacity] fp16 bits (PROD)             */
    int bits2;        /* 0: every coordinate at `bits`; else the second
                         channel group's bits (fractional rates, see above)  */
} tq_cache;

/* PolarQuant keys (mode TQ_POLAR; the comparison variant of [DS]
 * "PolarQuant" and [A2A] "Stage 1" PolarQuant bullets): y = Pi x / ||x||
 * (the same rotation as the other modes) is taken to polar coordinates by a
 * recursion over pairs: level 1 pairs (y_2i, y_2i+1) into a radius
 * rho_1,i = hypot and an angle psi_1,i = atan2(y_2i+1, y_2i) in (-pi, pi];
 * level l >= 2 pairs the radii of level l - 1 the same way (angles in
 * [0, pi/2]); log2(d) levels, d - 1 angles. The final radius is ||y|| = 1,
 * so the only magnitude kept is ||x|| (fp16 in the norm plane). Each angle is
 * quantized by the Lloyd-Max codebook of its level's law after a Haar
 * rotation (tq_polar_codebook): level-1 angles at `bits` bits, the others at
 * `bits2`. Ties go to the upper cell (code = #{j : t_j <= psi}).
 * Layout: codes[s] holds the angle codes as one LSB-first bit stream, level
 * 1 first (angle i at bits * i), then levels 2, 3, ... in order, each angle
 * at its level's width; stride tq_polar_code_bytes(d, bits, bits2). The
 * signs and rnorm planes are not used (may be NULL); m is ignored.
 * Supported: d = 128, bits and bits2 in 1..4 (tq_quantize_kv); decode takes
 * (bits, bits2) in {(2,2), (3,2), (4,2), (4,3), (3,3), (4,4)} with an MSE
 * value cache. The key logit is l_t = n_t <q', y_hat_t>, y_hat_t the inverse
 * recursion from the centroid angles (unit norm); no sign sketch. */
int tq_polar_code_bytes(int d, int bits, int bits2); /* 0 for invalid arguments */

/* Lloyd-Max codebook of the PolarQuant angles of one level (1 = coordinate
 * pairs, up to 8) after a Haar rotation: level 1 uniform on (-pi, pi] (equal
 * cells from -pi); level l >= 2 with density proportional to
 * (sin psi cos psi)^(2^(l-1) - 1) on [0, pi/2], i.e. sin^2 psi ~
 * Beta(k/2, k/2), k = 2^(l-1). centroids: host, 2^bits doubles ascending;
 * boundaries: host, 2^bits - 1 doubles, the midpoints. 1 <= bits <= 4.
 * Computed once per (level, bits), cached. */
tq_status tq_polar_codebook(int level, int bits, double* centroids, double* boundaries);

int tq_code_bytes(int d, int code_bits); /* per-slot stride of codes, bytes */
/* per-slot stride of a two-group cache's codes (code bits of the coordinates
 * with i % 16 < 8, of the others): the bit count rounded up to 8 bytes;
 * equals tq_code_bytes(d, code_bits) when the two are equal */
int tq_code_bytes2(int d, int code_bits, int code_bits2);
int tq_sign_bytes(int m);                /* per-slot stride of signs, bytes */

/* ------------------------------------------------------------------------ *
 * Quantize-on-append.                                                      *
 * ------------------------------------------------------------------------ *
 * For each input vector x: n = ||x||; y = Pi x / n (y = 0 if n = 0);
 * idx_i = #{j : y_i >= t_j}; store codes and fp16(n). PROD mode also:
 * r = y - c[idx], gamma = ||r||, z_j = [(S r)_j >= 0]; store signs and
 * fp16(gamma). ([A2A] "Stage 1" and "Stage 2"; [Qiita] "Rotate, then
 * quantize" and "One more stage so attention does not break".)
 * Destination slot of vector i:
 *   dst_slot != NULL  -> dst_slot[i] (device int64 [n]; slots outside
 *                        [0, rows*capacity) are skipped);
 *   else append_pos != NULL -> vector i = (b, h) with b = i / heads,
 *                        h = i % heads, slot = i * capacity + append_pos[b]
 *                        (device int32 [n / heads]; needs rows == n; a
 *                        position outside [0, capacity) is skipped);
 *   else              -> slot0 + i (checked on the host against the cache).
 * Kernels: d = 128 (keys m = 128) and n <= 256, one CTA per vector (an append
 * costs a few microseconds however few vectors it has); d = 128 and more
 * vectors with bf16 input (one code width, or the two widths of a
 * fractional-rate cache), tiles of 128 vectors on the 5th-generation tensor
 * cores (the rotation and S r as tcgen05 contractions with TMEM
 * accumulators); other d = 128 cases with 16-byte aligned rows (fp32 input),
 * 16 vectors per warp with the rotation and S r on mma.sync; any other d, one
 * warp per vector; PolarQuant caches, one warp per vector. All follow the same precision rules: every code is the
 * one an fp64 evaluation gives, up to ties within a few fp64 ulps. */
typedef struct {
    tq_cache cache;
    const tq_rotation* rot; /* uploaded; rot d == cache.d                     */
    const tq_qjl* qjl;      /* PROD: uploaded, m == cache.m, d == cache.d     */
    const void* x;          /* device [n][x_stride] of x_dtype                */
    int x_dtype;            /* TQ_F32 or TQ_BF16                              */
    int64_t x_stride;       /* elements between vectors, >= d                 */
    int64_t n;              /* vectors; 0 is a no-op                          */
    const int64_t* dst_slot;
    const int32_t* append_pos;
    int heads;              /* append_pos mode: vectors per position entry    */
    int64_t slot0;
} tq_quant_args;

tq_status tq_quantize_kv(const tq_quant_args* a, tq_stream stream);

/* ------------------------------------------------------------------------ *
 * Decode attention from the packed cache.                                  *
 * ------------------------------------------------------------------------ *
 * For batch b and query head h (KV head g = gqa_map[h]):
 *   q' = Pi q, u = S q'                       (query rotated once)
 *   l_t = n_t ( <q', cK[idx_t]> + sqrt(pi/2)/m * gamma_t <u, 2 z_t - 1> )
 *   p = softmax(scale * l) over t < seq_lens[b]
 *   a = sum_t p_t nV_t cV[idxV_t]  (rotated domain); out = Pi^T a
 * ([A2A] end of "Stage 2" and "How to implement": pre-rotated query, dot
 * products from the indices; softmax and value sum are this library's
 * reading). A sequence with no visible token gives out = 0.
 * Split-K over tokens: CTAs write partial (max, sum, a) to the workspace; a
 * second launch merges them and un-rotates. */
typedef struct {
    const void* q;          /* device [batch][hq][d] of q_dtype (or pinned host
                               memory the GPU addresses, see below)           */
    int q_dtype;            /* TQ_F32 or TQ_BF16                              */
    int batch, hq, hkv, d;  /* d = 128                                        */
    const int32_t* seq_lens;/* device int32 [batch], each in [0, capacity]    */
    int max_seq_len;        /* host: upper bound of seq_lens (split plan)     */
    const int32_t* gqa_map; /* HOST int32 [hq] in [0, hkv), or NULL = h/(hq/hkv);
                               every KV head must serve the same number G of
                               query heads, G in {1, 2, 4, 8}                 */
    const tq_rotation* rot; /* uploaded                                       */
    const tq_qjl* qjl;      /* uploaded, m == k.m                             */
    tq_cache k;             /* PROD cache, rows == batch*hkv                  */
    tq_cache v;             /* MSE cache, rows == batch*hkv                   */
    float scale;            /* softmax scale; 0 -> 1/sqrt(d)                  */
    int n_splits;           /* token splits per (b, KV head); 0 -> automatic  */
    void* out;              /* device [batch][hq][d] of out_dtype (or pinned
                               host memory the GPU addresses, see below)      */
    int out_dtype;          /* TQ_F32 or TQ_BF16                              */
    float* logits;          /* optional device fp32 [batch][hq][max_seq_len]:
                               raw l_t (before scale) for t < seq_lens[b]    */
    tq_event scan_begin;    /* optional: recorded on `stream` right before and */
    tq_event scan_end;      /* after the split-K scan kernel (for timing it)   */
} tq_decode_args;

/* Workspace bytes tq_attn_decode needs for these arguments (0 on error). */
size_t tq_attn_decode_workspace(const tq_decode_args* a);

/* workspace: device, >= tq_attn_decode_workspace(a) bytes, 256-byte aligned,
 * not used by anything else until the call's work on `stream` completes. */
tq_status tq_attn_decode(const tq_decode_args* a, void* workspace, size_t ws_bytes, tq_stream stream);

/* Decode attention that allocates nothing. No counterpart in the write-ups:
 * it exists for callers that may not allocate device memory when they run
 * decode, such as a plugin inside an engine that owns all device memory, work
 * enqueued during CUDA graph capture, or a runtime that forbids allocation
 * after start-up. Same arguments and results as tq_attn_decode, but the
 * scratch is an array compiled into the library, TQ_STATIC_DECODE_SCRATCH_BYTES
 * per device, held by every device that loads the library until the process
 * exits; the call itself calls no allocator.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero (each call writes every scratch
 *     byte it reads). Calls whose work overlaps on the GPU (several streams,
 *     threads or processes sharing a context) race on it: serialise them.
 *   - Returns TQ_ERR_WORKSPACE, with a message giving the size needed, when
 *     the arguments need more scratch than the array holds
 *     (tq_attn_decode_workspace(a) > TQ_STATIC_DECODE_SCRATCH_BYTES). */
#define TQ_STATIC_DECODE_SCRATCH_BYTES (8u << 20)
tq_status tq_attn_decode_static(const tq_decode_args* a, tq_stream stream);

/* ------------------------------------------------------------------------ *
 * One decode step: append the new token's K and V, then attend.            *
 * ------------------------------------------------------------------------ *
 * The quantize-on-append of [A2A] "How to implement" (every cache update)
 * followed by the decode attention above, in one call, as three launches on
 * `stream`: the query preparation with both appends (one CTA per query row
 * and per appended vector), then the scan and the merge, each a programmatic
 * dependent of the launch before it (it may start while that one finishes
 * and waits for its results). Same results, bit for bit, as tq_quantize_kv(K),
 * tq_quantize_kv(V) and tq_attn_decode on one stream when batch * hkv is at
 * most 256 (up to that count tq_quantize_kv takes the same per-vector
 * kernel). All of the step's work is ordered after what precedes the call
 * on `stream` and before what follows it (also under CUDA graph capture).
 * q, k_new, v_new and out may be pinned host memory that the GPU addresses
 * directly (cudaHostAlloc / cudaHostRegister under unified addressing; on a
 * Grace-Blackwell node the host memory is reached over NVLink-C2C): the
 * kernels then read the inputs and write the output there, with no copy
 * operation, and the output is in host memory once the step's work on
 * `stream` has completed. Same results, bit for bit, as on device buffers. */
typedef struct {
    tq_decode_args attn;        /* the attention call: caches, q, lengths, out */
    const void* k_new;          /* device [batch*hkv][d] keys of the new token,
                                   row b*hkv + h                              */
    const void* v_new;          /* device [batch*hkv][d] values of the new token */
    int new_dtype;              /* TQ_F32 or TQ_BF16                           */
    const int32_t* append_pos;  /* device int32 [batch]: the slot (position)
                                   the new token takes in every row of batch b;
                                   outside [0, capacity) skips that batch row */
} tq_step_args;

/* Workspace bytes of tq_decode_step (that of its attention call; 0 on error). */
size_t tq_decode_step_workspace(const tq_step_args* a);
tq_status tq_decode_step(const tq_step_args* a, void* workspace, size_t ws_bytes, tq_stream stream);

/* ------------------------------------------------------------------------ *
 * Chunked-prefill attention from the packed cache.                         *
 * ------------------------------------------------------------------------ *
 * The decode attention above for a chunk of C consecutive tokens of each
 * sequence at once (the 32k-128k+ context windows of [A2A] "The KV cache
 * bottleneck in modern LLMs"): query i of sequence b is the token at position
 * q_start[b] + i and sees the cache slots 0 .. q_start[b] + i (causal; capped
 * at min(capacity, max_context)); the chunk's own keys and values must have
 * been quantized into the cache before the call (tq_quantize_kv), like every
 * other token. Query head h reads KV head gqa_map[h] (default h / (hq / hkv)). The logits, softmax
 * and value sum are decode's; the write-ups give decode only, so the causal
 * chunk is this library's reading. A query with no visible slot gives 0.
 * Kernels: query prep (q' and u), the scan split over the tokens, and a merge
 * of the splits (one warp per query row) with the un-rotation. The scan runs
 * on the tcgen05 tensor cores (128 query rows per CTA against 128-token
 * tiles; scores and the value sum accumulated in TMEM) when the keys have 1
 * or 2 code bits (PROD bits 2 or 3, or the 3 / 2 fractional rate), else on
 * mma.sync (64 query rows per CTA against 16-token tiles). */
typedef struct {
    const void* q;          /* device [batch][chunk][hq][d] of q_dtype         */
    int q_dtype;            /* TQ_F32 or TQ_BF16                              */
    int batch, chunk, hq, hkv, d;  /* d = 128; hq / hkv in {1, 2, 4, 8}       */
    const int32_t* q_start; /* device int32 [batch]: position of the chunk's
                               first token in each sequence                   */
    int max_context;        /* host: upper bound of q_start[b] + chunk (the
                               split plan); <= capacity                       */
    const int32_t* gqa_map; /* HOST int32 [hq] in [0, hkv), or NULL = h/(hq/hkv);
                               every KV head must serve hq/hkv query heads    */
    const tq_rotation* rot; /* uploaded                                       */
    const tq_qjl* qjl;      /* uploaded, m == k.m                             */
    tq_cache k;             /* PROD cache, rows == batch*hkv, m = 128         */
    tq_cache v;             /* MSE cache, rows == batch*hkv                   */
    float scale;            /* softmax scale; 0 -> 1/sqrt(d)                  */
    int n_splits;           /* token splits; 0 -> automatic                   */
    void* out;              /* device [batch][chunk][hq][d] of out_dtype,
                               16-byte aligned                                */
    int out_dtype;          /* TQ_F32 or TQ_BF16                              */
    tq_event scan_begin;    /* optional: recorded on `stream` right before and */
    tq_event scan_end;      /* after the scan kernel (for timing it)           */
} tq_prefill_args;

/* Workspace bytes of tq_attn_prefill (0 on invalid arguments); the workspace
 * must be 256-byte aligned. */
size_t tq_attn_prefill_workspace(const tq_prefill_args* a);
tq_status tq_attn_prefill(const tq_prefill_args* a, void* workspace, size_t ws_bytes, tq_stream stream);

/* ------------------------------------------------------------------------ *
 * Inner-product search from the codes.                                     *
 * ------------------------------------------------------------------------ *
 * [A2A] "Benchmarks and real-world performance" (GloVe d = 200 top-k recall)
 * and "Applications" (vector databases). Score of database row t for query
 * q: the decode logit l_t above (PROD database; an MSE database drops the
 * sign term). Returns per query the k largest scores, ties to the lower row
 * id, sorted descending. */
typedef struct {
    const float* queries;   /* device fp32 [nq][d]                            */
    int nq, d;
    const tq_rotation* rot; /* uploaded                                       */
    const tq_qjl* qjl;      /* uploaded when db.mode == TQ_PROD               */
    tq_cache db;            /* rows == 1, capacity >= n_db                    */
    int64_t n_db;
    int k;                  /* 1..32                                          */
    int32_t* ids;           /* device int32 [nq][k]                           */
    float* scores;          /* device fp32 [nq][k]                            */
} tq_topk_args;

size_t tq_score_topk_workspace(const tq_topk_args* a);
/* Scores on the tcgen05 tensor cores (database tiles de-quantized into shared
 * memory, queries as fp16 hi/lo halves, fp32 accumulators in TMEM) when d and
 * m are at most 256; otherwise on a SIMT kernel. Both rank the same scores. */
tq_status tq_score_topk(const tq_topk_args* a, void* workspace, size_t ws_bytes, tq_stream stream);
/* Process-wide switch: on != 0 makes tq_score_topk use the SIMT scan for
 * every shape (to compare the two); returns the previous setting. */
int tq_topk_force_simt(int on);
/* Process-wide switch: on != 0 makes tq_quantize_kv use the mma.sync kernel
 * for bf16 input at d = 128 (where it would take the tcgen05 kernel), to
 * compare the two; returns the previous setting. Both give the same codes,
 * norms and signs (the exact fp64 decision near every boundary). */
int tq_quantize_force_mma_sync(int on);
/* Process-wide switch: on != 0 makes tq_attn_prefill use the mma.sync scan
 * where it would take the tcgen05 one, to compare the two; returns the
 * previous setting. Query the workspace again after switching (the split
 * plans differ). */
int tq_prefill_force_mma_sync(int on);

/* ------------------------------------------------------------------------ *
 * Device error word.                                                       *
 * ------------------------------------------------------------------------ *
 * Library-level diagnostics; the pages define nothing of the kind. Each
 * device the library runs on has one 32-bit error word, zero at load time.
 * A bounded device-side wait that runs out sets a bit instead of spinning:
 *   TQ_DEVERR_SCAN_WAIT      a decode scan tile's copies did not land within
 *                            one second; that call's output is not valid
 *   TQ_DEVERR_SELFTEST_WAIT  tq_selftest_bounded_wait ran out (its purpose)
 *   TQ_DEVERR_QUANT_WAIT     a quantize CTA's operand fragments did not land
 *                            within one second; that call's output is not valid
 * tq_device_errors synchronises the current device, stores the word in
 * *flags_out (host, may be NULL), clears it when reset != 0, and returns
 * TQ_ERR_TIMEOUT when any bit was set, TQ_OK when none was, TQ_ERR_CUDA when
 * the device could not be read. */
#define TQ_DEVERR_SCAN_WAIT 1u
#define TQ_DEVERR_SELFTEST_WAIT 2u
#define TQ_DEVERR_QUANT_WAIT 4u
tq_status tq_device_errors(uint32_t* flags_out, int reset);

/* Self-test of the bounded wait: launches one warp on `stream` that waits on
 * an mbarrier nothing ever arrives on, for at most limit_us microseconds
 * (1..1000000; a wait checks its limit at least every 20 us, between
 * suspensions), then returns after setting TQ_DEVERR_SELFTEST_WAIT. */
tq_status tq_selftest_bounded_wait(uint32_t limit_us, tq_stream stream);

/* Self-test of the 5th-generation tensor-core path (tcgen05.mma with TMEM
 * accumulators) that the search kernel is built on: d[128][n] = a[128][k] *
 * b[n][k]^T, a and b device fp16 row-major, d device fp32 row-major, n in
 * {16, 32, 64, 128}, k a multiple of 16 up to 128; one CTA on `stream`. */
tq_status tq_selftest_umma_gemm(const void* a, const void* b, float* d, int n, int k, tq_stream stream);
/* The same product with the A operand taken from tensor memory: a is written
 * into TMEM with tcgen05.st (row r in lane r, two fp16 along k per 32-bit
 * column) and tcgen05.mma reads it there, as the search kernel does. */
tq_status tq_selftest_umma_gemm_tmem_a(const void* a, const void* b, float* d, int n, int k, tq_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
