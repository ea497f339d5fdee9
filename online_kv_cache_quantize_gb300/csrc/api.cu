// C entry points of libtq that touch the GPU: device uploads of the set-up
// handles, argument validation and the launches of the hot path.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <string>
#include <vector>
#include <algorithm>
#include <map>
#include <mutex>

#include <cuda_fp16.h>

#include "tq_internal.h"
#include "tq_launch.h"

namespace tqk {
cudaError_t launch_quantize_dense(const QuantParams& p, int dtype, int vpl, int prod, int cb, cudaStream_t s);
cudaError_t launch_quantize_rht(const QuantParams& p, int dtype, int vpl, int prod, int cb, cudaStream_t s);
}  // namespace tqk

namespace {

using tq::fail;

template <typename T>
tq_status upload(T** dst, const std::vector<T>& host) {
    if (cudaMalloc((void**)dst, host.size() * sizeof(T)) != cudaSuccess)
        return fail(TQ_ERR_CUDA, "cudaMalloc failed while uploading a handle");
    if (cudaMemcpy(*dst, host.data(), host.size() * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess)
        return fail(TQ_ERR_CUDA, "cudaMemcpy failed while uploading a handle");
    return TQ_OK;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

tq_status check_rot(const tq_rotation* rot, int d) {
    if (!rot) return fail(TQ_ERR_INVALID_ARG, "rotation handle is NULL");
    if (rot->d != d) return fail(TQ_ERR_INVALID_ARG, "rotation d does not match");
    int dev = -1;
    cudaGetDevice(&dev);
    if (rot->device < 0 || !rot->d_pi32) return fail(TQ_ERR_NO_DEVICE_COPY, "rotation not uploaded (tq_rotation_to_device)");
    if (rot->device != dev) return fail(TQ_ERR_INVALID_ARG, "rotation uploaded to another device");
    return TQ_OK;
}

tq_status check_qjl(const tq_qjl* q, int m, int d) {
    if (!q) return fail(TQ_ERR_INVALID_ARG, "QJL handle is NULL");
    if (q->d != d || q->m != m) return fail(TQ_ERR_INVALID_ARG, "QJL m/d does not match the cache");
    int dev = -1;
    cudaGetDevice(&dev);
    if (q->device < 0 || !q->d_st32) return fail(TQ_ERR_NO_DEVICE_COPY, "QJL not uploaded (tq_qjl_to_device)");
    if (q->device != dev) return fail(TQ_ERR_INVALID_ARG, "QJL uploaded to another device");
    return TQ_OK;
}

// Validates a cache descriptor; returns the code bits per coordinate.
// code bits of the two channel groups (equal for a one-width cache) and
// the codes' per-slot stride
// A PolarQuant cache (allow_polar) gives its level-1 and higher-level code
// widths as code_bits and code_bits2.
tq_status check_cache(const tq_cache& c, const char* what, int* code_bits, int* code_bits2 = nullptr,
                      int* code_stride = nullptr, bool allow_polar = false) {
    std::string w(what);
    if (c.mode == TQ_POLAR) {
        if (!allow_polar)
            return fail(TQ_ERR_UNSUPPORTED, w + ": PolarQuant caches are taken by tq_quantize_kv and tq_attn_decode only");
        if (c.bits < 1 || c.bits > 4 || c.bits2 < 1 || c.bits2 > 4)
            return fail(TQ_ERR_UNSUPPORTED, w + ": PolarQuant bits and bits2 must be 1..4");
        if (c.d != 128) return fail(TQ_ERR_UNSUPPORTED, w + ": PolarQuant caches need d = 128");
        if (c.rows < 0 || c.capacity < 0) return fail(TQ_ERR_INVALID_ARG, w + ": negative rows/capacity");
        if (!c.codes || !c.norm) return fail(TQ_ERR_INVALID_ARG, w + ": codes/norm plane is NULL");
        if (!aligned(c.codes, 16) || !aligned(c.norm, 2)) return fail(TQ_ERR_ALIGNMENT, w + ": codes must be 16-byte aligned, norm 2-byte");
        *code_bits = c.bits;
        if (code_bits2) *code_bits2 = c.bits2;
        if (code_stride) *code_stride = tq_polar_code_bytes(c.d, c.bits, c.bits2);
        return TQ_OK;
    }
    if (c.mode != TQ_MSE && c.mode != TQ_PROD) return fail(TQ_ERR_INVALID_ARG, w + ": mode must be TQ_MSE, TQ_PROD or TQ_POLAR");
    if (c.mode == TQ_MSE && (c.bits < 1 || c.bits > 4)) return fail(TQ_ERR_UNSUPPORTED, w + ": MSE bits must be 1..4");
    if (c.mode == TQ_PROD && (c.bits < 2 || c.bits > 5)) return fail(TQ_ERR_UNSUPPORTED, w + ": PROD bits must be 2..5");
    if (c.d < 3 || c.d > 256) return fail(TQ_ERR_UNSUPPORTED, w + ": d must be 3..256");
    if (c.rows < 0 || c.capacity < 0) return fail(TQ_ERR_INVALID_ARG, w + ": negative rows/capacity");
    if (!c.codes || !c.norm) return fail(TQ_ERR_INVALID_ARG, w + ": codes/norm plane is NULL");
    if (!aligned(c.codes, 16) || !aligned(c.norm, 2)) return fail(TQ_ERR_ALIGNMENT, w + ": codes must be 16-byte aligned, norm 2-byte");
    if (c.mode == TQ_PROD) {
        if (c.m < 1 || c.m > 256) return fail(TQ_ERR_UNSUPPORTED, w + ": m must be 1..256");
        if (!c.signs || !c.rnorm) return fail(TQ_ERR_INVALID_ARG, w + ": signs/rnorm plane is NULL");
        if (!aligned(c.signs, 16) || !aligned(c.rnorm, 2)) return fail(TQ_ERR_ALIGNMENT, w + ": signs must be 16-byte aligned, rnorm 2-byte");
    }
    *code_bits = c.mode == TQ_PROD ? c.bits - 1 : c.bits;
    int cb2 = *code_bits;
    if (c.bits2 != 0 && c.bits2 != c.bits) {
        if (c.bits2 != c.bits - 1)
            return fail(TQ_ERR_UNSUPPORTED, w + ": a fractional-rate cache needs bits2 = bits - 1 (3/2 or 4/3)");
        if (c.d != 128) return fail(TQ_ERR_UNSUPPORTED, w + ": a fractional-rate cache needs d = 128");
        if (c.mode == TQ_MSE && (c.bits < 2 || c.bits > 4)) return fail(TQ_ERR_UNSUPPORTED, w + ": MSE bits/bits2 out of range");
        if (c.mode == TQ_PROD && (c.bits < 3 || c.bits > 5)) return fail(TQ_ERR_UNSUPPORTED, w + ": PROD bits/bits2 out of range");
        cb2 = c.mode == TQ_PROD ? c.bits2 - 1 : c.bits2;
    }
    if (code_bits2) *code_bits2 = cb2;
    if (code_stride) *code_stride = tq_code_bytes2(c.d, *code_bits, cb2);
    return TQ_OK;
}

tq_status fill_codebook(int d, int cb, tqk::Codebook* out) {
    std::vector<double> c, t;
    tq_status s = tq::codebook(d, cb, c, t);
    if (s != TQ_OK) return s;
    std::memset(out, 0, sizeof(*out));
    out->levels = (int)c.size();
    for (size_t i = 0; i < c.size(); ++i) out->c[i] = (float)c[i];
    for (size_t i = 0; i < t.size(); ++i) {
        out->t[i] = (float)t[i];
        out->t64[i] = t[i];
    }
    for (size_t i = t.size(); i < (size_t)tqk::kMaxLevels - 1; ++i) {
        out->t[i] = 3.0e38f;
        out->t64[i] = 1e300;
    }
    return TQ_OK;
}

int vpl_for(int d) {
    if (d <= 64) return 2;
    if (d <= 128) return 4;
    if (d <= 224) return 7;
    return 8;
}

tq_status cuda_status(cudaError_t e, const char* where) {
    if (e == cudaSuccess) return TQ_OK;
    return fail(TQ_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// nearest fp16 value of x (normal range), ties to even, as a double
double fp16_round(double x) {
    if (x == 0.0) return 0.0;
    int e = 0;
    double m = std::frexp(x, &e);
    return std::ldexp(std::nearbyint(m * 2048.0), e - 11);
}

uint32_t fp16_bits(double v) { return (uint32_t)__half_as_ushort(__float2half_rn((float)fp16_round(v))); }

// Scale lam for the fp16 centroid tables of the tensor-core scan: among
// lam = 2^e (1 + k/2^18) with lam * max|c| in [1, 2), the one whose products
// lam * c_i lie closest (relative) to fp16 values, so the table entries
// carry the centroids almost exactly. c holds the positive centroids of one
// codebook, or of both groups of a fractional-rate cache (one lam serves
// both tables). Cached per (d, key).
double pick_lambda(int d, int key, const std::vector<double>& c) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, double> cache;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find({d, key});
        if (it != cache.end()) return it->second;
    }
    double mx = 0.0;
    for (double v : c) mx = std::max(mx, std::fabs(v));
    int e = 0;
    std::frexp(mx, &e);                          // 2^(e-1) <= mx < 2^e
    const double base = std::ldexp(1.0, 1 - e);  // base * mx in [1, 2)
    const int n = 1 << 18;
    double best = 1e300, best_l = base;
    for (int k = 0; k < n; ++k) {
        const double l = base * (1.0 + (double)k / n);
        double err = 0.0;
        for (size_t v = 0; v < c.size() && err < best; ++v) {
            const double x = l * c[v];
            err = std::max(err, std::fabs(fp16_round(x) - x) / x);
        }
        if (err < best) {
            best = err;
            best_l = l;
        }
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[{d, key}] = best_l;
    return best_l;
}

// the positive centroids of the codebooks of code bits cb and cb2 (a
// Lloyd-Max codebook is symmetric about 0, sorted ascending)
std::vector<double> positive_centroids(const std::vector<double>& c, const std::vector<double>* c2) {
    std::vector<double> out(c.begin() + c.size() / 2, c.end());
    if (c2) out.insert(out.end(), c2->begin() + c2->size() / 2, c2->end());
    return out;
}

void pair_table(const std::vector<double>& c, int bits, double lam, uint32_t* out) {
    const int n = 1 << bits;
    for (int x = 0; x < n * n; ++x) out[x] = fp16_bits(lam * c[x & (n - 1)]) | (fp16_bits(lam * c[x >> bits]) << 16);
}

// the part of lam * c that the fp16 table above drops, as a second fp16 table
void pair_table_lo(const std::vector<double>& c, int bits, double lam, uint32_t* out) {
    const int n = 1 << bits;
    auto lo = [&](int i) { return fp16_bits(lam * c[i] - fp16_round(lam * c[i])); };
    for (int x = 0; x < n * n; ++x) out[x] = lo(x & (n - 1)) | (lo(x >> bits) << 16);
}

// The tensor-core scans' centroid tables (decode and prefill): pair tables of
// lam * c for the key codes (with the lo residual table) and the value codes,
// and of the second channel group when the caches are fractional-rate.
template <typename P>
tq_status scan_tables(int d, int kb, int kb2, int vb, int vb2, P* p) {
    const bool two = kb2 != kb;
    std::vector<double> kc, vc, kc2, vc2, t;
    tq_status s;
    if ((s = tq::codebook(d, kb, kc, t)) != TQ_OK) return s;
    if ((s = tq::codebook(d, vb, vc, t)) != TQ_OK) return s;
    if (two && (s = tq::codebook(d, kb2, kc2, t)) != TQ_OK) return s;
    if (two && (s = tq::codebook(d, vb2, vc2, t)) != TQ_OK) return s;
    const double lam_k = pick_lambda(d, 16 * kb + kb2, positive_centroids(kc, two ? &kc2 : nullptr));
    const double lam_v = pick_lambda(d, 16 * vb + vb2, positive_centroids(vc, two ? &vc2 : nullptr));
    pair_table(kc, kb, lam_k, p->klut);
    pair_table_lo(kc, kb, lam_k, p->klut_lo);
    pair_table(vc, vb, lam_v, p->vlut);
    if (two) {
        pair_table(kc2, kb2, lam_k, p->klut2);
        pair_table_lo(kc2, kb2, lam_k, p->klut2_lo);
        pair_table(vc2, vb2, lam_v, p->vlut2);
    }
    p->inv_lam_k = (float)(1.0 / lam_k);
    p->inv_lam_v = (float)(1.0 / lam_v);
    return TQ_OK;
}

struct DecodePlan {
    int n_splits = 1, chunk = 1, group = 1;
    size_t off_frag = 0, off_part = 0, total = 0;
};

tq_status plan_decode(const tq_decode_args* a, DecodePlan* pl) {
    if (!a) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: args are NULL");
    if (a->batch < 1 || a->hq < 1 || a->hkv < 1) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: batch/hq/hkv must be >= 1");
    if (a->d != 128) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: d must be 128");
    if (a->hq > 256) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: hq must be <= 256");
    if (a->max_seq_len < 0) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: max_seq_len < 0");
    if (a->hq % a->hkv) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: hq must be a multiple of hkv");
    int g = a->hq / a->hkv;
    if (g != 1 && g != 2 && g != 4 && g != 8) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: group size must be 1, 2, 4 or 8");
    pl->group = g;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // each split covers a multiple of 64 tokens (4 warps x 16-token tiles)
    const int L = a->max_seq_len > 0 ? a->max_seq_len : 1;
    long long want = a->n_splits;
    if (want <= 0) {
        long long units = (long long)a->batch * a->hkv;
        want = ((long long)sms * 4 + units - 1) / units;
    }
    if (want > 65535) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: too many splits");
    int chunk = (int)((L + want - 1) / want);
    chunk = std::max(64, (chunk + 63) / 64 * 64);
    const int splits = (L + chunk - 1) / chunk;
    pl->n_splits = splits;
    pl->chunk = chunk;
    const size_t rows = (size_t)a->batch * a->hq;
    pl->off_frag = 0;
    pl->off_part = round_up(rows * tqk::kFragWords * sizeof(uint32_t), 256);
    pl->total = pl->off_part + round_up(rows * (size_t)splits * (a->d + tqk::kPartPad) * sizeof(float), 256);
    return TQ_OK;
}

}  // namespace

namespace {

// B-operand fragments of mma.sync m16n8k16 for a 128 x 128 map y = W x:
// element (k, n) of n-tile nt in k-step kk is W[sigma(nt, n)][pi(kk, k)]
// with the output permutation sigma(nt, n) = 32 (n / 2) + 2 nt + n % 2 (so
// accumulators land in the quantize kernel's quad layout) and the input
// permutation pi(kk, 2c + e) = 32c + 4kk + e, pi(kk, 2c + 8 + e) = 32c + 4kk
// + 2 + e (so thread c of a quad builds its A fragments from its own
// coordinates 32c .. 32c + 31), stored [kk][nt][lane] as two words.
template <typename F>
std::vector<uint2v> mma_b_fragments(F wbits) {
    std::vector<uint2v> out((size_t)8 * 16 * 32);
    for (int kk = 0; kk < 8; ++kk)
        for (int nt = 0; nt < 16; ++nt)
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, c = lane & 3;
                const int o = 32 * (g >> 1) + 2 * nt + (g & 1);
                auto e = [&](int k) {
                    const int cc = (k & 7) >> 1, hi = k >> 3, ee = k & 1;
                    return (uint32_t)wbits(o, 32 * cc + 4 * kk + 2 * hi + ee);
                };
                uint2v v;
                v.x = e(2 * c) | (e(2 * c + 1) << 16);
                v.y = e(2 * c + 8) | (e(2 * c + 9) << 16);
                out[((size_t)kk * 16 + nt) * 32 + lane] = v;
            }
    return out;
}

uint16_t bf16_bits_of(double exact_bf16_value) {
    const float f = (float)exact_bf16_value;
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

// A 128 x 128 bf16 operand of tcgen05.mma, K-major with the 128-byte
// swizzle: two halves of 64 elements along K (16 KB each), row n of a half
// at n * 128 bytes, its 16-byte chunk j (elements 8j .. 8j+7) stored at chunk
// j ^ (n % 8); 8-row atoms of 1024 bytes.
template <typename F>
std::vector<uint16_t> umma_operand_128(F bits) {
    std::vector<uint16_t> out((size_t)128 * 128);
    for (int n = 0; n < 128; ++n)
        for (int k = 0; k < 128; ++k) {
            const int half = k >> 6, kk = k & 63;
            const size_t byte = (size_t)half * 16384 + (size_t)n * 128 + (size_t)(((kk >> 3) ^ (n & 7)) << 4) + (kk & 7) * 2;
            out[byte / 2] = bits(n, k);
        }
    return out;
}

}  // namespace

namespace {

// tq_score_topk uses the SIMT scan even where the tcgen05 scan fits (for
// comparing the two; see tq_topk_force_simt)
bool g_topk_simt = false;

// Appends of at most this many vectors (d = 128, keys m = 128) take the
// CTA-per-vector kernel: a few microseconds of latency however few vectors
// there are, where the 16-vector tiles of the tensor-core kernel would leave
// one warp working through a serial chain per tile.
constexpr int64_t kSmallAppend = 256;

// tq_quantize_kv may take the tcgen05 kernel (tq_quantize_force_mma_sync
// turns it off, for comparing the two kernels)
bool g_quant_umma = true;

// tq_attn_prefill takes the tcgen05 kernel where it applies
// (tq_prefill_force_mma_sync turns it off, for comparing the two kernels)
bool g_prefill_umma = true;

struct QuantLaunch {
    tqk::QuantParams p;
    int dtype = 0, vpl = 1, cb = 1;
    bool rht = false, prod = false, mma = false, small = false, umma = false, polar = false;
    tqk::PolarQuantParams pq;  // PolarQuant keys
    const void* w_umma = nullptr;
    const void* s_umma = nullptr;
};

// the append role of the step-prep launch for one quantize call
void step_append(const QuantLaunch& L, tqk::StepPrepParams* sp) {
    if (L.prod) {
        sp->k = L.p;
        sp->k_dtype = L.dtype;
        sp->k_cb = L.cb;
        sp->k_rht = L.rht ? 1 : 0;
    } else {
        sp->v = L.p;
        sp->v_dtype = L.dtype;
        sp->v_cb = L.cb;
        sp->v_rht = L.rht ? 1 : 0;
    }
}

struct DecodeLaunch {
    DecodePlan pl;
    tqk::PrepParams pp;
    tqk::DecodeParams dp;
    tqk::CombineParams cp;
    int kb = 0, vb = 0;
    bool two = false;  // fractional-rate key and value caches
    cudaEvent_t scan_begin = nullptr, scan_end = nullptr;
    bool polar = false;  // PolarQuant keys: the polar scan instead of the tensor-core one
    tqk::PolarDecodeParams pdp;
};

// The query heads of each KV head from a host gqa_map (every KV head serving
// `group` query heads); *use = 0 when gqa_map is NULL.
tq_status head_table(const tq_decode_args* a, int group, int16_t* table, int* use) {
    *use = 0;
    if (!a->gqa_map) return TQ_OK;
    std::vector<int> count(a->hkv, 0);
    for (int h = 0; h < a->hq; ++h) {
        const int g = a->gqa_map[h];
        if (g < 0 || g >= a->hkv) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: gqa_map entry out of range");
        if (count[g] >= group) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: every KV head must serve hq/hkv query heads");
        table[g * group + count[g]++] = (int16_t)h;
    }
    *use = 1;
    return TQ_OK;
}

// Decode over PolarQuant keys and a one-width MSE value cache: the query
// prep writes q' (fp32) where the tensor-core scan keeps its B operands,
// the polar scan writes the same split partials, the merge is shared.
tq_status polar_decode_prepare(const tq_decode_args* a, void* workspace, size_t ws_bytes, DecodeLaunch* D) {
    const DecodePlan& pl = D->pl;
    int kb = 0, kb2 = 0, kstride = 0, vb = 0, vb2 = 0, vstride = 0;
    tq_status s;
    if ((s = check_cache(a->k, "tq_attn_decode k", &kb, &kb2, &kstride, true)) != TQ_OK) return s;
    if ((s = check_cache(a->v, "tq_attn_decode v", &vb, &vb2, &vstride)) != TQ_OK) return s;
    if (a->v.mode != TQ_MSE || vb2 != vb)
        return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: PolarQuant keys take a one-width MSE value cache");
    if (!tqk::polar_decode_supported(kb, kb2))
        return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: PolarQuant (bits, bits2) must be (2,2), (3,2), (4,2), (4,3), (3,3) or (4,4)");
    if (a->k.d != a->d || a->v.d != a->d) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: cache d does not match");
    const int64_t rows = (int64_t)a->batch * a->hkv;
    if (a->k.rows != rows || a->v.rows != rows) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: cache rows must be batch*hkv");
    if (a->k.capacity != a->v.capacity) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: k and v capacity differ");
    if (a->max_seq_len > a->k.capacity) return fail(TQ_ERR_CAPACITY, "tq_attn_decode: max_seq_len exceeds the capacity");
    if (!aligned(a->v.codes, 16)) return fail(TQ_ERR_ALIGNMENT, "tq_attn_decode: value codes must be 16-byte aligned");
    if ((s = check_rot(a->rot, a->d)) != TQ_OK) return s;
    if (!a->q || !a->out || !a->seq_lens) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: q/out/seq_lens is NULL");
    if (a->q_dtype != TQ_F32 && a->q_dtype != TQ_BF16) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: q_dtype must be F32 or BF16");
    if (a->out_dtype != TQ_F32 && a->out_dtype != TQ_BF16) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: out_dtype must be F32 or BF16");
    tqk::PolarDecodeParams& dp = D->pdp;
    std::memset(&dp, 0, sizeof(dp));
    if ((s = head_table(a, pl.group, dp.head_table, &dp.use_table)) != TQ_OK) return s;
    // the workspace last: every other argument error takes precedence
    if (!workspace || ws_bytes < pl.total) return fail(TQ_ERR_WORKSPACE, "tq_attn_decode: workspace missing or too small");
    if (!aligned(workspace, 256)) return fail(TQ_ERR_ALIGNMENT, "tq_attn_decode: workspace must be 256-byte aligned");
    char* ws = (char*)workspace;
    float* qprime = (float*)(ws + pl.off_frag);  // rows x kFragWords words hold rows x 128 floats
    float* part = (float*)(ws + pl.off_part);

    tqk::PrepParams& pp = D->pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.q = a->q;
    pp.q_dtype = a->q_dtype == TQ_BF16 ? 1 : 0;
    pp.rows = (int64_t)a->batch * a->hq;
    pp.d = a->d;
    pp.pit32 = a->rot->d_pit32;
    pp.sgn = a->rot->d_sign;
    pp.rht = a->rot->kind == TQ_ROT_RHT;
    pp.inv_sqrt_d = (float)(1.0 / std::sqrt((double)a->d));
    pp.qprime = qprime;

    std::vector<double> vc, vt;
    if ((s = tq::codebook(a->d, vb, vc, vt)) != TQ_OK) return s;
    for (size_t i = 0; i < vc.size(); ++i) dp.vc[i] = (float)vc[i];
    for (int lev = 1; lev <= tqk::kPolarLevels; ++lev) {
        std::vector<double> cc, tt;
        if ((s = tq::polar_codebook(lev, lev == 1 ? kb : kb2, cc, tt)) != TQ_OK) return s;
        for (size_t i = 0; i < cc.size(); ++i) {
            const float co = (float)std::cos(cc[i]), si = (float)std::sin(cc[i]);
            if (lev == 1) {
                dp.c1cos[i] = co;
                dp.c1sin[i] = si;
            } else {
                dp.ccos[lev - 2][i] = co;
                dp.csin[lev - 2][i] = si;
            }
        }
    }
    dp.qprime = qprime;
    dp.batch = a->batch;
    dp.hq = a->hq;
    dp.hkv = a->hkv;
    dp.group = pl.group;
    dp.seq_lens = a->seq_lens;
    dp.capacity = a->k.capacity;
    dp.kcodes = a->k.codes;
    dp.kcode_stride = kstride;
    dp.knorm = a->k.norm;
    dp.vcodes = a->v.codes;
    dp.vcode_stride = vstride;
    dp.vnorm = a->v.norm;
    dp.vbits = vb;
    const double scale = a->scale != 0.0f ? (double)a->scale : 1.0 / std::sqrt((double)a->d);
    dp.scale_log2 = (float)(scale * 1.4426950408889634);
    dp.n_splits = pl.n_splits;
    dp.chunk = pl.chunk;
    dp.partial = part;
    dp.logits = a->logits;
    dp.max_seq_len = a->max_seq_len;
    D->polar = true;
    D->kb = kb;
    D->vb = kb2;  // the polar scan's (bits, bits2)
    D->scan_begin = (cudaEvent_t)a->scan_begin;
    D->scan_end = (cudaEvent_t)a->scan_end;

    tqk::CombineParams& cp = D->cp;
    std::memset(&cp, 0, sizeof(cp));
    cp.partial = part;
    cp.rows = a->batch * a->hq;
    cp.d = a->d;
    cp.n_splits = pl.n_splits;
    cp.pi32 = a->rot->d_pi32;
    cp.sgn = a->rot->d_sign;
    cp.rht = a->rot->kind == TQ_ROT_RHT;
    cp.inv_sqrt_d = (float)(1.0 / std::sqrt((double)a->d));
    cp.out = a->out;
    cp.out_dtype = a->out_dtype == TQ_BF16 ? 1 : 0;
    return TQ_OK;
}

// The PolarQuant part of a quantize launch: the angle codebooks of the 7
// levels (boundaries as fp32 cos/sin pairs and fp64 values) and the guard
// band. The fp32 rotation is good to a few 1e-7 of the unit vector (RHT
// butterflies, or a 128-term fp32 dot product for the dense Pi) and a cross
// product b cos t - a sin t moves by at most the error of its pair; the
// bands sit an order of magnitude above the typical error.
tq_status polar_prepare(const tq_cache& c, QuantLaunch* L) {
    tqk::PolarQuantParams& pq = L->pq;
    std::memset(&pq.cb, 0, sizeof(pq.cb));
    for (int lev = 1; lev <= tqk::kPolarLevels; ++lev) {
        std::vector<double> cc, tt;
        const tq_status s = tq::polar_codebook(lev, lev == 1 ? c.bits : c.bits2, cc, tt);
        if (s != TQ_OK) return s;
        for (size_t j = 0; j < tt.size(); ++j) {
            pq.cb.tc[lev - 1][j] = (float)std::cos(tt[j]);
            pq.cb.ts[lev - 1][j] = (float)std::sin(tt[j]);
            pq.cb.tc64[lev - 1][j] = std::cos(tt[j]);
            pq.cb.ts64[lev - 1][j] = std::sin(tt[j]);
        }
    }
    pq.q = L->p;
    pq.bits1 = c.bits;
    pq.bits2 = c.bits2;
    pq.guard = L->rht ? 3.0e-6f : 4.0e-6f;
    L->polar = true;
    return TQ_OK;
}

// Validates a quantize call and fills its launch; *empty = nothing to do.
tq_status quant_prepare(const tq_quant_args* a, QuantLaunch* L, bool* empty) {
    *empty = false;
    if (!a) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_kv: args are NULL");
    int cb = 0, cb2 = 0, cstride = 0;
    tq_status s = check_cache(a->cache, "tq_quantize_kv cache", &cb, &cb2, &cstride, true);
    if (s != TQ_OK) return s;
    const tq_cache& c = a->cache;
    if ((s = check_rot(a->rot, c.d)) != TQ_OK) return s;
    const bool prod = c.mode == TQ_PROD;
    if (prod && (s = check_qjl(a->qjl, c.m, c.d)) != TQ_OK) return s;
    if (a->n < 0) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_kv: n < 0");
    if (a->n == 0) {
        *empty = true;
        return TQ_OK;
    }
    if (!a->x) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_kv: x is NULL");
    if (a->x_dtype != TQ_F32 && a->x_dtype != TQ_BF16) return fail(TQ_ERR_UNSUPPORTED, "tq_quantize_kv: x_dtype must be TQ_F32 or TQ_BF16");
    const size_t esz = a->x_dtype == TQ_F32 ? 4 : 2;
    if (!aligned(a->x, esz)) return fail(TQ_ERR_ALIGNMENT, "tq_quantize_kv: x misaligned for its dtype");
    if (a->x_stride < c.d) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_kv: x_stride < d");
    const int64_t total = c.rows * c.capacity;
    if (a->dst_slot) {
        if (!aligned(a->dst_slot, 8)) return fail(TQ_ERR_ALIGNMENT, "tq_quantize_kv: dst_slot misaligned");
    } else if (a->append_pos) {
        if (a->heads < 1 || a->n % a->heads) return fail(TQ_ERR_INVALID_ARG, "tq_quantize_kv: n must be a multiple of heads");
        if (a->n != c.rows) return fail(TQ_ERR_CAPACITY, "tq_quantize_kv: append mode needs n == cache rows");
    } else {
        if (a->slot0 < 0 || a->slot0 + a->n > total) return fail(TQ_ERR_CAPACITY, "tq_quantize_kv: slot0 + n exceeds rows*capacity");
    }
    const bool rht = a->rot->kind == TQ_ROT_RHT;
    if (rht && c.d != 64 && c.d != 128 && c.d != 256) return fail(TQ_ERR_UNSUPPORTED, "tq_quantize_kv: RHT kernels need d in {64, 128, 256}");
    if (prod && c.m > 32 * vpl_for(c.d)) return fail(TQ_ERR_UNSUPPORTED, "tq_quantize_kv: m must be <= d rounded up to the kernel width");

    tqk::QuantParams& p = L->p;
    std::memset(&p, 0, sizeof(p));
    p.x = a->x;
    p.x_stride = a->x_stride;
    p.n = a->n;
    p.dst_slot = a->dst_slot;
    p.append_pos = a->append_pos;
    p.heads = a->heads;
    p.slot0 = a->slot0;
    p.total_slots = total;
    p.capacity = c.capacity;
    p.codes = c.codes;
    p.code_stride = cstride;
    p.signs = c.signs;
    p.sign_stride = prod ? tq_sign_bytes(c.m) : 0;
    p.norm = c.norm;
    p.rnorm = c.rnorm;
    p.pit32 = a->rot->d_pit32;
    p.pi64 = a->rot->d_pi64;
    p.sgn = a->rot->d_sign;
    p.st32 = prod ? a->qjl->d_st32 : nullptr;
    p.s16 = prod ? a->qjl->d_s16 : nullptr;
    p.d = c.d;
    p.m = prod ? c.m : 0;
    p.inv_sqrt_d = (float)(1.0 / std::sqrt((double)c.d));
    p.guard = rht ? 1.0e-6f : (float)(3.0e-8 * c.d);
    L->dtype = a->x_dtype == TQ_F32 ? 0 : 1;
    L->rht = rht;
    if (c.mode == TQ_POLAR) return polar_prepare(c, L);
    if ((s = fill_codebook(c.d, cb, &p.cb)) != TQ_OK) return s;
    p.code_bits2 = cb2 != cb ? cb2 : 0;
    if (p.code_bits2 && (s = fill_codebook(c.d, cb2, &p.cb2)) != TQ_OK) return s;
    if (cudaError_t ew = tqk::device_error_word(&p.err); ew != cudaSuccess) return cuda_status(ew, "tq_quantize_kv error word");
    L->dtype = a->x_dtype == TQ_F32 ? 0 : 1;
    L->vpl = vpl_for(c.d);
    L->rht = rht;
    L->prod = prod;
    L->cb = cb;
    p.pi_frag = a->rot->d_pi_frag;
    p.s_frag = prod ? a->qjl->d_s_frag : nullptr;
    // d = 128 (keys m = 128): up to kSmallAppend vectors the CTA-per-vector
    // kernel, more the tensor-core kernel (16-byte aligned rows); otherwise
    // the warp-per-vector kernel (any d <= 256). A two-width cache takes the
    // CTA-per-vector kernel where the tensor-core one does not apply.
    if (p.code_bits2 && prod && c.m != 128) return fail(TQ_ERR_UNSUPPORTED, "tq_quantize_kv: a fractional-rate key cache needs m = 128");
    const bool mma_ok = c.d == 128 && (!prod || (c.m == 128 && p.s_frag)) && (rht || p.pi_frag) &&
                        aligned(a->x, 16) && (a->x_stride * (int64_t)esz) % 16 == 0;
    L->small = c.d == 128 && (!prod || c.m == 128) && (a->n <= kSmallAppend || (p.code_bits2 != 0 && !mma_ok));
    L->mma = !L->small && mma_ok;
    // bf16 input at one code width: the tcgen05 kernel
    L->w_umma = a->rot->d_w_umma;
    L->s_umma = prod ? a->qjl->d_s_umma : nullptr;
    L->umma = L->mma && g_quant_umma && L->w_umma && (!prod || L->s_umma) &&
              tqk::quantize_umma_supported(p, L->dtype, cb);
    // The tensor-core rotation rounds only in its fp32 accumulation (8 steps
    // of 16 exact products for RHT; 24 with the dense limbs, whose split
    // itself is good to 2^-25 of each entry): at most about one fp32 ulp of
    // the largest partial sum per step, under 1e-6 of the unit vector for
    // RHT and 1.5e-6 dense. The guard bands sit above those bounds.
    if (L->umma) p.guard = rht ? 1.2e-6f : 2.0e-6f;
    return TQ_OK;
}

cudaError_t quant_launch(const QuantLaunch& L, cudaStream_t st) {
    if (L.polar) return tqk::launch_polar_quantize(L.pq, L.dtype, L.rht ? 1 : 0, st);
    if (L.small) {
        tqk::StepPrepParams sp;
        std::memset(&sp, 0, sizeof(sp));
        step_append(L, &sp);
        return tqk::launch_step_prep(sp, st);
    }
    if (L.umma) return tqk::launch_quantize_umma(L.p, L.w_umma, L.s_umma, L.rht ? 1 : 0, L.prod ? 1 : 0, L.cb, st);
    if (L.mma && L.p.code_bits2)
        return tqk::launch_quantize_mma2(L.p, L.dtype, L.rht ? 1 : 0, L.prod ? 1 : 0, L.cb, st);
    if (L.mma) return tqk::launch_quantize_mma(L.p, L.dtype, L.rht ? 1 : 0, L.prod ? 1 : 0, L.cb, st);
    if (L.rht) return tqk::launch_quantize_rht(L.p, L.dtype, L.vpl, L.prod ? 1 : 0, L.cb, st);
    return tqk::launch_quantize_dense(L.p, L.dtype, L.vpl, L.prod ? 1 : 0, L.cb, st);
}

// Validates a decode call and fills its three launches.
tq_status decode_prepare(const tq_decode_args* a, void* workspace, size_t ws_bytes, DecodeLaunch* D) {
    DecodePlan& pl = D->pl;
    tq_status s = plan_decode(a, &pl);
    if (s != TQ_OK) return s;
    if (a->k.mode == TQ_POLAR) return polar_decode_prepare(a, workspace, ws_bytes, D);
    int kb = 0, vb = 0, kb2 = 0, vb2 = 0;
    if ((s = check_cache(a->k, "tq_attn_decode k", &kb, &kb2)) != TQ_OK) return s;
    if ((s = check_cache(a->v, "tq_attn_decode v", &vb, &vb2)) != TQ_OK) return s;
    const bool two = kb2 != kb;
    if ((vb2 != vb) != two)
        return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: keys and values must both be fractional-rate caches, or neither");
    if (a->k.mode != TQ_PROD || a->v.mode != TQ_MSE) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: keys must be PROD and values MSE");
    if (a->k.d != a->d || a->v.d != a->d) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: cache d does not match");
    if (a->k.m != 128) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: m must be 128");
    const int64_t rows = (int64_t)a->batch * a->hkv;
    if (a->k.rows != rows || a->v.rows != rows) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: cache rows must be batch*hkv");
    if (a->k.capacity != a->v.capacity) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: k and v capacity differ");
    if (a->max_seq_len > a->k.capacity) return fail(TQ_ERR_CAPACITY, "tq_attn_decode: max_seq_len exceeds the capacity");
    if (a->k.capacity % 16) return fail(TQ_ERR_ALIGNMENT, "tq_attn_decode: cache capacity must be a multiple of 16");
    if (!aligned(a->k.norm, 16) || !aligned(a->k.rnorm, 16) || !aligned(a->v.norm, 16) || !aligned(a->v.codes, 16))
        return fail(TQ_ERR_ALIGNMENT, "tq_attn_decode: every cache plane must be 16-byte aligned (bulk copies)");
    if ((s = check_rot(a->rot, a->d)) != TQ_OK) return s;
    if ((s = check_qjl(a->qjl, a->k.m, a->d)) != TQ_OK) return s;
    if (!a->q || !a->out || !a->seq_lens) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: q/out/seq_lens is NULL");
    if (a->q_dtype != TQ_F32 && a->q_dtype != TQ_BF16) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: q_dtype must be F32 or BF16");
    if (a->out_dtype != TQ_F32 && a->out_dtype != TQ_BF16) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_decode: out_dtype must be F32 or BF16");
    tqk::DecodeParams& dp = D->dp;
    std::memset(&dp, 0, sizeof(dp));
    if ((s = head_table(a, pl.group, dp.head_table, &dp.use_table)) != TQ_OK) return s;
    // the workspace last: every other argument error takes precedence
    if (!workspace || ws_bytes < pl.total) return fail(TQ_ERR_WORKSPACE, "tq_attn_decode: workspace missing or too small");
    if (!aligned(workspace, 256)) return fail(TQ_ERR_ALIGNMENT, "tq_attn_decode: workspace must be 256-byte aligned");
    char* ws = (char*)workspace;
    uint32_t* frag = (uint32_t*)(ws + pl.off_frag);
    float* part = (float*)(ws + pl.off_part);

    tqk::PrepParams& pp = D->pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.q = a->q;
    pp.q_dtype = a->q_dtype == TQ_BF16 ? 1 : 0;
    pp.rows = (int64_t)a->batch * a->hq;
    pp.d = a->d;
    pp.m = a->k.m;
    pp.pit32 = a->rot->d_pit32;
    pp.sgn = a->rot->d_sign;
    pp.rht = a->rot->kind == TQ_ROT_RHT;
    pp.inv_sqrt_d = (float)(1.0 / std::sqrt((double)a->d));
    pp.st32 = a->qjl->d_st32;
    pp.s16 = a->qjl->d_s16;
    pp.frag = frag;
    pp.qjl_scale = (float)(std::sqrt(M_PI / 2.0) / a->k.m);

    std::vector<double> kc, kt, vc, vt;
    if ((s = tq::codebook(a->d, kb, kc, kt)) != TQ_OK) return s;
    if ((s = tq::codebook(a->d, vb, vc, vt)) != TQ_OK) return s;
    dp.frag = frag;
    dp.batch = a->batch;
    dp.hq = a->hq;
    dp.hkv = a->hkv;
    dp.d = a->d;
    dp.m = a->k.m;
    dp.group = pl.group;
    dp.seq_lens = a->seq_lens;
    dp.capacity = a->k.capacity;
    dp.kcodes = a->k.codes;
    dp.kcode_stride = tq_code_bytes2(a->d, kb, kb2);
    dp.ksigns = a->k.signs;
    dp.ksign_stride = tq_sign_bytes(a->k.m);
    dp.knorm = a->k.norm;
    dp.krnorm = a->k.rnorm;
    dp.vcodes = a->v.codes;
    dp.vcode_stride = tq_code_bytes2(a->d, vb, vb2);
    dp.vnorm = a->v.norm;
    for (size_t i = 0; i < kc.size(); ++i) dp.kc[i] = (float)kc[i];
    for (size_t i = 0; i < vc.size(); ++i) dp.vc[i] = (float)vc[i];
    if ((s = scan_tables(a->d, kb, kb2, vb, vb2, &dp)) != TQ_OK) return s;
    dp.qjl_scale = (float)(std::sqrt(M_PI / 2.0) / a->k.m);
    const double scale = a->scale != 0.0f ? (double)a->scale : 1.0 / std::sqrt((double)a->d);
    dp.scale_log2 = (float)(scale * 1.4426950408889634);
    dp.n_splits = pl.n_splits;
    dp.chunk = pl.chunk;
    dp.partial = part;
    dp.logits = a->logits;
    dp.max_seq_len = a->max_seq_len;
    cudaError_t e = tqk::device_error_word(&dp.err);
    if (e != cudaSuccess) return cuda_status(e, "tq_attn_decode error word");
    D->kb = kb;
    D->vb = vb;
    D->two = two;
    D->scan_begin = (cudaEvent_t)a->scan_begin;
    D->scan_end = (cudaEvent_t)a->scan_end;

    tqk::CombineParams& cp = D->cp;
    std::memset(&cp, 0, sizeof(cp));
    cp.partial = part;
    cp.rows = a->batch * a->hq;
    cp.d = a->d;
    cp.n_splits = pl.n_splits;
    cp.pi32 = a->rot->d_pi32;
    cp.sgn = a->rot->d_sign;
    cp.err = dp.err;
    cp.rht = a->rot->kind == TQ_ROT_RHT;
    cp.inv_sqrt_d = (float)(1.0 / std::sqrt((double)a->d));
    cp.out = a->out;
    cp.out_dtype = a->out_dtype == TQ_BF16 ? 1 : 0;
    return TQ_OK;
}

// The step-prep launch (the query prep, plus the appends a decode step adds
// to `sp`), then the scan and the merge, each a programmatic dependent of the
// launch before it on st.
tq_status decode_launch(const DecodeLaunch& D, cudaStream_t st, tqk::StepPrepParams* sp) {
    tqk::StepPrepParams own;
    if (!sp) {
        std::memset(&own, 0, sizeof(own));
        sp = &own;
    }
    sp->pp = D.pp;
    cudaError_t e = tqk::launch_step_prep(*sp, st);
    if (e != cudaSuccess) return cuda_status(e, "tq_attn_decode query prep");
    if (D.scan_begin && (e = cudaEventRecord(D.scan_begin, st)) != cudaSuccess)
        return cuda_status(e, "tq_attn_decode scan_begin");
    e = D.polar ? tqk::launch_polar_decode(D.pdp, D.kb, D.vb, st) : tqk::launch_decode_mma(D.dp, D.kb, D.vb, D.two, st);
    if (e != cudaSuccess) return cuda_status(e, "tq_attn_decode scan");
    if (D.scan_end && (e = cudaEventRecord(D.scan_end, st)) != cudaSuccess)
        return cuda_status(e, "tq_attn_decode scan_end");
    // many rows with few splits each (batched decode): one warp per row;
    // otherwise the wide merge, whose 1024 threads per row load the splits of
    // a long row in one round of latency
    const bool few = D.cp.n_splits <= 16 && D.cp.rows >= 128 && D.cp.d == 128 && aligned(D.cp.out, 16);
    e = few ? tqk::launch_merge_rows(D.cp, st) : tqk::launch_combine(D.cp, st);
    return cuda_status(e, "tq_attn_decode combine");
}

}  // namespace

namespace {

// One prepared decode call per thread. A decode loop passes the same
// arguments every step (only the device-side lengths, positions and the
// data change), so the last call's validation, split plan, lookup tables and
// parameter blocks are reused when its argument bytes, the host GQA map, the
// workspace, the current device and the handle generation all match; any
// difference prepares the call from scratch.
struct PreparedCall {
    bool valid = false;
    std::vector<unsigned char> key, probe;
    DecodeLaunch D;
    tqk::StepPrepParams sp;

    void build(std::vector<unsigned char>& k, const void* args, size_t n, const tq_decode_args& at, const void* ws,
               size_t wsb) const {
        int dev = -1;
        cudaGetDevice(&dev);
        const uint64_t gen = tq::handle_generation();
        const size_t nmap = at.gqa_map ? (size_t)std::max(at.hq, 0) * sizeof(int32_t) : 0;
        k.resize(n + nmap + sizeof(ws) + sizeof(wsb) + sizeof(dev) + sizeof(gen));
        unsigned char* o = k.data();
        std::memcpy(o, args, n);
        o += n;
        if (nmap) std::memcpy(o, at.gqa_map, nmap);
        o += nmap;
        std::memcpy(o, &ws, sizeof(ws));
        o += sizeof(ws);
        std::memcpy(o, &wsb, sizeof(wsb));
        o += sizeof(wsb);
        std::memcpy(o, &dev, sizeof(dev));
        o += sizeof(dev);
        std::memcpy(o, &gen, sizeof(gen));
    }
    bool match(const void* args, size_t n, const tq_decode_args& at, const void* ws, size_t wsb) {
        build(probe, args, n, at, ws, wsb);
        return valid && probe == key;
    }
    void remember() {  // after a successful prepare of the arguments last passed to match()
        key.swap(probe);
        valid = true;
    }
};
thread_local PreparedCall t_decode_call, t_step_call;

}  // namespace

extern "C" {

tq_status tq_rotation_to_device(tq_rotation* rot) {
    tq::bump_handle_generation();
    if (!rot) return fail(TQ_ERR_INVALID_ARG, "tq_rotation_to_device: NULL handle");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(TQ_ERR_CUDA, "tq_rotation_to_device: no CUDA device");
    if (rot->device == dev && rot->d_pi32) return TQ_OK;
    if (rot->device >= 0) return fail(TQ_ERR_INVALID_ARG, "tq_rotation_to_device: already on another device");
    const int d = rot->d;
    std::vector<float> pi32((size_t)d * d), pit32((size_t)d * d);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            pi32[(size_t)i * d + j] = (float)rot->pi[(size_t)i * d + j];
            pit32[(size_t)j * d + i] = (float)rot->pi[(size_t)i * d + j];
        }
    std::vector<float> sg(d, 1.0f);
    for (int i = 0; i < d && i < (int)rot->signs.size(); ++i) sg[i] = (float)rot->signs[i];
    tq_status s;
    if ((s = upload(&rot->d_pi32, pi32)) != TQ_OK) return s;
    if ((s = upload(&rot->d_pit32, pit32)) != TQ_OK) return s;
    if ((s = upload(&rot->d_pi64, rot->pi)) != TQ_OK) return s;
    if ((s = upload(&rot->d_sign, sg)) != TQ_OK) return s;
    if (d == 128 && rot->kind == TQ_ROT_DENSE_QR) {
        // three bf16 limbs of Pi (about 24 bits), concatenated limb-major
        std::vector<double> l1((size_t)d * d), l2((size_t)d * d), l3((size_t)d * d);
        for (size_t i = 0; i < l1.size(); ++i) {
            l1[i] = tq::round_bf16(rot->pi[i]);
            l2[i] = tq::round_bf16(rot->pi[i] - l1[i]);
            l3[i] = tq::round_bf16(rot->pi[i] - l1[i] - l2[i]);
        }
        std::vector<uint2v> frag;
        for (const std::vector<double>* l : {&l1, &l2, &l3}) {
            auto f = mma_b_fragments([&](int o, int k) { return bf16_bits_of((*l)[(size_t)o * d + k]); });
            frag.insert(frag.end(), f.begin(), f.end());
        }
        if ((s = upload(&rot->d_pi_frag, frag)) != TQ_OK) return s;
        std::vector<uint16_t> w;
        for (const std::vector<double>* l : {&l1, &l2, &l3}) {
            auto t = umma_operand_128([&](int n, int k) { return bf16_bits_of((*l)[(size_t)n * d + k]); });
            w.insert(w.end(), t.begin(), t.end());
        }
        if ((s = upload(&rot->d_w_umma, w)) != TQ_OK) return s;
    }
    if (d == 128 && rot->kind == TQ_ROT_RHT) {
        // sqrt(d) Pi = H diag(s): every entry +-1, exact in bf16
        auto w = umma_operand_128([&](int n, int k) {
            return bf16_bits_of(rot->pi[(size_t)n * d + k] > 0.0 ? 1.0 : -1.0);
        });
        if ((s = upload(&rot->d_w_umma, w)) != TQ_OK) return s;
    }
    rot->device = dev;
    return TQ_OK;
}

tq_status tq_free_rotation(tq_rotation* rot) {
    tq::bump_handle_generation();
    if (!rot) return TQ_OK;
    if (rot->device >= 0) {
        int cur = -1;
        cudaGetDevice(&cur);
        cudaSetDevice(rot->device);
        cudaFree(rot->d_pi32);
        cudaFree(rot->d_pit32);
        cudaFree(rot->d_pi64);
        cudaFree(rot->d_sign);
        cudaFree(rot->d_pi_frag);
        cudaFree(rot->d_w_umma);
        if (cur >= 0) cudaSetDevice(cur);
    }
    delete rot;
    return TQ_OK;
}

tq_status tq_qjl_to_device(tq_qjl* q) {
    tq::bump_handle_generation();
    if (!q) return fail(TQ_ERR_INVALID_ARG, "tq_qjl_to_device: NULL handle");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(TQ_ERR_CUDA, "tq_qjl_to_device: no CUDA device");
    if (q->device == dev && q->d_st32) return TQ_OK;
    if (q->device >= 0) return fail(TQ_ERR_INVALID_ARG, "tq_qjl_to_device: already on another device");
    const int m = q->m, d = q->d;
    std::vector<float> st((size_t)d * m), s32((size_t)m * d);
    for (int j = 0; j < m; ++j)
        for (int i = 0; i < d; ++i) {
            st[(size_t)i * m + j] = (float)q->s[(size_t)j * d + i];
            s32[(size_t)j * d + i] = (float)q->s[(size_t)j * d + i];
        }
    tq_status s;
    if ((s = upload(&q->d_st32, st)) != TQ_OK) return s;
    if ((s = upload(&q->d_s32, s32)) != TQ_OK) return s;
    if (m == 128 && d == 128) {
        // the append kernel's copy of S: 16-byte unit (u, j) = S[j][8u .. 8u+7] at u * 128 + j
        std::vector<uint16_t> s16((size_t)m * d);
        for (int u = 0; u < d / 8; ++u)
            for (int j = 0; j < m; ++j)
                for (int e = 0; e < 8; ++e)
                    s16[((size_t)u * m + j) * 8 + e] = bf16_bits_of(q->s[(size_t)j * d + 8 * u + e]);
        if ((s = upload(&q->d_s16, s16)) != TQ_OK) return s;
        auto frag = mma_b_fragments([&](int o, int k) { return bf16_bits_of(q->s[(size_t)o * d + k]); });
        if ((s = upload(&q->d_s_frag, frag)) != TQ_OK) return s;
        auto su = umma_operand_128([&](int j, int k) { return bf16_bits_of(q->s[(size_t)j * d + k]); });
        if ((s = upload(&q->d_s_umma, su)) != TQ_OK) return s;
    }
    q->device = dev;
    return TQ_OK;
}

tq_status tq_free_qjl(tq_qjl* q) {
    tq::bump_handle_generation();
    if (!q) return TQ_OK;
    if (q->device >= 0) {
        int cur = -1;
        cudaGetDevice(&cur);
        cudaSetDevice(q->device);
        cudaFree(q->d_st32);
        cudaFree(q->d_s32);
        cudaFree(q->d_s16);
        cudaFree(q->d_s_frag);
        cudaFree(q->d_s_umma);
        if (cur >= 0) cudaSetDevice(cur);
    }
    delete q;
    return TQ_OK;
}

tq_status tq_quantize_kv(const tq_quant_args* a, tq_stream stream) {
    QuantLaunch L;
    bool empty = false;
    tq_status s = quant_prepare(a, &L, &empty);
    if (s != TQ_OK || empty) return s;
    return cuda_status(quant_launch(L, (cudaStream_t)stream), "tq_quantize_kv launch");
}

size_t tq_attn_decode_workspace(const tq_decode_args* a) {
    DecodePlan pl;
    if (plan_decode(a, &pl) != TQ_OK) return 0;
    return pl.total;
}

tq_status tq_attn_decode(const tq_decode_args* a, void* workspace, size_t ws_bytes, tq_stream stream) {
    if (!a) return fail(TQ_ERR_INVALID_ARG, "tq_attn_decode: args are NULL");
    PreparedCall& pc = t_decode_call;
    if (pc.match(a, sizeof(*a), *a, workspace, ws_bytes)) return decode_launch(pc.D, (cudaStream_t)stream, nullptr);
    pc.valid = false;
    DecodeLaunch D;  // prepared from scratch: no field of an earlier call survives
    tq_status s = decode_prepare(a, workspace, ws_bytes, &D);
    if (s != TQ_OK) return s;
    pc.D = D;
    pc.remember();
    return decode_launch(D, (cudaStream_t)stream, nullptr);
}

size_t tq_score_topk_workspace(const tq_topk_args* a) {
    if (!a || a->nq < 0 || a->k < 1 || a->k > 32 || a->d < 3 || a->d > 256 || a->n_db < 0) return 0;
    const int m = a->db.mode == TQ_PROD ? a->db.m : 0;
    const int64_t chunk_rows = 4096;
    const int64_t n_chunks = std::max<int64_t>(1, (a->n_db + chunk_rows - 1) / chunk_rows);
    size_t q = round_up((size_t)a->nq * a->d * 4, 256);
    size_t u = round_up((size_t)a->nq * std::max(m, 1) * 4, 256);
    size_t cs = round_up((size_t)a->nq * n_chunks * a->k * 4, 256);
    return q + u + 2 * cs;
}

tq_status tq_score_topk(const tq_topk_args* a, void* workspace, size_t ws_bytes, tq_stream stream) {
    if (!a) return fail(TQ_ERR_INVALID_ARG, "tq_score_topk: args are NULL");
    if (a->k < 1 || a->k > 32) return fail(TQ_ERR_UNSUPPORTED, "tq_score_topk: k must be 1..32");
    if (a->nq < 0 || a->n_db < 0) return fail(TQ_ERR_INVALID_ARG, "tq_score_topk: negative sizes");
    int cb = 0, cb2 = 0;
    tq_status s = check_cache(a->db, "tq_score_topk db", &cb, &cb2);
    if (s != TQ_OK) return s;
    if (cb2 != cb) return fail(TQ_ERR_UNSUPPORTED, "tq_score_topk: fractional-rate databases are not supported");
    if (a->db.d != a->d) return fail(TQ_ERR_INVALID_ARG, "tq_score_topk: db d does not match");
    if (a->n_db > a->db.rows * a->db.capacity) return fail(TQ_ERR_CAPACITY, "tq_score_topk: n_db exceeds the db planes");
    if (a->n_db > 0x7ffffffe) return fail(TQ_ERR_UNSUPPORTED, "tq_score_topk: n_db must fit int32 ids");
    const bool prod = a->db.mode == TQ_PROD;
    if ((s = check_rot(a->rot, a->d)) != TQ_OK) return s;
    if (prod && (s = check_qjl(a->qjl, a->db.m, a->d)) != TQ_OK) return s;
    if (prod && a->db.m > 32 * vpl_for(a->d)) return fail(TQ_ERR_UNSUPPORTED, "tq_score_topk: m too large for d");
    if (a->nq == 0) return TQ_OK;
    if (!a->queries || !a->ids || !a->scores) return fail(TQ_ERR_INVALID_ARG, "tq_score_topk: NULL buffer");
    if (a->n_db < a->k) return fail(TQ_ERR_INVALID_ARG, "tq_score_topk: n_db < k");
    size_t need = tq_score_topk_workspace(a);
    if (!workspace || ws_bytes < need) return fail(TQ_ERR_WORKSPACE, "tq_score_topk: workspace missing or too small");
    if (!aligned(workspace, 256)) return fail(TQ_ERR_ALIGNMENT, "tq_score_topk: workspace must be 256-byte aligned");
    const int m = prod ? a->db.m : 0;
    const int64_t chunk_rows = 4096;
    const int64_t n_chunks = std::max<int64_t>(1, (a->n_db + chunk_rows - 1) / chunk_rows);
    char* ws = (char*)workspace;
    size_t off_u = round_up((size_t)a->nq * a->d * 4, 256);
    size_t off_cs = off_u + round_up((size_t)a->nq * std::max(m, 1) * 4, 256);
    size_t off_ci = off_cs + round_up((size_t)a->nq * n_chunks * a->k * 4, 256);
    cudaStream_t st = (cudaStream_t)stream;

    tqk::PrepParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.q = a->queries;
    pp.q_dtype = 0;
    pp.rows = a->nq;
    pp.d = a->d;
    pp.m = m;
    pp.pit32 = a->rot->d_pit32;
    pp.sgn = a->rot->d_sign;
    pp.rht = a->rot->kind == TQ_ROT_RHT;
    pp.inv_sqrt_d = (float)(1.0 / std::sqrt((double)a->d));
    pp.st32 = prod ? a->qjl->d_st32 : nullptr;
    pp.qprime = (float*)ws;
    pp.u = prod ? (float*)(ws + off_u) : nullptr;
    cudaError_t e = tqk::launch_query_prep(pp, st);
    if (e != cudaSuccess) return cuda_status(e, "tq_score_topk query prep");

    tqk::TopkParams tp;
    std::memset(&tp, 0, sizeof(tp));
    std::vector<double> c, t;
    if ((s = tq::codebook(a->d, cb, c, t)) != TQ_OK) return s;
    for (size_t i = 0; i < c.size(); ++i) tp.c[i] = (float)c[i];
    tp.qprime = (float*)ws;
    tp.u = pp.u;
    tp.nq = a->nq;
    tp.d = a->d;
    tp.m = m;
    tp.codes = a->db.codes;
    tp.code_stride = tq_code_bytes(a->d, cb);
    tp.signs = a->db.signs;
    tp.sign_stride = prod ? tq_sign_bytes(m) : 0;
    tp.norm = a->db.norm;
    tp.rnorm = a->db.rnorm;
    tp.n_db = a->n_db;
    tp.qjl_scale = prod ? (float)(std::sqrt(M_PI / 2.0) / m) : 0.0f;
    tp.k = a->k;
    tp.n_chunks = (int)n_chunks;
    tp.chunk_rows = chunk_rows;
    tp.cand_score = (float*)(ws + off_cs);
    tp.cand_id = (int32_t*)(ws + off_ci);
    tp.ids = a->ids;
    tp.scores = a->scores;
    // the tcgen05 scan where its shared-memory plan fits (d, m <= 256 padded
    // to a multiple of 16), the SIMT scan otherwise
    const double lam = pick_lambda(a->d, 16 * cb + cb, positive_centroids(c, nullptr));
    pair_table(c, cb, lam, tp.ktab);
    pair_table_lo(c, cb, lam, tp.ktab_lo);
    tp.inv_lam = (float)(1.0 / lam);
    tp.ks = (int)round_up((size_t)std::max(a->d, m), 16);
    if ((e = tqk::device_error_word(&tp.err)) != cudaSuccess) return cuda_status(e, "tq_score_topk error word");
    // the tensor-core scan takes 16x longer chunks: a list restarts once per
    // chunk, so longer chunks mean fewer insertions per row (the expected
    // count per list grows only with the log of its rows); it needs no more
    // candidate slots than the workspace holds
    tqk::TopkParams tu = tp;
    tu.chunk_rows = 16 * chunk_rows;
    tu.n_chunks = (int)std::max<int64_t>(1, (a->n_db + tu.chunk_rows - 1) / tu.chunk_rows);
    e = g_topk_simt ? cudaErrorNotSupported : tqk::launch_topk_umma(tu, cb, prod ? 1 : 0, cb >= 3 ? 1 : 0, st);
    if (e == cudaErrorNotSupported) {
        (void)cudaGetLastError();  // nothing was launched
        e = tqk::launch_topk(tp, cb, prod ? 1 : 0, st);
    }
    return cuda_status(e, "tq_score_topk");
}

int tq_topk_force_simt(int on) {
    tq::bump_handle_generation();
    const int prev = g_topk_simt ? 1 : 0;
    g_topk_simt = on != 0;
    return prev;
}

int tq_prefill_force_mma_sync(int on) {
    tq::bump_handle_generation();
    const int prev = g_prefill_umma ? 0 : 1;
    g_prefill_umma = on == 0;
    return prev;
}

int tq_quantize_force_mma_sync(int on) {
    tq::bump_handle_generation();
    const int prev = g_quant_umma ? 0 : 1;
    g_quant_umma = on == 0;
    return prev;
}

size_t tq_decode_step_workspace(const tq_step_args* a) { return a ? tq_attn_decode_workspace(&a->attn) : 0; }

tq_status tq_decode_step(const tq_step_args* a, void* workspace, size_t ws_bytes, tq_stream stream) {
    if (!a) return fail(TQ_ERR_INVALID_ARG, "tq_decode_step: args are NULL");
    PreparedCall& pc = t_step_call;
    if (pc.match(a, sizeof(*a), a->attn, workspace, ws_bytes)) {
        tqk::StepPrepParams sp = pc.sp;
        return decode_launch(pc.D, (cudaStream_t)stream, &sp);
    }
    pc.valid = false;
    const tq_decode_args& at = a->attn;
    if (at.k.mode == TQ_POLAR)
        return fail(TQ_ERR_UNSUPPORTED, "tq_decode_step: PolarQuant keys are appended with tq_quantize_kv, then tq_attn_decode");
    if (!a->k_new || !a->v_new || !a->append_pos) return fail(TQ_ERR_INVALID_ARG, "tq_decode_step: k_new/v_new/append_pos is NULL");
    tq_quant_args qk;
    std::memset(&qk, 0, sizeof(qk));
    qk.cache = at.k;
    qk.rot = at.rot;
    qk.qjl = at.qjl;
    qk.x = a->k_new;
    qk.x_dtype = a->new_dtype;
    qk.x_stride = at.d;
    qk.n = (int64_t)at.batch * at.hkv;
    qk.append_pos = a->append_pos;
    qk.heads = at.hkv;
    tq_quant_args qv = qk;
    qv.cache = at.v;
    qv.qjl = nullptr;
    qv.x = a->v_new;
    // everything is validated before anything is enqueued
    QuantLaunch LK, LV;
    bool ek = false, ev = false;
    tq_status s;
    if ((s = quant_prepare(&qk, &LK, &ek)) != TQ_OK) return s;
    if ((s = quant_prepare(&qv, &LV, &ev)) != TQ_OK) return s;
    DecodeLaunch D;
    if ((s = decode_prepare(&at, workspace, ws_bytes, &D)) != TQ_OK) return s;
    // the appends ride in the query prep's launch (one CTA per vector, the
    // kernel tq_quantize_kv uses for up to kSmallAppend vectors)
    tqk::StepPrepParams sp;
    std::memset(&sp, 0, sizeof(sp));
    if (!ek) step_append(LK, &sp);
    if (!ev) step_append(LV, &sp);
    D.dp.append_pos = a->append_pos;
    pc.D = D;
    pc.sp = sp;
    pc.remember();
    return decode_launch(D, (cudaStream_t)stream, &sp);
}

}  // extern "C"

namespace {

struct PrefillPlan {
    int group = 0, n_splits = 0, split_tokens = 0, lim_cap = 0;
    bool umma = false;  // the tcgen05 kernel (128 rows x 128-token tiles per CTA)
    int qbs = 0, unit_tiles = 0, tiles_per_cta = 0;  // its stream-K plan
    size_t off_u = 0, off_part = 0, total = 0;
};

// key / value code bits of a prefill's caches as the kernels see them, or -1
// where the caches are not a PROD / MSE pair (the checks come later)
void prefill_bits(const tq_prefill_args* a, int* kb, int* vb, bool* two) {
    *kb = a->k.mode == TQ_PROD ? a->k.bits - 1 : -1;
    *vb = a->v.mode == TQ_MSE ? a->v.bits : -1;
    *two = a->k.bits2 != 0 && a->k.bits2 != a->k.bits;
}

tq_status plan_prefill(const tq_prefill_args* a, PrefillPlan* pl) {
    if (!a) return fail(TQ_ERR_INVALID_ARG, "tq_attn_prefill: args are NULL");
    if (a->batch < 1 || a->chunk < 0 || a->hq < 1 || a->hkv < 1)
        return fail(TQ_ERR_INVALID_ARG, "tq_attn_prefill: batch/hq/hkv must be >= 1 and chunk >= 0");
    if (a->d != 128) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: d must be 128");
    if (a->hq % a->hkv) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: hq must be a multiple of hkv");
    const int g = a->hq / a->hkv;
    if (g != 1 && g != 2 && g != 4 && g != 8) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: hq / hkv must be 1, 2, 4 or 8");
    if (a->max_context < 0) return fail(TQ_ERR_INVALID_ARG, "tq_attn_prefill: max_context < 0");
    if (a->max_context > a->k.capacity) return fail(TQ_ERR_CAPACITY, "tq_attn_prefill: max_context exceeds the capacity");
    if (a->hq > 256) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: hq must be <= 256");
    const int64_t rows = (int64_t)a->batch * a->chunk * a->hq;
    if (rows > (1ll << 31) / 128) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: too many query rows");
    int kb = 0, vb = 0;
    bool two = false;
    prefill_bits(a, &kb, &vb, &two);
    pl->umma = g_prefill_umma && tqk::prefill_umma_supported(kb, vb, two);
    const int rows_per_cta = pl->umma ? tqk::kPuRows : tqk::kPfRows;
    const int tile = pl->umma ? tqk::kPuTok : 64;  // split granularity in tokens
    const int64_t qbs = ((int64_t)a->chunk * g + rows_per_cta - 1) / rows_per_cta;
    if (qbs > 0x7fffffff || (int64_t)a->batch * a->hkv > 65535)
        return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: grid too large");
    pl->group = g;
    pl->lim_cap = a->max_context;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int ctx = std::max(a->max_context, 1);
    const long long base = std::max<long long>(1, qbs * a->batch * a->hkv);
    if (pl->umma) {
        // Stream-K over the (unit, tile) sequence: unit u = (batch row, KV
        // head, query block) owns ntile 128-token tiles; one CTA per SM takes
        // an equal share of the whole sequence, crossing unit boundaries, so
        // no SM idles when the units do not fill whole waves. An explicit
        // split count instead pads each unit to n equal splits, one per CTA.
        const long long ntile = (ctx + tile - 1) / tile;
        long long nt_unit = ntile, tpc;
        if (a->n_splits > 0) {
            const long long per = (ntile + a->n_splits - 1) / a->n_splits;
            nt_unit = per * ((ntile + per - 1) / per);
            tpc = per;
        } else {
            const long long c = std::min<long long>(sms, base * ntile);
            tpc = (base * ntile + c - 1) / c;
            // at most kPuMaxSeg - 1 segments per CTA
            tpc = std::max(1LL, std::min(tpc, (long long)(tqk::kPuMaxSeg - 2) * ntile));
        }
        const long long ctas = (base * nt_unit + tpc - 1) / tpc;
        if (ctas > 0x7fffffff || nt_unit > 0x7fffffff) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: grid too large");
        // slots per row: the most CTAs one unit spans
        long long slots = 1;
        for (long long u = 0; u < base; ++u)
            slots = std::max(slots, ((u + 1) * nt_unit - 1) / tpc - (u * nt_unit) / tpc + 1);
        if (slots > 65535) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: too many splits");
        pl->qbs = (int)qbs;
        pl->unit_tiles = (int)nt_unit;
        pl->tiles_per_cta = (int)tpc;
        pl->n_splits = (int)slots;
        pl->split_tokens = (int)std::min<long long>(tpc * tile, 0x7fffffff);
    } else {
        long long want = a->n_splits;
        if (want <= 0) want = ((long long)sms * 4 + base - 1) / base;  // about four CTAs per SM (two resident)
        if (want > 65535) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: too many splits");
        int st = (int)((ctx + want - 1) / want);
        st = std::max(tile, (st + tile - 1) / tile * tile);
        pl->split_tokens = st;
        pl->n_splits = (ctx + st - 1) / st;
    }
    const size_t r = (size_t)rows;
    pl->off_u = round_up(r * 128 * sizeof(float), 256);
    pl->off_part = pl->off_u + round_up(r * 128 * sizeof(float), 256);
    pl->total = std::max<size_t>(256, pl->off_part + round_up(r * (size_t)pl->n_splits * (128 + tqk::kPartPad) * sizeof(float), 256));
    return TQ_OK;
}

}  // namespace

extern "C" {

size_t tq_attn_prefill_workspace(const tq_prefill_args* a) {
    PrefillPlan pl;
    if (plan_prefill(a, &pl) != TQ_OK) return 0;
    return pl.total;
}

tq_status tq_attn_prefill(const tq_prefill_args* a, void* workspace, size_t ws_bytes, tq_stream stream) {
    PrefillPlan pl;
    tq_status s = plan_prefill(a, &pl);
    if (s != TQ_OK) return s;
    int kb = 0, vb = 0, kb2 = 0, vb2 = 0;
    if ((s = check_cache(a->k, "tq_attn_prefill k", &kb, &kb2)) != TQ_OK) return s;
    if ((s = check_cache(a->v, "tq_attn_prefill v", &vb, &vb2)) != TQ_OK) return s;
    const bool two = kb2 != kb;
    if ((vb2 != vb) != two)
        return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: keys and values must both be fractional-rate caches, or neither");
    if (a->k.mode != TQ_PROD || a->v.mode != TQ_MSE) return fail(TQ_ERR_INVALID_ARG, "tq_attn_prefill: keys must be PROD and values MSE");
    if (a->k.d != a->d || a->v.d != a->d) return fail(TQ_ERR_INVALID_ARG, "tq_attn_prefill: cache d does not match");
    if (a->k.m != 128) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: m must be 128");
    const int64_t kvrows = (int64_t)a->batch * a->hkv;
    if (a->k.rows != kvrows || a->v.rows != kvrows) return fail(TQ_ERR_INVALID_ARG, "tq_attn_prefill: cache rows must be batch*hkv");
    if (a->k.capacity != a->v.capacity) return fail(TQ_ERR_INVALID_ARG, "tq_attn_prefill: k and v capacity differ");
    if (a->k.capacity % 16) return fail(TQ_ERR_ALIGNMENT, "tq_attn_prefill: cache capacity must be a multiple of 16");
    if (!aligned(a->k.norm, 16) || !aligned(a->k.rnorm, 16) || !aligned(a->v.norm, 16) || !aligned(a->v.codes, 16))
        return fail(TQ_ERR_ALIGNMENT, "tq_attn_prefill: every cache plane must be 16-byte aligned (bulk copies)");
    if ((s = check_rot(a->rot, a->d)) != TQ_OK) return s;
    if ((s = check_qjl(a->qjl, a->k.m, a->d)) != TQ_OK) return s;
    if (a->chunk == 0) return TQ_OK;
    if (!a->q || !a->out || !a->q_start) return fail(TQ_ERR_INVALID_ARG, "tq_attn_prefill: q/out/q_start is NULL");
    if (a->q_dtype != TQ_F32 && a->q_dtype != TQ_BF16) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: q_dtype must be F32 or BF16");
    if (a->out_dtype != TQ_F32 && a->out_dtype != TQ_BF16) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: out_dtype must be F32 or BF16");
    if (!aligned(a->out, 16)) return fail(TQ_ERR_ALIGNMENT, "tq_attn_prefill: out must be 16-byte aligned (vector stores)");
    if (!workspace || ws_bytes < pl.total) return fail(TQ_ERR_WORKSPACE, "tq_attn_prefill: workspace missing or too small");
    if (!aligned(workspace, 256)) return fail(TQ_ERR_ALIGNMENT, "tq_attn_prefill: workspace must be 256-byte aligned");

    char* ws = (char*)workspace;
    const int64_t rows = (int64_t)a->batch * a->chunk * a->hq;
    tqk::PrepParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.q = a->q;
    pp.q_dtype = a->q_dtype == TQ_BF16 ? 1 : 0;
    pp.rows = rows;
    pp.d = a->d;
    pp.m = a->k.m;
    pp.pit32 = a->rot->d_pit32;
    pp.sgn = a->rot->d_sign;
    pp.rht = a->rot->kind == TQ_ROT_RHT;
    pp.inv_sqrt_d = (float)(1.0 / std::sqrt((double)a->d));
    pp.st32 = a->qjl->d_st32;
    pp.s16 = a->qjl->d_s16;
    pp.qprime = (float*)ws;
    pp.u = (float*)(ws + pl.off_u);

    tqk::PrefillParams fp;
    std::memset(&fp, 0, sizeof(fp));
    fp.qprime = pp.qprime;
    fp.u = pp.u;
    fp.batch = a->batch;
    fp.chunk = a->chunk;
    fp.hq = a->hq;
    fp.hkv = a->hkv;
    fp.group = pl.group;
    fp.q_start = a->q_start;
    if (a->gqa_map) {
        std::vector<int> count(a->hkv, 0);
        for (int h = 0; h < a->hq; ++h) {
            const int g = a->gqa_map[h];
            if (g < 0 || g >= a->hkv) return fail(TQ_ERR_INVALID_ARG, "tq_attn_prefill: gqa_map entry out of range");
            if (count[g] >= pl.group) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_prefill: every KV head must serve hq/hkv query heads");
            fp.head_table[g * pl.group + count[g]++] = (int16_t)h;
        }
        fp.use_table = 1;
    }
    fp.lim_cap = pl.lim_cap;
    fp.capacity = a->k.capacity;
    fp.kcodes = a->k.codes;
    fp.ksigns = a->k.signs;
    fp.knorm = a->k.norm;
    fp.krnorm = a->k.rnorm;
    fp.vcodes = a->v.codes;
    fp.vnorm = a->v.norm;
    if ((s = scan_tables(a->d, kb, kb2, vb, vb2, &fp)) != TQ_OK) return s;
    fp.qjl_scale = (float)(std::sqrt(M_PI / 2.0) / a->k.m);
    const double scale = a->scale != 0.0f ? (double)a->scale : 1.0 / std::sqrt((double)a->d);
    fp.scale_log2 = (float)(scale * 1.4426950408889634);
    fp.n_splits = pl.n_splits;
    fp.split_tokens = pl.split_tokens;
    fp.partial = (float*)(ws + pl.off_part);
    fp.qbs = pl.qbs;
    fp.unit_tiles = pl.unit_tiles;
    fp.tiles_per_cta = pl.tiles_per_cta;
    cudaError_t e = tqk::device_error_word(&fp.err);
    if (e != cudaSuccess) return cuda_status(e, "tq_attn_prefill error word");

    tqk::CombineParams cp;
    std::memset(&cp, 0, sizeof(cp));
    cp.partial = fp.partial;
    cp.rows = (int)rows;
    cp.d = a->d;
    cp.n_splits = pl.n_splits;
    cp.pi32 = a->rot->d_pi32;
    cp.sgn = a->rot->d_sign;
    cp.rht = a->rot->kind == TQ_ROT_RHT;
    cp.inv_sqrt_d = (float)(1.0 / std::sqrt((double)a->d));
    cp.out = a->out;
    cp.out_dtype = a->out_dtype == TQ_BF16 ? 1 : 0;

    cudaStream_t st = (cudaStream_t)stream;
    if ((e = tqk::launch_rows_prep(pp, st)) != cudaSuccess) return cuda_status(e, "tq_attn_prefill query prep");
    if (a->scan_begin && (e = cudaEventRecord((cudaEvent_t)a->scan_begin, st)) != cudaSuccess)
        return cuda_status(e, "tq_attn_prefill scan_begin");
    e = pl.umma ? tqk::launch_prefill_umma(fp, kb, vb, two, st) : tqk::launch_prefill_mma(fp, kb, vb, two, st);
    if (e != cudaSuccess) return cuda_status(e, "tq_attn_prefill scan");
    if (a->scan_end && (e = cudaEventRecord((cudaEvent_t)a->scan_end, st)) != cudaSuccess)
        return cuda_status(e, "tq_attn_prefill scan_end");
    return cuda_status(tqk::launch_merge_rows(cp, st), "tq_attn_prefill merge");
}

tq_status tq_device_errors(uint32_t* flags_out, int reset) {
    uint32_t* word = nullptr;
    cudaError_t e = tqk::device_error_word(&word);
    if (e != cudaSuccess) return cuda_status(e, "tq_device_errors");
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_status(e, "tq_device_errors");
    uint32_t v = 0;
    if ((e = cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_status(e, "tq_device_errors read");
    if (reset && (e = cudaMemset(word, 0, sizeof(v))) != cudaSuccess) return cuda_status(e, "tq_device_errors reset");
    if (reset && (e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_status(e, "tq_device_errors reset");
    if (flags_out) *flags_out = v;
    return v ? fail(TQ_ERR_TIMEOUT, "tq_device_errors: a device-side wait ran out (flags " + std::to_string(v) + ")")
             : TQ_OK;
}

namespace {
tq_status umma_selftest(const void* a, const void* b, float* d, int n, int k, int a_tmem, tq_stream stream) {
    if (!a || !b || !d) return fail(TQ_ERR_INVALID_ARG, "tq_selftest_umma_gemm: NULL operand");
    if ((n != 16 && n != 32 && n != 64 && n != 128) || k < 16 || k > 128 || k % 16)
        return fail(TQ_ERR_UNSUPPORTED, "tq_selftest_umma_gemm: n must be 16/32/64/128 and k a multiple of 16 up to 128");
    if (!aligned(a, 4) || !aligned(b, 4) || !aligned(d, 4)) return fail(TQ_ERR_ALIGNMENT, "tq_selftest_umma_gemm: misaligned");
    uint32_t* word = nullptr;
    cudaError_t e = tqk::device_error_word(&word);
    if (e != cudaSuccess) return cuda_status(e, "tq_selftest_umma_gemm");
    e = tqk::launch_umma_selftest(a, b, d, n, k, a_tmem, word, (cudaStream_t)stream);
    return cuda_status(e, "tq_selftest_umma_gemm");
}
}  // namespace

tq_status tq_selftest_umma_gemm(const void* a, const void* b, float* d, int n, int k, tq_stream stream) {
    return umma_selftest(a, b, d, n, k, 0, stream);
}

tq_status tq_selftest_umma_gemm_tmem_a(const void* a, const void* b, float* d, int n, int k, tq_stream stream) {
    return umma_selftest(a, b, d, n, k, 1, stream);
}

tq_status tq_selftest_bounded_wait(uint32_t limit_us, tq_stream stream) {
    if (limit_us < 1 || limit_us > 1000000) return fail(TQ_ERR_INVALID_ARG, "tq_selftest_bounded_wait: limit_us must be 1..1000000");
    uint32_t* word = nullptr;
    cudaError_t e = tqk::device_error_word(&word);
    if (e != cudaSuccess) return cuda_status(e, "tq_selftest_bounded_wait");
    e = tqk::launch_wait_selftest(word, (uint64_t)limit_us * 1000ull, (cudaStream_t)stream);
    return cuda_status(e, "tq_selftest_bounded_wait");
}

}  // extern "C"
