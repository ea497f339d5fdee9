// Host set-up math of libtq: the random stream, the Haar rotation from a
// Householder QR, the bfloat16 rounding of the QJL projection and the
// Lloyd-Max codebook of the post-rotation Beta law. Plain C++17, fp64.
//
// Sources: the rotation is "the QR factorisation of a Gaussian matrix", a
// data-independent transform generated once (A2A TurboQuant explainer,
// "Stage 1: random rotation"); after it each coordinate follows
// Beta((d-1)/2,(d-1)/2) on [-1,1] and a Lloyd-Max quantizer precomputed for
// that law is applied per coordinate (A2A "Stage 1"; Qiita TurboQuant
// article, "Rotate, then quantize").

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "tq_internal.h"

namespace tq {

static thread_local std::string g_last_error;

tq_status fail(tq_status s, const std::string& msg) {
    g_last_error = msg;
    return s;
}

void clear_error() { g_last_error.clear(); }

namespace {
std::atomic<uint64_t> g_generation{0};
}
uint64_t handle_generation() { return g_generation.load(std::memory_order_acquire); }
void bump_handle_generation() { g_generation.fetch_add(1, std::memory_order_acq_rel); }

// ---------------------------------------------------------------------------
// SplitMix64 (Steele, Lea & Flood 2014), counter form: the k-th draw of a
// stream is the finaliser applied to seed + (k+1) * golden_gamma.
// ---------------------------------------------------------------------------
uint64_t splitmix64_at(uint64_t seed, uint64_t k) {
    uint64_t z = seed + (k + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

// Box-Muller: pair p takes draws 2p (radius) and 2p+1 (angle); the first
// uniform is shifted to (0, 1] so the logarithm is finite.
void gaussians(uint64_t seed, int64_t count, double* out) {
    const double two_pi = 2.0 * M_PI;
    for (int64_t p = 0; 2 * p < count; ++p) {
        uint64_t a = splitmix64_at(seed, 2 * (uint64_t)p);
        uint64_t b = splitmix64_at(seed, 2 * (uint64_t)p + 1);
        double u1 = ((double)(a >> 11) + 1.0) * 0x1.0p-53;
        double u2 = (double)(b >> 11) * 0x1.0p-53;
        double rad = std::sqrt(-2.0 * std::log(u1));
        double ang = two_pi * u2;
        out[2 * p] = rad * std::cos(ang);
        if (2 * p + 1 < count) out[2 * p + 1] = rad * std::sin(ang);
    }
}

// Nearest bfloat16 (8 significant bits), ties to even, straight from fp64.
double round_bf16(double x) {
    if (x == 0.0 || !std::isfinite(x)) return x;
    int e = 0;
    double m = std::frexp(x, &e);  // x = m 2^e, 0.5 <= |m| < 1
    return std::ldexp(std::nearbyint(m * 256.0), e - 8);
}

// ---------------------------------------------------------------------------
// Haar rotation: G = QR by Householder reflections, Pi = Q diag(sign diag R).
// ---------------------------------------------------------------------------
void householder_haar(const double* g, int d, double* pi_out) {
    std::vector<double> a(g, g + (size_t)d * d);  // row-major, reduced in place
    std::vector<double> v((size_t)d * d, 0.0);    // reflector k in row k of v
    std::vector<double> vn2(d, 0.0), rdiag(d, 0.0);
    for (int k = 0; k < d; ++k) {
        double nrm = 0.0;
        for (int i = k; i < d; ++i) nrm += a[(size_t)i * d + k] * a[(size_t)i * d + k];
        nrm = std::sqrt(nrm);
        double x0 = a[(size_t)k * d + k];
        double alpha = x0 >= 0.0 ? -nrm : nrm;
        double* vk = &v[(size_t)k * d];
        vk[k] = x0 - alpha;
        for (int i = k + 1; i < d; ++i) vk[i] = a[(size_t)i * d + k];
        double s2 = 0.0;
        for (int i = k; i < d; ++i) s2 += vk[i] * vk[i];
        vn2[k] = s2;
        if (s2 > 0.0) {
            for (int j = k; j < d; ++j) {
                double s = 0.0;
                for (int i = k; i < d; ++i) s += vk[i] * a[(size_t)i * d + j];
                double f = 2.0 * s / s2;
                for (int i = k; i < d; ++i) a[(size_t)i * d + j] -= f * vk[i];
            }
        }
        rdiag[k] = a[(size_t)k * d + k];
    }
    // Q = H_0 H_1 ... H_{d-1} I, applied right to left.
    std::vector<double> q((size_t)d * d, 0.0);
    for (int i = 0; i < d; ++i) q[(size_t)i * d + i] = 1.0;
    for (int k = d - 1; k >= 0; --k) {
        if (vn2[k] <= 0.0) continue;
        const double* vk = &v[(size_t)k * d];
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int i = k; i < d; ++i) s += vk[i] * q[(size_t)i * d + j];
            double f = 2.0 * s / vn2[k];
            for (int i = k; i < d; ++i) q[(size_t)i * d + j] -= f * vk[i];
        }
    }
    for (int i = 0; i < d; ++i)
        for (int k = 0; k < d; ++k) {
            double sg = rdiag[k] < 0.0 ? -1.0 : 1.0;
            pi_out[(size_t)i * d + k] = q[(size_t)i * d + k] * sg;
        }
}

// ---------------------------------------------------------------------------
// Lloyd-Max codebook of f(t) ~ (1 - t^2)^(alpha - 1) on [-1, 1], alpha = (d-1)/2.
// Cell masses by composite 16-point Gauss-Legendre quadrature (nodes found by
// Newton's method on the Legendre polynomial); first moments in closed form,
//   int_a^b t (1-t^2)^(alpha-1) dt = ((1-a^2)^alpha - (1-b^2)^alpha) / (2 alpha).
// ---------------------------------------------------------------------------
namespace {

struct GaussLegendre16 {
    double x[16], w[16];
    GaussLegendre16() {
        const int n = 16;
        for (int i = 0; i < n; ++i) {
            double z = std::cos(M_PI * (i + 0.75) / (n + 0.5));
            for (int it = 0; it < 100; ++it) {
                double p0 = 1.0, p1 = z;  // P_0, P_1
                for (int k = 2; k <= n; ++k) {
                    double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
                    p0 = p1;
                    p1 = p2;
                }
                double dp = n * (z * p1 - p0) / (z * z - 1.0);
                double dz = p1 / dp;
                z -= dz;
                if (std::fabs(dz) < 1e-17) break;
            }
            double p0 = 1.0, p1 = z;
            for (int k = 2; k <= n; ++k) {
                double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
                p0 = p1;
                p1 = p2;
            }
            double dp = n * (z * p1 - p0) / (z * z - 1.0);
            x[i] = z;
            w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
        }
    }
};

const GaussLegendre16& gl16() {
    static const GaussLegendre16 g;
    return g;
}

struct BetaLaw {
    int d;
    double alpha, km1, z, h;
    explicit BetaLaw(int d_) : d(d_) {
        alpha = 0.5 * (d - 1);
        km1 = alpha - 1.0;
        h = std::min(1.0 / 64.0, 0.25 / std::sqrt((double)d));
        z = raw(-1.0, 1.0);
    }
    double dens(double t) const {  // unnormalised (1 - t^2)^(alpha-1)
        double s = 1.0 - t * t;
        if (s <= 0.0) return 0.0;
        return std::exp(km1 * std::log1p(-t * t));
    }
    double raw(double a, double b) const {  // int_a^b (1-t^2)^(alpha-1) dt
        if (b <= a) return 0.0;
        int panels = (int)std::ceil((b - a) / h);
        if (panels < 1) panels = 1;
        double w = (b - a) / panels, tot = 0.0;
        const GaussLegendre16& g = gl16();
        for (int p = 0; p < panels; ++p) {
            double lo = a + p * w, mid = lo + 0.5 * w, acc = 0.0;
            for (int i = 0; i < 16; ++i) acc += g.w[i] * dens(mid + 0.5 * w * g.x[i]);
            tot += 0.5 * w * acc;
        }
        return tot;
    }
    double mass(double a, double b) const { return raw(a, b) / z; }
    double moment(double a, double b) const {
        double ua = std::exp(alpha * std::log1p(-a * a));
        double ub = std::exp(alpha * std::log1p(-b * b));
        if (a <= -1.0) ua = 0.0;
        if (b >= 1.0) ub = 0.0;
        return (ua - ub) / (2.0 * alpha * z);
    }
    double quantile(double p) const {  // by bisection on the CDF
        double lo = -1.0, hi = 1.0;
        for (int it = 0; it < 80; ++it) {
            double mid = 0.5 * (lo + hi);
            double f = mid >= 0.0 ? 0.5 + mass(0.0, mid) : 0.5 - mass(mid, 0.0);
            if (f < p) lo = mid; else hi = mid;
        }
        return 0.5 * (lo + hi);
    }
};

void symmetrize(std::vector<double>& c) {
    size_t L = c.size();
    std::vector<double> s(L);
    for (size_t i = 0; i < L; ++i) s[i] = 0.5 * (c[i] - c[L - 1 - i]);
    c.swap(s);
}

std::mutex g_cb_mutex;
std::map<std::pair<int, int>, std::pair<std::vector<double>, std::vector<double>>> g_cb_cache;

}  // namespace

tq_status codebook(int d, int bits, std::vector<double>& c_out, std::vector<double>& t_out) {
    if (d < 3 || d > 4096) return fail(TQ_ERR_INVALID_ARG, "codebook: d must be in 3..4096");
    if (bits < 1 || bits > 4) return fail(TQ_ERR_INVALID_ARG, "codebook: bits must be in 1..4");
    {
        std::lock_guard<std::mutex> lk(g_cb_mutex);
        auto it = g_cb_cache.find({d, bits});
        if (it != g_cb_cache.end()) {
            c_out = it->second.first;
            t_out = it->second.second;
            return TQ_OK;
        }
    }
    const int L = 1 << bits;
    BetaLaw law(d);
    std::vector<double> c(L), t(L - 1), edges(L + 1), nc(L);
    for (int i = 0; i < L; ++i) c[i] = law.quantile((i + 0.5) / L);
    symmetrize(c);
    const double tol = 64.0 * 2.220446049250313e-16;
    double best = 1e300;
    int since_best = 0;
    bool done = false;
    for (int it = 0; it < 200000 && !done; ++it) {
        for (int j = 0; j < L - 1; ++j) t[j] = 0.5 * (c[j] + c[j + 1]);
        t[L / 2 - 1] = 0.0;
        edges[0] = -1.0;
        for (int j = 0; j < L - 1; ++j) edges[j + 1] = t[j];
        edges[L] = 1.0;
        for (int i = 0; i < L; ++i) nc[i] = law.moment(edges[i], edges[i + 1]) / law.mass(edges[i], edges[i + 1]);
        symmetrize(nc);
        double delta = 0.0, cmax = 0.0;
        for (int i = 0; i < L; ++i) {
            delta = std::max(delta, std::fabs(nc[i] - c[i]));
            cmax = std::max(cmax, std::fabs(nc[i]));
        }
        c = nc;
        delta /= cmax;
        if (delta <= tol) done = true;
        if (delta < best) {
            best = delta;
            since_best = 0;
        } else if (++since_best >= 200 && best < 1e-9) {
            done = true;
        }
    }
    if (!done) return fail(TQ_ERR_INVALID_ARG, "codebook: Lloyd-Max did not converge");
    for (int j = 0; j < L - 1; ++j) t[j] = 0.5 * (c[j] + c[j + 1]);
    t[L / 2 - 1] = 0.0;
    {
        std::lock_guard<std::mutex> lk(g_cb_mutex);
        g_cb_cache[{d, bits}] = {c, t};
    }
    c_out = c;
    t_out = t;
    return TQ_OK;
}

// ---------------------------------------------------------------------------
// PolarQuant angle codebooks. After a Haar rotation the level-1 angle of a
// coordinate pair is uniform on (-pi, pi]; the level-l angle (l >= 2) pairs
// the norms of two independent 2^(l-1)-dimensional Gaussian blocks, so its
// density on [0, pi/2] is proportional to (sin psi cos psi)^(k-1), k =
// 2^(l-1). Level 1: equal cells from -pi (the Lloyd-Max optimum of a
// uniform law). Higher levels: the Lloyd-Max fixed point, cell masses and
// first moments by composite 16-point Gauss-Legendre quadrature of the
// unnormalised density (the normalisation cancels in each centroid), the
// centroids kept symmetric about pi/4.
// ---------------------------------------------------------------------------
namespace {

struct AngleLaw {
    double km1, h;
    explicit AngleLaw(int level) {
        const double k = std::ldexp(1.0, level - 1);
        km1 = k - 1.0;
        // panels well inside the width of the peak at pi/4 (about 1/sqrt(2k))
        h = std::min(M_PI / 256.0, 0.05 / std::sqrt(k));
    }
    double dens(double u) const {  // (sin u cos u)^(k-1) = (sin 2u / 2)^(k-1)
        const double s = 0.5 * std::sin(2.0 * u);
        return s <= 0.0 ? 0.0 : std::exp(km1 * std::log(s));
    }
    // (mass, first moment) of [a, b]
    std::pair<double, double> cell(double a, double b) const {
        if (b <= a) return {0.0, 0.0};
        int panels = std::max(1, (int)std::ceil((b - a) / h));
        const double w = (b - a) / panels;
        const GaussLegendre16& g = gl16();
        double m0 = 0.0, m1 = 0.0;
        for (int p = 0; p < panels; ++p) {
            const double mid = a + (p + 0.5) * w;
            double s0 = 0.0, s1 = 0.0;
            for (int i = 0; i < 16; ++i) {
                const double u = mid + 0.5 * w * g.x[i];
                const double f = g.w[i] * dens(u);
                s0 += f;
                s1 += f * u;
            }
            m0 += 0.5 * w * s0;
            m1 += 0.5 * w * s1;
        }
        return {m0, m1};
    }
};

std::mutex g_pcb_mutex;
std::map<std::pair<int, int>, std::pair<std::vector<double>, std::vector<double>>> g_pcb_cache;

}  // namespace

tq_status polar_codebook(int level, int bits, std::vector<double>& c_out, std::vector<double>& t_out) {
    if (level < 1 || level > 8) return fail(TQ_ERR_INVALID_ARG, "polar codebook: level must be 1..8");
    if (bits < 1 || bits > 4) return fail(TQ_ERR_INVALID_ARG, "polar codebook: bits must be 1..4");
    {
        std::lock_guard<std::mutex> lk(g_pcb_mutex);
        auto it = g_pcb_cache.find({level, bits});
        if (it != g_pcb_cache.end()) {
            c_out = it->second.first;
            t_out = it->second.second;
            return TQ_OK;
        }
    }
    const int L = 1 << bits;
    std::vector<double> c(L), t(L - 1);
    if (level == 1) {
        const double w = (M_PI - (-M_PI)) / L;
        for (int j = 1; j < L; ++j) t[j - 1] = -M_PI + w * j;
        for (int i = 0; i < L; ++i) c[i] = -M_PI + w * (i + 0.5);
    } else {
        const AngleLaw law(level);
        // start: equal-mass cells of the law (CDF by quadrature and bisection)
        const double total = law.cell(0.0, 0.5 * M_PI).first;
        for (int i = 0; i < L; ++i) {
            const double target = (i + 0.5) / L * total;
            double lo = 0.0, hi = 0.5 * M_PI;
            for (int it = 0; it < 80; ++it) {
                const double mid = 0.5 * (lo + hi);
                if (law.cell(0.0, mid).first < target) lo = mid; else hi = mid;
            }
            c[i] = 0.5 * (lo + hi);
        }
        std::vector<double> nc(L);
        bool done = false;
        for (int it = 0; it < 100000 && !done; ++it) {
            double prev = 0.0;
            for (int i = 0; i < L; ++i) {
                const double next = i + 1 < L ? 0.5 * (c[i] + c[i + 1]) : 0.5 * M_PI;
                const auto mm = law.cell(prev, next);
                nc[i] = mm.first > 0.0 ? mm.second / mm.first : 0.5 * (prev + next);
                prev = next;
            }
            double delta = 0.0;
            for (int i = 0; i < L; ++i) {
                const double sym = 0.5 * (nc[i] + (0.5 * M_PI - nc[L - 1 - i]));
                delta = std::max(delta, std::fabs(sym - c[i]));
                c[i] = sym;
            }
            done = delta < 1e-15;
        }
        if (!done) return fail(TQ_ERR_INVALID_ARG, "polar codebook: Lloyd-Max did not converge");
        for (int j = 0; j < L - 1; ++j) t[j] = 0.5 * (c[j] + c[j + 1]);
    }
    {
        std::lock_guard<std::mutex> lk(g_pcb_mutex);
        g_pcb_cache[{level, bits}] = {c, t};
    }
    c_out = c;
    t_out = t;
    return TQ_OK;
}

}  // namespace tq

// ---------------------------------------------------------------------------
// Host-only C entry points (set-up).
// ---------------------------------------------------------------------------
extern "C" {

const char* tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "TQ_OK";
        case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG";
        case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED";
        case TQ_ERR_ALIGNMENT: return "TQ_ERR_ALIGNMENT";
        case TQ_ERR_CAPACITY: return "TQ_ERR_CAPACITY";
        case TQ_ERR_CUDA: return "TQ_ERR_CUDA";
        case TQ_ERR_TIMEOUT: return "TQ_ERR_TIMEOUT";
        case TQ_ERR_WORKSPACE: return "TQ_ERR_WORKSPACE";
        case TQ_ERR_NO_DEVICE_COPY: return "TQ_ERR_NO_DEVICE_COPY";
    }
    return "unknown tq_status";
}

const char* tq_last_error(void) { return tq::g_last_error.c_str(); }

size_t tq_abi_struct_size(const char* name) {
    if (!name) return 0;
    if (!std::strcmp(name, "tq_cache")) return sizeof(tq_cache);
    if (!std::strcmp(name, "tq_quant_args")) return sizeof(tq_quant_args);
    if (!std::strcmp(name, "tq_decode_args")) return sizeof(tq_decode_args);
    if (!std::strcmp(name, "tq_topk_args")) return sizeof(tq_topk_args);
    if (!std::strcmp(name, "tq_step_args")) return sizeof(tq_step_args);
    if (!std::strcmp(name, "tq_prefill_args")) return sizeof(tq_prefill_args);
    return 0;
}

tq_status tq_random_stream(uint64_t seed, uint64_t start, int64_t count, uint64_t* host_out) {
    if (count < 0 || (count > 0 && !host_out)) return tq::fail(TQ_ERR_INVALID_ARG, "tq_random_stream: bad count/out");
    for (int64_t k = 0; k < count; ++k) host_out[k] = tq::splitmix64_at(seed, start + (uint64_t)k);
    return TQ_OK;
}

tq_status tq_make_rotation(uint64_t seed, int d, int kind, tq_rotation** out) {
    if (!out) return tq::fail(TQ_ERR_INVALID_ARG, "tq_make_rotation: out is NULL");
    *out = nullptr;
    if (kind != TQ_ROT_DENSE_QR && kind != TQ_ROT_RHT)
        return tq::fail(TQ_ERR_INVALID_ARG, "tq_make_rotation: unknown kind");
    if (d < 3 || d > 256) return tq::fail(TQ_ERR_UNSUPPORTED, "tq_make_rotation: d must be in 3..256");
    if (kind == TQ_ROT_RHT && (d < 4 || (d & (d - 1))))
        return tq::fail(TQ_ERR_UNSUPPORTED, "tq_make_rotation: RHT needs d a power of two >= 4");
    tq_rotation* r = new tq_rotation();
    r->d = d;
    r->kind = kind;
    r->seed = seed;
    r->pi.assign((size_t)d * d, 0.0);
    if (kind == TQ_ROT_DENSE_QR) {
        std::vector<double> g((size_t)d * d);
        tq::gaussians(seed, (int64_t)d * d, g.data());
        tq::householder_haar(g.data(), d, r->pi.data());
    } else {
        r->signs.resize(d);
        for (int i = 0; i < d; ++i) r->signs[i] = (tq::splitmix64_at(seed, i) >> 63) ? -1.0 : 1.0;
        const double inv = 1.0 / std::sqrt((double)d);
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) {
                double h = (__builtin_popcount((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
                r->pi[(size_t)i * d + j] = h * r->signs[j] * inv;
            }
    }
    *out = r;
    tq::bump_handle_generation();
    return TQ_OK;
}

tq_status tq_rotation_get(const tq_rotation* rot, double* host_out) {
    if (!rot || !host_out) return tq::fail(TQ_ERR_INVALID_ARG, "tq_rotation_get: NULL argument");
    std::memcpy(host_out, rot->pi.data(), rot->pi.size() * sizeof(double));
    return TQ_OK;
}

tq_status tq_rotation_info(const tq_rotation* rot, int* d, int* kind) {
    if (!rot) return tq::fail(TQ_ERR_INVALID_ARG, "tq_rotation_info: NULL handle");
    if (d) *d = rot->d;
    if (kind) *kind = rot->kind;
    return TQ_OK;
}

tq_status tq_make_qjl(uint64_t seed, int m, int d, tq_qjl** out) {
    if (!out) return tq::fail(TQ_ERR_INVALID_ARG, "tq_make_qjl: out is NULL");
    *out = nullptr;
    if (m < 1 || m > 256 || d < 3 || d > 256) return tq::fail(TQ_ERR_UNSUPPORTED, "tq_make_qjl: m in 1..256, d in 3..256");
    tq_qjl* q = new tq_qjl();
    q->m = m;
    q->d = d;
    q->seed = seed;
    q->s.resize((size_t)m * d);
    tq::gaussians(seed, (int64_t)m * d, q->s.data());
    for (double& v : q->s) v = tq::round_bf16(v);
    *out = q;
    tq::bump_handle_generation();
    return TQ_OK;
}

tq_status tq_qjl_get(const tq_qjl* qjl, double* host_out) {
    if (!qjl || !host_out) return tq::fail(TQ_ERR_INVALID_ARG, "tq_qjl_get: NULL argument");
    std::memcpy(host_out, qjl->s.data(), qjl->s.size() * sizeof(double));
    return TQ_OK;
}

tq_status tq_codebook(int d, int bits, double* centroids, double* boundaries) {
    std::vector<double> c, t;
    tq_status s = tq::codebook(d, bits, c, t);
    if (s != TQ_OK) return s;
    if (centroids) std::memcpy(centroids, c.data(), c.size() * sizeof(double));
    if (boundaries) std::memcpy(boundaries, t.data(), t.size() * sizeof(double));
    return TQ_OK;
}

int tq_code_bytes(int d, int code_bits) {
    if (d <= 0 || code_bits <= 0) return 0;
    int bytes = (code_bits * d + 7) / 8;
    return (bytes + 15) / 16 * 16;
}

int tq_code_bytes2(int d, int code_bits, int code_bits2) {
    if (code_bits2 == code_bits) return tq_code_bytes(d, code_bits);
    if (d <= 0 || code_bits <= 0 || code_bits2 <= 0) return 0;
    int n1 = 0;
    for (int i = 0; i < d; ++i) n1 += (i % 16) < 8 ? 1 : 0;
    const int bytes = (code_bits * n1 + code_bits2 * (d - n1) + 7) / 8;
    return (bytes + 7) / 8 * 8;
}

int tq_sign_bytes(int m) {
    if (m <= 0) return 0;
    return ((m + 7) / 8 + 15) / 16 * 16;
}

int tq_polar_code_bytes(int d, int bits1, int bits2) {
    if (d < 2 || (d & (d - 1)) || bits1 < 1 || bits1 > 4 || bits2 < 1 || bits2 > 4) return 0;
    const int bits = (d / 2) * bits1 + (d / 2 - 1) * bits2;
    return ((bits + 7) / 8 + 15) / 16 * 16;
}

tq_status tq_polar_codebook(int level, int bits, double* centroids, double* boundaries) {
    tq::clear_error();
    if (!centroids || !boundaries) return tq::fail(TQ_ERR_INVALID_ARG, "tq_polar_codebook: NULL output");
    std::vector<double> c, t;
    tq_status s = tq::polar_codebook(level, bits, c, t);
    if (s != TQ_OK) return s;
    std::copy(c.begin(), c.end(), centroids);
    std::copy(t.begin(), t.end(), boundaries);
    return TQ_OK;
}

}  // extern "C"
