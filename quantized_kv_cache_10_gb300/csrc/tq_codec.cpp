// tq_codec.cpp -- host construction of the codec tables (once per
// (dim, bits, seed), shared by every layer that uses it: "add TurboQuant KV
// cache compression", Design, "Shared codecs").
//
//  * Rademacher signs for the WHT rotation ("How I built VeloxQuant-MLX",
//    Stage 1: random +-1 diagonal, then the Hadamard transform).
//  * Dense orthogonal rotation for other head sizes (same page, Stage 1: QR of
//    a random Gaussian matrix), by Householder reflections with the signs of
//    R's diagonal made positive.
//  * Lloyd-Max codebook of N(0,1) with 2^bits levels ("How I built
//    VeloxQuant-MLX", The Core Idea and Stage 2): boundaries are midpoints,
//    centroids are conditional means, with the closed form
//    E[X | a < X < b] = (phi(a) - phi(b)) / (Phi(b) - Phi(a)).  Solved for the
//    thresholds of the positive half line by damped Newton steps from the
//    companding (Panter-Dite) start, not by Lloyd's alternation.
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "tq_internal.h"

namespace tq {

namespace {

// SplitMix64 (Steele, Lea and Flood, OOPSLA 2014), from its published definition.
struct SplitMix64 {
    uint64_t s;
    explicit SplitMix64(uint64_t seed) : s(seed) {}
    uint64_t next() {
        s += 0x9E3779B97F4A7C15ULL;
        uint64_t z = s;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
        return z ^ (z >> 31);
    }
};

constexpr double kInvSqrt2Pi = 0.39894228040143267793994605993438;
constexpr double kInvSqrt2 = 0.70710678118654752440084436210485;

double pdf(double x) { return std::isinf(x) ? 0.0 : std::exp(-0.5 * x * x) * kInvSqrt2Pi; }
double upper_tail(double x) { return 0.5 * std::erfc(x * kInvSqrt2); }  // P(X > x)

}  // namespace

void rademacher_signs(int dim, uint64_t seed, std::vector<int8_t>& s) {
    SplitMix64 g(seed);
    s.resize(dim);
    for (int i = 0; i < dim; ++i) s[i] = (g.next() >> 63) ? int8_t(-1) : int8_t(1);
}

// Gaussian matrix from Box-Muller on 53-bit uniforms u1 in (0,1], u2 in [0,1),
// filled row-major; then Q from Householder QR with diag(R) > 0 (the unique
// QR factor).  z = Q k.  Returns 0 on success.
void gaussian_stream(size_t n, uint64_t seed, std::vector<double>& A) {
    A.resize(n);
    SplitMix64 g(seed);
    const double two_pi = 6.283185307179586476925286766559;
    for (size_t i = 0; i < n; i += 2) {
        double u1 = double((g.next() >> 11) + 1) * 0x1.0p-53;
        double u2 = double(g.next() >> 11) * 0x1.0p-53;
        double r = std::sqrt(-2.0 * std::log(u1));
        A[i] = r * std::cos(two_pi * u2);
        if (i + 1 < n) A[i + 1] = r * std::sin(two_pi * u2);
    }
}

int dense_rotation(int dim, uint64_t seed, std::vector<float>& qout) {
    const int d = dim;
    const size_t dd = size_t(d) * d;
    std::vector<double> A;
    gaussian_stream(dd, seed, A);
    // Householder: A (row-major, A[i*d + j]) -> R in the upper triangle.
    std::vector<double> V(dd, 0.0);  // reflector k stored in V[k*d + i], i >= k
    for (int k = 0; k < d; ++k) {
        double nrm = 0.0;
        for (int i = k; i < d; ++i) nrm += A[size_t(i) * d + k] * A[size_t(i) * d + k];
        nrm = std::sqrt(nrm);
        if (!(nrm > 1e-300)) return -1;
        double x0 = A[size_t(k) * d + k];
        double alpha = (x0 >= 0.0) ? -nrm : nrm;
        double* v = &V[size_t(k) * d];
        for (int i = k; i < d; ++i) v[i] = A[size_t(i) * d + k];
        v[k] -= alpha;
        double vn = 0.0;
        for (int i = k; i < d; ++i) vn += v[i] * v[i];
        vn = std::sqrt(vn);
        if (vn > 0.0)
            for (int i = k; i < d; ++i) v[i] /= vn;
        for (int j = k; j < d; ++j) {
            double dot = 0.0;
            for (int i = k; i < d; ++i) dot += v[i] * A[size_t(i) * d + j];
            for (int i = k; i < d; ++i) A[size_t(i) * d + j] -= 2.0 * v[i] * dot;
        }
    }
    // Q = H_0 H_1 ... H_{d-1}: apply reflectors in reverse to the identity.
    std::vector<double> Q(dd, 0.0);
    for (int i = 0; i < d; ++i) Q[size_t(i) * d + i] = 1.0;
    for (int k = d - 1; k >= 0; --k) {
        const double* v = &V[size_t(k) * d];
        for (int j = 0; j < d; ++j) {
            double dot = 0.0;
            for (int i = k; i < d; ++i) dot += v[i] * Q[size_t(i) * d + j];
            for (int i = k; i < d; ++i) Q[size_t(i) * d + j] -= 2.0 * v[i] * dot;
        }
    }
    // Make diag(R) positive: negate column j of Q where R_jj < 0.
    qout.resize(dd);
    for (int j = 0; j < d; ++j) {
        double sg = (A[size_t(j) * d + j] < 0.0) ? -1.0 : 1.0;
        for (int i = 0; i < d; ++i) qout[size_t(i) * d + j] = float(sg * Q[size_t(i) * d + j]);
    }
    return 0;
}

// Lloyd-Max codebook of N(0,1) with n = 2^bits levels ("How I built VeloxQuant-MLX",
// Stage 2: boundaries are the midpoints of neighbouring centroids, each centroid the
// conditional mean of its cell).  The density is even, so the codebook is antisymmetric
// and only the positive half line is solved: m = n/2 cells (t_{j-1}, t_j), t_0 = 0,
// t_m = +inf, with the m - 1 inner thresholds as the unknowns,
//   F_j(t) = t_j - (mu_j + mu_{j+1}) / 2 = 0,   mu_j = E[X | t_{j-1} < X < t_j],
// started from the companding (Panter-Dite) point density p^(1/3) -- for N(0,1) a
// normal of variance 3, so t_j = sqrt(3) Phi^-1(1/2 + j/n) -- and solved by damped
// Newton steps (tridiagonal Jacobian; a step is halved while it does not lower max|F|).
namespace {

// E[X | a < X < b] for 0 <= a < b <= inf, its cell mass and the partial derivatives.
struct HalfCell {
    double mass, mean, d_lo, d_hi;  // d_lo = d mean / d a, d_hi = d mean / d b
};

HalfCell half_cell(double a, double b) {
    HalfCell h;
    h.mass = upper_tail(a) - upper_tail(b);
    const double pa = pdf(a), pb = pdf(b);
    h.mean = (pa - pb) / h.mass;
    h.d_lo = pa * (h.mean - a) / h.mass;
    h.d_hi = std::isinf(b) ? 0.0 : pb * (b - h.mean) / h.mass;
    return h;
}

// x >= 0 with P(X > x) = q, 0 < q <= 1/2 (bisection; the tail is decreasing).
double upper_quantile(double q) {
    double lo = 0.0, hi = 40.0;
    for (int it = 0; it < 200 && hi - lo > 0.0; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (mid == lo || mid == hi) break;
        (upper_tail(mid) > q ? lo : hi) = mid;
    }
    return 0.5 * (lo + hi);
}

}  // namespace

void lloyd_max_gaussian(int bits, std::vector<double>& c) {
    const int n = 1 << bits, m = n / 2;
    c.assign(n, 0.0);
    if (n == 1) return;
    // t[0] = 0, t[1..m-1] unknown, t[m] = inf
    std::vector<double> t(m + 1), F(m), sub(m), dia(m), sup(m), step(m), trial(m + 1);
    t[0] = 0.0;
    t[m] = INFINITY;
    const double s3 = std::sqrt(3.0);
    for (int j = 1; j < m; ++j) t[j] = s3 * upper_quantile(0.5 - double(j) / double(n));
    std::vector<HalfCell> cell(m + 1);
    auto residual = [&](const std::vector<double>& tt) {
        for (int j = 1; j <= m; ++j) cell[j] = half_cell(tt[j - 1], tt[j]);
        double r = 0.0;
        for (int j = 1; j < m; ++j) {
            F[j] = tt[j] - 0.5 * (cell[j].mean + cell[j + 1].mean);
            r = std::fmax(r, std::fabs(F[j]));
        }
        return r;
    };
    double r = residual(t);
    for (int it = 0; it < 100 && r > 0.0; ++it) {
        // Jacobian rows j = 1 .. m-1: dF_j / dt_{j-1}, dt_j, dt_{j+1}
        for (int j = 1; j < m; ++j) {
            sub[j] = (j > 1) ? -0.5 * cell[j].d_lo : 0.0;
            dia[j] = 1.0 - 0.5 * (cell[j].d_hi + cell[j + 1].d_lo);
            sup[j] = (j + 1 < m) ? -0.5 * cell[j + 1].d_hi : 0.0;
            step[j] = -F[j];
        }
        // tridiagonal elimination, then back substitution
        for (int j = 2; j < m; ++j) {
            const double f = sub[j] / dia[j - 1];
            dia[j] -= f * sup[j - 1];
            step[j] -= f * step[j - 1];
        }
        for (int j = m - 1; j >= 1; --j) step[j] = (step[j] - ((j + 1 < m) ? sup[j] * step[j + 1] : 0.0)) / dia[j];
        // damping: keep the thresholds increasing and max|F| falling
        double lam = 1.0, rn = r, smax = 0.0;
        for (int tries = 0; tries < 40; ++tries, lam *= 0.5) {
            bool ordered = true;
            trial[0] = 0.0;
            trial[m] = INFINITY;
            for (int j = 1; j < m; ++j) {
                trial[j] = t[j] + lam * step[j];
                if (!(trial[j] > trial[j - 1])) ordered = false;
            }
            if (!ordered) continue;
            rn = residual(trial);
            if (rn < r) break;
        }
        smax = 0.0;
        for (int j = 1; j < m; ++j) smax = std::fmax(smax, std::fabs(trial[j] - t[j]));
        if (!(rn < r)) {  // no decrease: at the rounding floor
            residual(t);
            break;
        }
        t.swap(trial);
        r = rn;
        if (smax < 1e-16) break;
    }
    residual(t);  // the cells of the final thresholds
    for (int j = 1; j <= m; ++j) {
        c[m - 1 + j] = cell[j].mean;
        c[m - j] = -cell[j].mean;
    }
}

int num_sms(int device) {
    static std::mutex mu;
    static std::vector<int> cache;
    std::lock_guard<std::mutex> lk(mu);
    if (device < 0) return 1;
    if (size_t(device) >= cache.size()) cache.resize(device + 1, 0);
    if (cache[device] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0)
            v = 1;
        cache[device] = v;
    }
    return cache[device];
}

}  // namespace tq

// ---------------------------------------------------------------------------
// Decode-table construction lives with the tensor-core kernel that reads it.
namespace tq {
void build_decode_tables(tq_codec& c, std::vector<uint32_t>& ktab, std::vector<uint32_t>& vtab);
}

namespace {

template <typename T>
cudaError_t upload(T** dst, const T* src, size_t n) {
    if (n == 0) return cudaSuccess;
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(dst), n * sizeof(T));
    if (e != cudaSuccess) return e;
    return cudaMemcpy(*dst, src, n * sizeof(T), cudaMemcpyHostToDevice);
}

void free_device(tq_codec* c) {
    cudaFree(c->d_centroids);
    cudaFree(c->d_midpoints);
    cudaFree(c->d_sign_bits);
    cudaFree(c->d_q);
    cudaFree(c->d_qt);
    cudaFree(c->d_ktab);
    cudaFree(c->d_vtab);
    cudaFree(c->d_sketch);
    cudaFree(c->d_sketch_t);
}

}  // namespace

extern "C" {

int tq_version(void) { return 10000; }

const char* tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID_ARG: return "invalid argument";
        case TQ_ERR_UNSUPPORTED: return "unsupported";
        case TQ_ERR_CUDA: return "CUDA error";
        case TQ_ERR_OOM: return "out of memory";
        case TQ_ERR_WORKSPACE: return "workspace too small";
        case TQ_ERR_DEVICE_CHECK: return "device-side check failed";
    }
    return "unknown status";
}

tq_status tq_codec_create(int dim, int bits, uint64_t seed, tq_codec** out) {
    if (!out) return TQ_ERR_INVALID_ARG;
    *out = nullptr;
    if (dim < 32 || dim > 512 || dim % 32 != 0) return TQ_ERR_INVALID_ARG;
    if (!(bits == 2 || bits == 3 || bits == 4 || bits == 8 || bits == 16)) return TQ_ERR_INVALID_ARG;
    tq_codec* c = new (std::nothrow) tq_codec();
    if (!c) return TQ_ERR_OOM;
    c->dim = dim;
    c->bits = bits;
    c->seed = seed;
    c->is_wht = (dim & (dim - 1)) == 0;
    c->bytes_per_vec = (bits == 16) ? dim * 2 : dim * bits / 8;
    if (cudaGetDevice(&c->device) != cudaSuccess) {
        delete c;
        return TQ_ERR_CUDA;
    }
    if (c->is_wht) {
        tq::rademacher_signs(dim, seed, c->signs);
    } else if (tq::dense_rotation(dim, seed, c->dense_q) != 0) {
        delete c;
        return TQ_ERR_INVALID_ARG;
    }
    if (bits != 16) {
        std::vector<double> c64;
        tq::lloyd_max_gaussian(bits, c64);
        const int n = 1 << bits;
        c->centroids.resize(n);
        for (int i = 0; i < n; ++i) c->centroids[i] = float(c64[i]);
        c->midpoints.resize(n - 1);
        for (int i = 0; i + 1 < n; ++i)
            c->midpoints[i] = (double(c->centroids[i]) + double(c->centroids[i + 1])) * 0.5;
    }
    cudaError_t e = cudaSuccess;
    if (bits != 16) {
        e = upload(&c->d_centroids, c->centroids.data(), c->centroids.size());
        if (e == cudaSuccess) e = upload(&c->d_midpoints, c->midpoints.data(), c->midpoints.size());
    }
    if (e == cudaSuccess && c->is_wht) {
        std::vector<uint32_t> sb(dim / 32 < 4 ? 4 : dim / 32, 0u);  // >= 16 B: read by 16-byte bulk copies
        for (int j = 0; j < dim; ++j)
            if (c->signs[j] < 0) sb[j / 32] |= 1u << (j % 32);
        e = upload(&c->d_sign_bits, sb.data(), sb.size());
    }
    if (e == cudaSuccess && !c->is_wht) {
        std::vector<float> qt(size_t(dim) * dim);
        for (int i = 0; i < dim; ++i)
            for (int j = 0; j < dim; ++j) qt[size_t(j) * dim + i] = c->dense_q[size_t(i) * dim + j];
        e = upload(&c->d_q, c->dense_q.data(), c->dense_q.size());
        if (e == cudaSuccess) e = upload(&c->d_qt, qt.data(), qt.size());
    }
    if (e == cudaSuccess) {
        std::vector<uint32_t> kt, vt;
        tq::build_decode_tables(*c, kt, vt);
        c->ktab_words = int(kt.size());
        c->vtab_words = int(vt.size());
        e = upload(&c->d_ktab, kt.data(), kt.size());
        if (e == cudaSuccess) e = upload(&c->d_vtab, vt.data(), vt.size());
    }
    if (e != cudaSuccess) {
        free_device(c);
        delete c;
        return e == cudaErrorMemoryAllocation ? TQ_ERR_OOM : TQ_ERR_CUDA;
    }
    *out = c;
    return TQ_OK;
}

tq_status tq_codec_create_qjl(int dim, int bits, uint64_t seed, tq_codec** out) {
    if (!out) return TQ_ERR_INVALID_ARG;
    *out = nullptr;
    if ((dim & (dim - 1)) != 0 || !(bits == 2 || bits == 3 || bits == 4)) return TQ_ERR_INVALID_ARG;
    tq_codec* c = nullptr;
    tq_status s = tq_codec_create(dim, bits, seed, &c);
    if (s != TQ_OK) return s;
    // S: the Gaussian stream of seed + 2 ("How I built VeloxQuant-MLX", Stage 3: a random
    // Johnson-Lindenstrauss projection of the residual), rounded to fp32
    std::vector<double> g;
    tq::gaussian_stream(size_t(dim) * dim, seed + 2, g);
    c->sketch.resize(g.size());
    for (size_t i = 0; i < g.size(); ++i) c->sketch[i] = float(g[i]);
    std::vector<float> st(c->sketch.size());
    for (int j = 0; j < dim; ++j)
        for (int i = 0; i < dim; ++i) st[size_t(i) * dim + j] = c->sketch[size_t(j) * dim + i];
    cudaError_t e = upload(&c->d_sketch, c->sketch.data(), c->sketch.size());
    if (e == cudaSuccess) e = upload(&c->d_sketch_t, st.data(), st.size());
    if (e != cudaSuccess) {
        tq_codec_destroy(c);
        return e == cudaErrorMemoryAllocation ? TQ_ERR_OOM : TQ_ERR_CUDA;
    }
    c->qjl = 1;
    *out = c;
    return TQ_OK;
}

tq_status tq_codec_export_sketch(const tq_codec* c, float* sketch) {
    if (!c || !sketch || !c->qjl) return TQ_ERR_INVALID_ARG;
    std::memcpy(sketch, c->sketch.data(), c->sketch.size() * sizeof(float));
    return TQ_OK;
}

void tq_codec_destroy(tq_codec* c) {
    if (!c) return;
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != c->device) cudaSetDevice(c->device);
    free_device(c);
    if (prev >= 0 && prev != c->device) cudaSetDevice(prev);
    delete c;
}

tq_status tq_codec_info(const tq_codec* c, int* dim, int* bits, int* bytes_per_vec, int* is_wht,
                        const float** centroids_host) {
    if (!c) return TQ_ERR_INVALID_ARG;
    if (dim) *dim = c->dim;
    if (bits) *bits = c->bits;
    if (bytes_per_vec) *bytes_per_vec = c->bytes_per_vec;
    if (is_wht) *is_wht = c->is_wht;
    if (centroids_host) *centroids_host = (c->bits != 16) ? c->centroids.data() : nullptr;
    return TQ_OK;
}

tq_status tq_codec_export_rotation(const tq_codec* c, int8_t* signs, float* dense_q) {
    return tq_codec_export(c, signs, dense_q, nullptr, nullptr);
}

tq_status tq_codebook_gaussian(int bits, float* centroids, double* midpoints) {
    if (bits < 1 || bits > 8 || !centroids) return TQ_ERR_INVALID_ARG;
    std::vector<double> c64;
    tq::lloyd_max_gaussian(bits, c64);
    const int n = 1 << bits;
    for (int i = 0; i < n; ++i) centroids[i] = float(c64[i]);
    if (midpoints)
        for (int i = 0; i + 1 < n; ++i) midpoints[i] = (double(centroids[i]) + double(centroids[i + 1])) * 0.5;
    return TQ_OK;
}

tq_status tq_codec_export(const tq_codec* c, int8_t* signs, float* dense_q, float* centroids,
                          double* midpoints) {
    if (!c) return TQ_ERR_INVALID_ARG;
    if (signs && c->is_wht) std::memcpy(signs, c->signs.data(), c->signs.size());
    if (dense_q && !c->is_wht) std::memcpy(dense_q, c->dense_q.data(), c->dense_q.size() * sizeof(float));
    if (c->bits != 16) {
        if (centroids) std::memcpy(centroids, c->centroids.data(), c->centroids.size() * sizeof(float));
        if (midpoints) std::memcpy(midpoints, c->midpoints.data(), c->midpoints.size() * sizeof(double));
    }
    return TQ_OK;
}

}  // extern "C"
