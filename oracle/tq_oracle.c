/*
 * tq_oracle.c -- plain, slow CPU oracle for the TurboQuant KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only tests/, the smoke check and the CPU-baseline leg of the bench
 * use it.  It shares no code, header or table with the CUDA library: every
 * table it needs (signs, dense rotation, codebook) it builds itself from
 * (dim, bits, seed).
 *
 * Sources (titles of the pages and their sections):
 *  [PR]   "add TurboQuant KV cache compression" (mlx-swift-lm pull request #232):
 *         sections "Schemes" and "Design".
 *  [VQ]   VeloxQuant-MLX blog, post "How I built VeloxQuant-MLX":
 *         "Stage 1: Random Rotation", "Stage 2: Lloyd-Max Scalar Quantization",
 *         "The Core Idea", "The Bit-Packing Problem".
 *  [RVQ]  VeloxQuant-MLX blog, RVQ benchmark post, "The Throughput Problem"
 *         (Hadamard op count, boundary-sum quantisation).
 *  [TW]   "anyone still talking about mlx-swift-lm?" post: fused decode
 *         (score, softmax, inline dequant, K read in its rotated basis).
 *
 * Arithmetic (the reading this oracle fixes where the pages leave a choice open):
 *  - fp16 inputs are turned into exact integers k = x * 2^24 (|k| < 2^40).
 *  - Power-of-two d: w = H * (s (.) k) with the explicit Sylvester matrix
 *    H[i][j] = (-1)^popcount(i & j), in exact int64 ([VQ] Stage 1: random +-1
 *    diagonal applied before the Hadamard transform).
 *  - Other d: z_j = fma-chain over i ascending of Q[j][i] * k_i in fp64, Q the
 *    fp32-rounded orthogonal factor of a seeded Gaussian matrix ([PR] Design:
 *    dense fallback; [VQ] Stage 1: QR of a random Gaussian matrix).
 *  - S = sum k_i^2 as exact 128-bit integer; D = RN64(sqrt(RN64(S))).
 *    Stored norm = RN16(D * 2^-24) ([VQ] Stage 2: norm kept as fp16).
 *  - Codebook: Lloyd-Max for N(0,1) with 2^b levels, by numerical integration
 *    ([VQ] The Core Idea / Stage 2).  Centroids rounded to fp32, midpoints
 *    m_i = (c_i + c_{i+1}) / 2 in fp64 (exact).
 *  - code_j = #{ i : w_j > RN64(m_i * D) }  ([RVQ] boundary-sum: the index is
 *    the number of midpoints the value exceeds; ties go to the lower code).
 *    Dense path: z_j and D' = RN64(D / RN64(sqrt(d))) in place of w_j and D.
 *  - Bit packing LSB-first ([VQ] The Bit-Packing Problem).
 *  - Dequant x^ = n16 * R^T (c[codes] / sqrt(d)) with explicit matrices, fp64.
 *  - Attention: dequantise, then naive two-pass softmax in fp64.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no FMA contraction; fma()
 * only where written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef __int128 i128;
typedef unsigned __int128 u128;

/* ------------------------------------------------------------------------ */
/* SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number     */
/* generators", OOPSLA 2014), written from its published definition.        */
/* ------------------------------------------------------------------------ */
static uint64_t orc_sm64_next(uint64_t *state)
{
    uint64_t z;
    *state += 0x9E3779B97F4A7C15ULL;
    z = *state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

void orc_splitmix64(uint64_t seed, int64_t n, uint64_t *out)
{
    uint64_t s = seed;
    for (int64_t i = 0; i < n; ++i) out[i] = orc_sm64_next(&s);
}

/* Random signs for the WHT rotation: s_i = -1 when the top bit of the i-th
 * SplitMix64 output (state = seed) is set, else +1. */
void orc_signs(int d, uint64_t seed, int8_t *s)
{
    uint64_t st = seed;
    for (int i = 0; i < d; ++i) s[i] = (orc_sm64_next(&st) >> 63) ? -1 : 1;
}

/* Seeded standard normals by Box-Muller on 53-bit uniforms:
 * u1 = (x1 >> 11 + 1) 2^-53 in (0, 1], u2 = (x2 >> 11) 2^-53 in [0, 1),
 * z0 = r cos(2 pi u2), z1 = r sin(2 pi u2), r = sqrt(-2 ln u1). */
void orc_gaussian(int64_t n, uint64_t seed, double *out)
{
    uint64_t st = seed;
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t i = 0; i < n; i += 2) {
        double u1 = (double)((orc_sm64_next(&st) >> 11) + 1) * 0x1.0p-53;
        double u2 = (double)(orc_sm64_next(&st) >> 11) * 0x1.0p-53;
        double r = sqrt(-2.0 * log(u1));
        out[i] = r * cos(two_pi * u2);
        if (i + 1 < n) out[i + 1] = r * sin(two_pi * u2);
    }
}

/* Explicit Sylvester-ordered Hadamard matrix H[i][j] = (-1)^popcount(i&j). */
void orc_hadamard(int d, int32_t *H)
{
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            H[(int64_t)i * d + j] = (__builtin_popcount((unsigned)(i & j)) & 1) ? -1 : 1;
}

/* Dense rotation for non-power-of-two d: G (d x d, row-major, filled from
 * orc_gaussian(d*d, seed)) = Q R with diag(R) > 0, by modified Gram-Schmidt
 * on the columns of G, applied twice for orthogonality to rounding level.
 * The rotation is z = Q k, Q[j][i] = row j, column i.  Returned in fp32 (RN).
 * Returns 0, or -1 if a column is numerically dependent. */
int orc_dense_q(int d, uint64_t seed, float *Qout)
{
    int64_t dd = (int64_t)d * d;
    double *G = (double *)malloc(sizeof(double) * dd);
    double *Qc = (double *)malloc(sizeof(double) * dd); /* column-major work */
    if (!G || !Qc) { free(G); free(Qc); return -1; }
    orc_gaussian(dd, seed, G);
    for (int j = 0; j < d; ++j)
        for (int i = 0; i < d; ++i) Qc[(int64_t)j * d + i] = G[(int64_t)i * d + j];
    for (int j = 0; j < d; ++j) {
        double *v = Qc + (int64_t)j * d;
        for (int pass = 0; pass < 2; ++pass) {
            for (int p = 0; p < j; ++p) {
                const double *u = Qc + (int64_t)p * d;
                double dot = 0.0;
                for (int i = 0; i < d; ++i) dot += u[i] * v[i];
                for (int i = 0; i < d; ++i) v[i] -= dot * u[i];
            }
        }
        double nrm = 0.0;
        for (int i = 0; i < d; ++i) nrm += v[i] * v[i];
        nrm = sqrt(nrm);
        if (!(nrm > 1e-300)) { free(G); free(Qc); return -1; }
        for (int i = 0; i < d; ++i) v[i] /= nrm;
    }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) Qout[(int64_t)i * d + j] = (float)Qc[(int64_t)j * d + i];
    free(G); free(Qc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Lloyd-Max codebook for N(0,1) by numerical integration ([VQ] The Core Idea:
 * boundaries are midpoints of neighbouring centroids, each centroid is the
 * conditional mean of the density over its cell).                          */
/* ------------------------------------------------------------------------ */
static double orc_pdf(double x) { return exp(-0.5 * x * x) * 0.39894228040143267793994605993438; }

#define ORC_SUPPORT 12.0   /* mass beyond |x| = 12 is below 1e-32 */
#define ORC_H0 (1.0 / 4096.0)

/* Composite Simpson on [a, b] of f(x) and x f(x); at least 64 panels and
 * panel width at most 1/4096. */
static void orc_cell_integrals(double a, double b, double *mass, double *first)
{
    if (a < -ORC_SUPPORT) a = -ORC_SUPPORT;
    if (b > ORC_SUPPORT) b = ORC_SUPPORT;
    if (!(b > a)) { *mass = 0.0; *first = 0.0; return; }
    int64_t n = (int64_t)ceil((b - a) / ORC_H0);
    if (n < 64) n = 64;
    if (n & 1) ++n;
    double h = (b - a) / (double)n;
    double s0 = 0.0, s1 = 0.0;
    for (int64_t k = 0; k <= n; ++k) {
        double x = a + h * (double)k;
        if (k == n) x = b;
        double w = (k == 0 || k == n) ? 1.0 : ((k & 1) ? 4.0 : 2.0);
        double f = orc_pdf(x);
        s0 += w * f;
        s1 += w * x * f;
    }
    *mass = s0 * h / 3.0;
    *first = s1 * h / 3.0;
}

/* One evaluation of the cell statistics for centroids c[0..n-1]:
 * D_i (mass), E_i (conditional mean), and the density at the cell ends. */
static void orc_cells(int n, const double *c, double *D, double *E, double *fa, double *fb,
                      double *lo, double *hi)
{
    for (int i = 0; i < n; ++i) {
        double a = (i == 0) ? -ORC_SUPPORT : 0.5 * (c[i - 1] + c[i]);
        double b = (i == n - 1) ? ORC_SUPPORT : 0.5 * (c[i] + c[i + 1]);
        double m0, m1;
        orc_cell_integrals(a, b, &m0, &m1);
        D[i] = m0;
        E[i] = m1 / m0;
        lo[i] = a; hi[i] = b;
        fa[i] = (i == 0) ? 0.0 : orc_pdf(a);
        fb[i] = (i == n - 1) ? 0.0 : orc_pdf(b);
    }
}

/* Lloyd-Max fixed point for N(0,1) with n = 2^bits levels.
 * 1. Start from n points evenly spaced on [-3, 3].
 * 2. Lloyd steps: boundaries <- midpoints, centroids <- conditional means,
 *    until the largest move is below 1e-14 or 200 steps.
 * 3. Newton steps on the same conditions F_i(c) = c_i - E_i(c) = 0 (the plain
 *    Lloyd step contracts too slowly at 256 levels); the tridiagonal Jacobian
 *    follows from dE/db = f(b)(b - E)/D and dE/da = f(a)(E - a)/D.
 * 4. Symmetrise (c_i = -c_{n-1-i}), round to fp32, midpoints in fp64.
 * Outputs: c64[n] (fp64 fixed point), c32[n] (fp32), mid[n-1] (fp64), and
 * the final residual max|c - E| in *resid.  Returns the number of steps. */
int orc_lloyd_max(int bits, double *c64, float *c32, double *mid, double *resid)
{
    int n = 1 << bits;
    double *c = c64;
    double *D = (double *)malloc(sizeof(double) * n * 8);
    if (!D) return -1;
    double *E = D + n, *fa = D + 2 * n, *fb = D + 3 * n, *lo = D + 4 * n, *hi = D + 5 * n;
    double *sub = D + 6 * n, *tmp = D + 7 * n;
    int steps = 0;
    if (n == 1) { c[0] = 0.0; }
    else for (int i = 0; i < n; ++i) c[i] = -3.0 + 6.0 * (double)i / (double)(n - 1);
    if (n > 1) {
        for (int it = 0; it < 200; ++it) {
            orc_cells(n, c, D, E, fa, fb, lo, hi);
            double mv = 0.0;
            for (int i = 0; i < n; ++i) { double dlt = fabs(E[i] - c[i]); if (dlt > mv) mv = dlt; c[i] = E[i]; }
            ++steps;
            if (mv < 1e-14) break;
        }
        for (int it = 0; it < 60; ++it) {
            orc_cells(n, c, D, E, fa, fb, lo, hi);
            /* J dc = -F with J tridiagonal: J_ii = 1 - (dE_i/da + dE_i/db)/2,
             * J_i,i-1 = -(dE_i/da)/2, J_i,i+1 = -(dE_i/db)/2 (Thomas algorithm). */
            double *cp = sub, *dp = tmp;
            for (int i = 0; i < n; ++i) {
                double dEa = (i == 0) ? 0.0 : fa[i] * (E[i] - lo[i]) / D[i];
                double dEb = (i == n - 1) ? 0.0 : fb[i] * (hi[i] - E[i]) / D[i];
                double dgi = 1.0 - 0.5 * dEa - 0.5 * dEb;
                double lower = -0.5 * dEa;
                double upper = -0.5 * dEb;
                double r = E[i] - c[i];
                if (i == 0) { cp[i] = upper / dgi; dp[i] = r / dgi; }
                else {
                    double den = dgi - lower * cp[i - 1];
                    cp[i] = upper / den;
                    dp[i] = (r - lower * dp[i - 1]) / den;
                }
            }
            for (int i = n - 2; i >= 0; --i) dp[i] -= cp[i] * dp[i + 1];
            double mv = 0.0;
            for (int i = 0; i < n; ++i) { c[i] += dp[i]; if (fabs(dp[i]) > mv) mv = fabs(dp[i]); }
            ++steps;
            if (mv < 1e-15) break;
        }
        for (int i = 0; i < n / 2; ++i) {
            double v = 0.5 * (c[n - 1 - i] - c[i]);
            c[n - 1 - i] = v;
            c[i] = -v;
        }
        orc_cells(n, c, D, E, fa, fb, lo, hi);
        double r = 0.0;
        for (int i = 0; i < n; ++i) { double dlt = fabs(c[i] - E[i]); if (dlt > r) r = dlt; }
        if (resid) *resid = r;
    } else if (resid) *resid = 0.0;
    for (int i = 0; i < n; ++i) c32[i] = (float)c[i];
    for (int i = 0; i + 1 < n; ++i) mid[i] = ((double)c32[i] + (double)c32[i + 1]) * 0.5;
    free(D);
    return steps;
}

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 conversions written from the format definition.        */
/* ------------------------------------------------------------------------ */
double orc_f16_to_f64(uint16_t h)
{
    int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024), e - 25);
    return sign ? -v : v;
}

/* Round-to-nearest-even from fp64 to binary16, overflow to infinity. */
uint16_t orc_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return 0x7E00;
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1) */
    int ue = e - 1;                /* a = 1.xxx * 2^ue */
    int q;                         /* quantum exponent: ulp = 2^q */
    if (ue < -14) q = -24;         /* subnormal range: ulp 2^-24 */
    else q = ue - 10;
    double scaled = ldexp(a, -q);  /* exact: a / ulp */
    double fl = floor(scaled);
    double rem = scaled - fl;      /* exact */
    uint64_t mant = (uint64_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (mant & 1))) mant += 1;
    /* mant * 2^q is the rounded magnitude */
    if (q == -24) {
        if (mant >= 1024) return (uint16_t)(sign | (1 << 10) | (mant - 1024)); /* rounds up to min normal */
        return (uint16_t)(sign | mant);
    }
    if (mant == 2048) { mant = 1024; q += 1; ue += 1; }
    int biased = ue + 15;
    if (biased >= 31) return (uint16_t)(sign | 0x7C00);
    return (uint16_t)(sign | (biased << 10) | (mant - 1024));
}

/* fp16 bit pattern -> exact integer k = x * 2^24 (finite inputs only). */
static int64_t orc_f16_exact(uint16_t h)
{
    int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    int64_t k = (e == 0) ? (int64_t)m : ((int64_t)(m + 1024) << (e - 1));
    return sign ? -k : k;
}

/* ------------------------------------------------------------------------ */
/* Bit packing: bit (j*b + t) of a vector's stream is bit t of code j;       */
/* stream bit p lives in byte p/8 at bit p%8 ([VQ] The Bit-Packing Problem). */
/* ------------------------------------------------------------------------ */
void orc_pack(const int32_t *codes, int d, int bits, uint8_t *out)
{
    int nbytes = (d * bits + 7) / 8;
    memset(out, 0, (size_t)nbytes);
    for (int j = 0; j < d; ++j)
        for (int t = 0; t < bits; ++t)
            if ((codes[j] >> t) & 1) {
                int p = j * bits + t;
                out[p / 8] |= (uint8_t)(1u << (p % 8));
            }
}

void orc_unpack(const uint8_t *in, int d, int bits, int32_t *codes)
{
    for (int j = 0; j < d; ++j) {
        int v = 0;
        for (int t = 0; t < bits; ++t) {
            int p = j * bits + t;
            if ((in[p / 8] >> (p % 8)) & 1) v |= 1 << t;
        }
        codes[j] = v;
    }
}

/* ------------------------------------------------------------------------ */
/* Codec: everything the oracle needs for one (dim, bits, seed).            */
/* ------------------------------------------------------------------------ */
typedef struct {
    int d, bits, is_wht;
    int8_t *s;          /* [d] signs (WHT) */
    int32_t *H;         /* [d*d] explicit Hadamard (WHT) */
    float *Q;           /* [d*d] dense rotation (other d) */
    double *c64;        /* [2^b] */
    float *c32;         /* [2^b] */
    double *mid;        /* [2^b - 1] */
} orc_codec;

void orc_codec_free(orc_codec *c)
{
    if (!c) return;
    free(c->s); free(c->H); free(c->Q); free(c->c64); free(c->c32); free(c->mid);
    free(c);
}

/* bits == 16 means raw fp16 (no codebook, no rotation use). */
orc_codec *orc_codec_new(int d, int bits, uint64_t seed)
{
    orc_codec *c = (orc_codec *)calloc(1, sizeof(orc_codec));
    if (!c) return NULL;
    c->d = d; c->bits = bits;
    c->is_wht = (d > 0) && ((d & (d - 1)) == 0);
    if (c->is_wht) {
        c->s = (int8_t *)malloc((size_t)d);
        c->H = (int32_t *)malloc(sizeof(int32_t) * (size_t)d * d);
        if (!c->s || !c->H) { orc_codec_free(c); return NULL; }
        orc_signs(d, seed, c->s);
        orc_hadamard(d, c->H);
    } else {
        c->Q = (float *)malloc(sizeof(float) * (size_t)d * d);
        if (!c->Q || orc_dense_q(d, seed, c->Q) != 0) { orc_codec_free(c); return NULL; }
    }
    if (bits != 16) {
        int n = 1 << bits;
        c->c64 = (double *)malloc(sizeof(double) * n);
        c->c32 = (float *)malloc(sizeof(float) * n);
        c->mid = (double *)malloc(sizeof(double) * (n > 1 ? n - 1 : 1));
        if (!c->c64 || !c->c32 || !c->mid) { orc_codec_free(c); return NULL; }
        double r;
        orc_lloyd_max(bits, c->c64, c->c32, c->mid, &r);
    }
    return c;
}

int orc_codec_dim(const orc_codec *c) { return c->d; }
int orc_codec_is_wht(const orc_codec *c) { return c->is_wht; }
void orc_codec_tables(const orc_codec *c, int8_t *s, float *Q, float *c32, double *mid)
{
    int d = c->d;
    if (s && c->s) memcpy(s, c->s, (size_t)d);
    if (Q && c->Q) memcpy(Q, c->Q, sizeof(float) * (size_t)d * d);
    if (c->bits != 16) {
        int n = 1 << c->bits;
        if (c32) memcpy(c32, c->c32, sizeof(float) * n);
        if (mid) memcpy(mid, c->mid, sizeof(double) * (n - 1));
    }
}

/* Rotated coordinates of one fp16 vector, unnormalised:
 * WHT: w = H (s . k) exactly (returned as double, |w| < 2^53);
 * dense: z_j = fma-chain(Q[j][i], k_i) over i ascending.
 * Also returns D = RN64(sqrt(RN64(S))) and the threshold scale. */
static void orc_rotate(const orc_codec *c, const uint16_t *x, double *w, double *Dout, double *scale_out)
{
    int d = c->d;
    int64_t *k = (int64_t *)malloc(sizeof(int64_t) * d);
    u128 S = 0;
    for (int i = 0; i < d; ++i) {
        k[i] = orc_f16_exact(x[i]);
        int64_t a = k[i] < 0 ? -k[i] : k[i];
        S += (u128)a * (u128)a;
    }
    double Sd = (double)S;            /* correctly rounded conversion */
    double D = sqrt(Sd);
    if (c->is_wht) {
        for (int j = 0; j < d; ++j) {
            i128 acc = 0;
            for (int i = 0; i < d; ++i)
                acc += (i128)c->H[(int64_t)j * d + i] * (i128)(c->s[i] * k[i]);
            w[j] = (double)(int64_t)acc;
        }
        *scale_out = D;
    } else {
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc = fma((double)c->Q[(int64_t)j * d + i], (double)k[i], acc);
            w[j] = acc;
        }
        *scale_out = D / sqrt((double)d);
    }
    *Dout = D;
    free(k);
}

/* Encode n vectors (row stride x_stride elements) into packed codes (row
 * stride code_stride bytes) and fp16 norms.  Cross-checks every coordinate
 * against brute-force nearest-centroid search in long double on t = w / D:
 * *n_neartie counts coordinates where the two disagree but t lies within
 * 1e-12 of a midpoint (an allowed near-tie); *n_mismatch counts any other
 * disagreement (expected 0). */
int orc_encode(const orc_codec *c, const uint16_t *x, int64_t n, int64_t x_stride,
               uint8_t *codes, int64_t code_stride, uint16_t *norms,
               int64_t *n_neartie, int64_t *n_mismatch)
{
    int d = c->d, b = c->bits, L = 1 << b;
    double *w = (double *)malloc(sizeof(double) * d);
    int32_t *cd = (int32_t *)malloc(sizeof(int32_t) * d);
    double *T = (double *)malloc(sizeof(double) * L);
    int64_t ties = 0, mism = 0;
    if (!w || !cd || !T) { free(w); free(cd); free(T); return -1; }
    for (int64_t v = 0; v < n; ++v) {
        double D, sc;
        orc_rotate(c, x + v * x_stride, w, &D, &sc);
        for (int i = 0; i + 1 < L; ++i) T[i] = c->mid[i] * sc;
        for (int j = 0; j < d; ++j) {
            int cnt = 0;
            for (int i = 0; i + 1 < L; ++i) if (w[j] > T[i]) ++cnt;
            cd[j] = cnt;
            /* brute force: argmin |t - c_i|, ties to the lower index */
            if (sc > 0.0) {
                long double t = (long double)w[j] / (long double)sc;
                int best = 0; long double bd = fabsl(t - (long double)c->c32[0]);
                for (int i = 1; i < L; ++i) {
                    long double dd = fabsl(t - (long double)c->c32[i]);
                    if (dd < bd) { bd = dd; best = i; }
                }
                if (best != cnt) {
                    int lo = best < cnt ? best : cnt;
                    int near = 0;
                    for (int i = lo; i < (best > cnt ? best : cnt); ++i) {
                        long double m = (long double)c->mid[i];
                        long double tol = 1e-12L * (fabsl(m) > 1.0L ? fabsl(m) : 1.0L);
                        if (fabsl(t - m) <= tol) near = 1;
                    }
                    if (near) ++ties; else ++mism;
                }
            }
        }
        orc_pack(cd, d, b, codes + v * code_stride);
        norms[v] = orc_f64_to_f16(ldexp(D, -24));
    }
    if (n_neartie) *n_neartie = ties;
    if (n_mismatch) *n_mismatch = mism;
    free(w); free(cd); free(T);
    return 0;
}

/* Integer codes of one vector (for tests of the quantiser itself). */
int orc_encode_codes(const orc_codec *c, const uint16_t *x, int32_t *codes_out, double *w_out, double *D_out)
{
    int d = c->d, L = 1 << c->bits;
    double *w = (double *)malloc(sizeof(double) * d);
    double D, sc;
    if (!w) return -1;
    orc_rotate(c, x, w, &D, &sc);
    for (int j = 0; j < d; ++j) {
        int cnt = 0;
        for (int i = 0; i + 1 < L; ++i) if (w[j] > c->mid[i] * sc) ++cnt;
        codes_out[j] = cnt;
        if (w_out) w_out[j] = w[j];
    }
    if (D_out) *D_out = D;
    free(w);
    return 0;
}

/* R^T applied to y (fp64): x = R^T y with R = H diag(s) / sqrt(d) (WHT) or Q. */
static void orc_rotate_back(const orc_codec *c, const double *y, double *x)
{
    int d = c->d;
    double inv = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        if (c->is_wht) {
            for (int j = 0; j < d; ++j) acc += (double)c->H[(int64_t)j * d + i] * y[j];
            x[i] = acc * (double)c->s[i] * inv;
        } else {
            for (int j = 0; j < d; ++j) acc += (double)c->Q[(int64_t)j * d + i] * y[j];
            x[i] = acc;
        }
    }
}

/* Dequantise n packed vectors: x^ = n16 * R^T (c[codes] / sqrt(d)), fp64. */
int orc_dequant(const orc_codec *c, const uint8_t *codes, int64_t code_stride, const uint16_t *norms,
                int64_t n, double *out)
{
    int d = c->d;
    int32_t *cd = (int32_t *)malloc(sizeof(int32_t) * d);
    double *y = (double *)malloc(sizeof(double) * d);
    if (!cd || !y) { free(cd); free(y); return -1; }
    double rs = 1.0 / sqrt((double)d);
    for (int64_t v = 0; v < n; ++v) {
        orc_unpack(codes + v * code_stride, d, c->bits, cd);
        double nn = orc_f16_to_f64(norms[v]);
        for (int j = 0; j < d; ++j) y[j] = (double)c->c32[cd[j]] * rs * nn;
        orc_rotate_back(c, y, out + v * d);
    }
    free(cd); free(y);
    return 0;
}

/* ---------------------------------------------------------------------------
 * QJL residual sketch (TurboQuantProd: "How I built VeloxQuant-MLX", Stage 3:
 * QJL Residual Correction).  A key keeps its b-bit MSE codes and norm (the
 * codec above, b = its bits) plus one sign bit per sketch row of its residual
 * and the residual's norm.  Readings fixed here, where the page leaves them open:
 *  - sketch S: m = d rows of iid N(0,1), the Gaussian stream of seed + 2
 *    (orc_gaussian), rounded to fp32, row-major S[j][i];
 *  - residual, in the rotated basis and scaled by sqrt(d) (power-of-two d):
 *    rho_i = RN64(w_i 2^-24 - n16 c[code_i]) (one fma), rounded to fp32;
 *  - sign bit j = 1 when t_j < 0, t_j = fp32 fma chain over i ascending of
 *    S[j][i] rho_i (the decision is taken in fp32, in this order), packed
 *    LSB-first, d / 8 bytes per vector;
 *  - residual norm gamma = RN16(RN64(sqrt(G2 / d))), G2 = fp64 chain over i
 *    ascending of rho_i^2 (exact products), so gamma = |k - k^_MSE|;
 *  - estimator (unbiased, the QJL form): <q, k> ~ <q, k^_MSE>
 *    + gamma sqrt(pi/2) / m sum_j z_j <S_j, R q>, z_j = +1 / -1 for bit 0 / 1.
 *    (The page prints the correction with sign(<S_j, q>) and pi/(2m); that
 *    product of two signs estimates an angle, not the inner product, and is
 *    not unbiased as the page says the correction is: the unbiased QJL form is
 *    taken.) */
float *orc_qjl_sketch(int d, uint64_t seed)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)d * d);
    float *S = (float *)malloc(sizeof(float) * (size_t)d * d);
    if (!g || !S) { free(g); free(S); return NULL; }
    orc_gaussian((int64_t)d * d, seed + 2, g);
    for (int64_t i = 0; i < (int64_t)d * d; ++i) S[i] = (float)g[i];
    free(g);
    return S;
}

void orc_qjl_sketch_copy(int d, uint64_t seed, float *out)
{
    float *S = orc_qjl_sketch(d, seed);
    if (S) { memcpy(out, S, sizeof(float) * (size_t)d * d); free(S); }
}

/* Encode n vectors with the MSE codec c (power-of-two d) plus the QJL sketch of
 * their residuals: codes / norms as orc_encode, signs [n][d/8] (row stride
 * sign_stride bytes), rnorms [n] fp16. */
int orc_encode_qjl(const orc_codec *c, uint64_t seed, const uint16_t *x, int64_t n, int64_t x_stride,
                   uint8_t *codes, int64_t code_stride, uint16_t *norms, uint8_t *signs, int64_t sign_stride,
                   uint16_t *rnorms)
{
    int d = c->d;
    if (!c->is_wht || c->bits == 16) return -1;
    if (orc_encode(c, x, n, x_stride, codes, code_stride, norms, NULL, NULL) != 0) return -1;
    float *S = orc_qjl_sketch(d, seed);
    double *w = (double *)malloc(sizeof(double) * d);
    int32_t *cd = (int32_t *)malloc(sizeof(int32_t) * d);
    float *rho = (float *)malloc(sizeof(float) * d);
    if (!S || !w || !cd || !rho) { free(S); free(w); free(cd); free(rho); return -1; }
    for (int64_t v = 0; v < n; ++v) {
        double D, sc;
        orc_rotate(c, x + v * x_stride, w, &D, &sc);
        orc_unpack(codes + v * code_stride, d, c->bits, cd);
        double n16 = orc_f16_to_f64(norms[v]);
        double G2 = 0.0;
        for (int i = 0; i < d; ++i) {
            double r64 = fma(-n16, (double)c->c32[cd[i]], ldexp(w[i], -24));
            rho[i] = (float)r64;
            G2 = fma((double)rho[i], (double)rho[i], G2);
        }
        rnorms[v] = orc_f64_to_f16(sqrt(G2 / (double)d));
        uint8_t *sg = signs + v * sign_stride;
        memset(sg, 0, (size_t)d / 8);
        for (int j = 0; j < d; ++j) {
            float t = 0.0f;
            for (int i = 0; i < d; ++i) t = fmaf(S[(int64_t)j * d + i], rho[i], t);
            if (t < 0.0f) sg[j >> 3] |= (uint8_t)(1u << (j & 7));
        }
    }
    free(S); free(w); free(cd); free(rho);
    return 0;
}

/* Estimated inner products <q_g, k_n> (unscaled) of G queries [G][d] with len
 * keys stored as MSE codes + norms + QJL signs + residual norms, fp64:
 * <q, k^_MSE> + gamma sqrt(pi/2) / d sum_j z_j (S R q)_j. */
int orc_qjl_scores(const orc_codec *ck, uint64_t seed, const uint16_t *q, int G, const uint8_t *k_codes,
                   const uint16_t *k_norms, const uint8_t *k_signs, const uint16_t *k_rnorms, int64_t len,
                   double *out)
{
    int d = ck->d;
    if (!ck->is_wht || ck->bits == 16) return -1;
    if (len <= 0) return 0;
    int bpk = d * ck->bits / 8;
    float *S = orc_qjl_sketch(d, seed);
    double *Kh = (double *)malloc(sizeof(double) * (size_t)len * d);
    double *rq = (double *)malloc(sizeof(double) * d);
    double *u = (double *)malloc(sizeof(double) * d);
    if (!S || !Kh || !rq || !u) { free(S); free(Kh); free(rq); free(u); return -1; }
    orc_dequant(ck, k_codes, bpk, k_norms, len, Kh);
    const double coef = sqrt(acos(-1.0) / 2.0) / (double)d;
    for (int g = 0; g < G; ++g) {
        const uint16_t *qg = q + (int64_t)g * d;
        /* R q = H diag(s) q / sqrt(d), explicit matrix */
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += (double)ck->H[(int64_t)j * d + i] * (double)ck->s[i] * orc_f16_to_f64(qg[i]);
            rq[j] = acc / sqrt((double)d);
        }
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += (double)S[(int64_t)j * d + i] * rq[i];
            u[j] = acc;
        }
        for (int64_t t = 0; t < len; ++t) {
            double mse = 0.0, corr = 0.0;
            for (int i = 0; i < d; ++i) mse += orc_f16_to_f64(qg[i]) * Kh[t * d + i];
            const uint8_t *sg = k_signs + t * (d / 8);
            for (int j = 0; j < d; ++j) corr += ((sg[j >> 3] >> (j & 7)) & 1u) ? -u[j] : u[j];
            out[(int64_t)g * len + t] = mse + orc_f16_to_f64(k_rnorms[t]) * coef * corr;
        }
    }
    free(S); free(Kh); free(rq); free(u);
    return 0;
}

/* Decode attention of G query heads over len keys stored with the QJL sketch
 * (scores from orc_qjl_scores, times scale) and MSE-coded values: naive
 * two-pass softmax, fp64.  len == 0 gives zeros. */
int orc_attention_qjl_unit(const orc_codec *ck, uint64_t seed, const orc_codec *cv, const uint16_t *q, int G,
                           const uint8_t *k_codes, const uint16_t *k_norms, const uint8_t *k_signs,
                           const uint16_t *k_rnorms, const uint8_t *v_codes, const uint16_t *v_norms, int64_t len,
                           double scale, double *out)
{
    int d = cv->d;
    memset(out, 0, sizeof(double) * (size_t)G * d);
    if (len <= 0) return 0;
    double *sc = (double *)malloc(sizeof(double) * (size_t)G * len);
    double *Vh = (double *)malloc(sizeof(double) * (size_t)len * d);
    if (!sc || !Vh) { free(sc); free(Vh); return -1; }
    if (orc_qjl_scores(ck, seed, q, G, k_codes, k_norms, k_signs, k_rnorms, len, sc) != 0 ||
        orc_dequant(cv, v_codes, d * cv->bits / 8, v_norms, len, Vh) != 0) {
        free(sc); free(Vh); return -1;
    }
    for (int g = 0; g < G; ++g) {
        double *s = sc + (int64_t)g * len;
        double mx = -INFINITY;
        for (int64_t t = 0; t < len; ++t) { s[t] *= scale; if (s[t] > mx) mx = s[t]; }
        double l = 0.0;
        for (int64_t t = 0; t < len; ++t) { s[t] = exp(s[t] - mx); l += s[t]; }
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int64_t t = 0; t < len; ++t) acc += s[t] * Vh[t * d + i];
            out[(int64_t)g * d + i] = acc / l;
        }
    }
    free(sc); free(Vh);
    return 0;
}

/* Decode attention of G query heads over the first `len` cached tokens of one
 * (batch, KV head) unit followed by `n_tail` raw fp16 tokens (k_tail, v_tail,
 * [n_tail][d]): tokens kept unencoded -- the pending tokens that wait in fp16
 * for a full batch ("add TurboQuant KV cache compression", Design) and fp16
 * sink tokens (turboquant-mlx guide "KV cache compression") -- read in the
 * same softmax as the packed cache.  The definition written out:
 * dequantise the cache, append the tail, naive two-pass softmax in fp64.
 * lse (optional, [G]) receives log(sum_t exp(s_t)) of the scaled scores.
 * With no token at all the output is zero and lse is -inf. */
int orc_attention_unit_tail(const orc_codec *ck, const orc_codec *cv, const uint16_t *q, int G,
                            const void *k, const uint16_t *k_norms, const uint8_t *v_codes,
                            const uint16_t *v_norms, int64_t len, const uint16_t *k_tail,
                            const uint16_t *v_tail, int64_t n_tail, double scale, double *out,
                            double *lse)
{
    int d = cv->d;
    if (len < 0) len = 0;
    if (n_tail < 0) n_tail = 0;
    int64_t n = len + n_tail;
    if (n <= 0) {
        memset(out, 0, sizeof(double) * (size_t)G * d);
        if (lse) for (int g = 0; g < G; ++g) lse[g] = -INFINITY;
        return 0;
    }
    int bpk = d * ck->bits / 8, bpv = d * cv->bits / 8;
    double *Kh = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *Vh = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!Kh || !Vh || !s) { free(Kh); free(Vh); free(s); return -1; }
    if (len > 0) {
        if (ck->bits == 16) {
            const uint16_t *kr = (const uint16_t *)k;
            for (int64_t i = 0; i < len * d; ++i) Kh[i] = orc_f16_to_f64(kr[i]);
        } else {
            orc_dequant(ck, (const uint8_t *)k, bpk, k_norms, len, Kh);
        }
        orc_dequant(cv, v_codes, bpv, v_norms, len, Vh);
    }
    for (int64_t i = 0; i < n_tail * d; ++i) {
        Kh[len * d + i] = orc_f16_to_f64(k_tail[i]);
        Vh[len * d + i] = orc_f16_to_f64(v_tail[i]);
    }
    for (int g = 0; g < G; ++g) {
        double mx = -INFINITY;
        for (int64_t t = 0; t < n; ++t) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += orc_f16_to_f64(q[(int64_t)g * d + i]) * Kh[t * d + i];
            s[t] = scale * acc;
            if (s[t] > mx) mx = s[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < n; ++t) { s[t] = exp(s[t] - mx); l += s[t]; }
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int64_t t = 0; t < n; ++t) acc += s[t] * Vh[t * d + i];
            out[(int64_t)g * d + i] = acc / l;
        }
        if (lse) lse[g] = mx + log(l);
    }
    free(Kh); free(Vh); free(s);
    return 0;
}

/* Attention of L consecutive query positions per query head over one (batch,
 * KV head) unit: the L query rows of each of the G heads sharing the KV head
 * ("add TurboQuant KV cache compression", review of the NR0 path: a query
 * chunk holds L rows per head, and a row's KV head follows from its query head).
 * The sequence is the first `len` cached tokens followed by `n_tail` raw fp16
 * tokens, P = len + n_tail tokens at positions 0 .. P-1; the queries are the
 * last L positions, query l at position P - L + l, and each attends to the
 * tokens at positions up to its own (causal).  The definition written out: the
 * full score matrix of every query against every token, an additive mask of
 * -inf above each query's position, a naive two-pass softmax per row, fp64.
 * q, out: [G][L][d] (head-major rows).  A row with no visible token gives 0. */
int orc_attention_multi_unit(const orc_codec *ck, const orc_codec *cv, const uint16_t *q, int G, int L,
                             const void *k, const uint16_t *k_norms, const uint8_t *v_codes,
                             const uint16_t *v_norms, int64_t len, const uint16_t *k_tail,
                             const uint16_t *v_tail, int64_t n_tail, double scale, double *out)
{
    int d = cv->d;
    if (len < 0) len = 0;
    if (n_tail < 0) n_tail = 0;
    if (G <= 0 || L <= 0) return -1;
    int64_t n = len + n_tail;
    int64_t rows = (int64_t)G * L;
    memset(out, 0, sizeof(double) * (size_t)rows * d);
    if (n <= 0) return 0;
    int bpk = d * ck->bits / 8, bpv = d * cv->bits / 8;
    double *Kh = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *Vh = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *S = (double *)malloc(sizeof(double) * (size_t)rows * n);
    if (!Kh || !Vh || !S) { free(Kh); free(Vh); free(S); return -1; }
    if (len > 0) {
        if (ck->bits == 16) {
            const uint16_t *kr = (const uint16_t *)k;
            for (int64_t i = 0; i < len * d; ++i) Kh[i] = orc_f16_to_f64(kr[i]);
        } else {
            orc_dequant(ck, (const uint8_t *)k, bpk, k_norms, len, Kh);
        }
        orc_dequant(cv, v_codes, bpv, v_norms, len, Vh);
    }
    for (int64_t i = 0; i < n_tail * d; ++i) {
        Kh[len * d + i] = orc_f16_to_f64(k_tail[i]);
        Vh[len * d + i] = orc_f16_to_f64(v_tail[i]);
    }
    /* scores with the causal mask: row r = g * L + l sits at position n - L + l */
    for (int64_t r = 0; r < rows; ++r) {
        int64_t pos = n - L + (r % L);
        for (int64_t t = 0; t < n; ++t) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += orc_f16_to_f64(q[r * d + i]) * Kh[t * d + i];
            S[r * n + t] = (t <= pos) ? scale * acc : -INFINITY;
        }
    }
    for (int64_t r = 0; r < rows; ++r) {
        double *s = S + r * n;
        double mx = -INFINITY;
        for (int64_t t = 0; t < n; ++t) if (s[t] > mx) mx = s[t];
        if (mx == -INFINITY) continue;  /* no visible token: the row stays 0 */
        double l = 0.0;
        for (int64_t t = 0; t < n; ++t) { s[t] = exp(s[t] - mx); l += s[t]; }
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int64_t t = 0; t < n; ++t) acc += s[t] * Vh[t * d + i];
            out[r * d + i] = acc / l;
        }
    }
    free(Kh); free(Vh); free(S);
    return 0;
}

int orc_attention_unit(const orc_codec *ck, const orc_codec *cv, const uint16_t *q, int G,
                       const void *k, const uint16_t *k_norms, const uint8_t *v_codes,
                       const uint16_t *v_norms, int64_t len, double scale, double *out)
{
    return orc_attention_unit_tail(ck, cv, q, G, k, k_norms, v_codes, v_norms, len, NULL, NULL, 0, scale,
                                   out, NULL);
}
