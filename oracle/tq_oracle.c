/*
 * tq_oracle.c -- plain, slow, scalar CPU oracle for rotated + quantized KV-cache
 * compression and for decode attention over the compressed cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load, link or run
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant generator with the CUDA
 * library; the two meet only in the byte format documented below.
 *
 * Sources (web pages on the subject, cited by page title and section):
 *   [MLX]  "turboquant-mlx" (TurboQuant-MLX v2.0 README): "Walsh-Hadamard Rotation"
 *          (SRHT D @ H @ D, O(n log n)), "Asymmetric K/V Compression" (QJL on keys
 *          only), "FP16 Attention Sinks", "Dynamic Chunk Buffering", "How It Works /
 *          Pipeline", "RaBitQ vs QJL correction" (QJLSketch(head_dim, sketch_dim)).
 *   [MOQ]  "TurboMOQ" (turboMOQ README): "Architecture" (keys: rotate -> symmetric
 *          quantize; values: Lloyd-Max codebook -> grid quantize; per-head 1-8 bits;
 *          optional QJL residual), "Progressive temporal tiering", "QJL residual
 *          correction (sub-2-bit)" (corrected = quantized + correction), "Project
 *          Structure" (bit packing utilities).
 *   [SKL]  "turboquant-mlx" skill note: "Standalone Benchmark" (per-layer seed 42 + i),
 *          "Optimisations Metal" (inverse transform pulled out of V-attention).
 *
 * Readings taken where the pages are silent:
 *   - PRNG: SplitMix64 (Steele, Lea, Flood 2014).
 *   - D @ H @ D uses ONE sign diagonal on both sides, so R = D H D / sqrt(d) is
 *     symmetric and R R = I; its inverse is R itself.
 *   - Compression arithmetic is a fixed sequence of IEEE-754 binary32 operations
 *     (round to nearest even, no fused multiply-add), so the codes are a pure
 *     function of the fp16 input; attention is evaluated in binary64.
 *   - Keys: midrise uniform grid with 2^b cells on [-m, m], m = max |y_i|.
 *     Values: Gaussian Lloyd-Max codebook applied to y / sigma, sigma = RMS of y.
 *   - Packing: code i of a vector occupies bits [b*i, b*i + b) of its record,
 *     little-endian (LSB-first) bitstream; a record is d*b/8 bytes.
 *   - QJL: S is jl x d with N(0,1) entries (Box-Muller on SplitMix64 words);
 *     sign bit j = 1 iff (S r)_j >= 0; residual norm rho = ||r||_2.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared -lm
 * (-ffp-contract=off matters: GCC contracts a*b+c into an FMA by default on arm64.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TQO_MAX_D 1024
#define TQO_PI 3.14159265358979323846

/* ------------------------------------------------------------------------ */
/* SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number      */
/* generators", OOPSLA 2014): add the golden-gamma, then the variant-13 mix.  */
/* ------------------------------------------------------------------------ */
static uint64_t sm64_next(uint64_t *state) {
    uint64_t z;
    *state += 0x9E3779B97F4A7C15ull;
    z = *state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void tqo_splitmix64(uint64_t seed, int n, uint64_t *out) {
    uint64_t s = seed;
    for (int i = 0; i < n; i++) out[i] = sm64_next(&s);
}

/* Sign diagonal D of the SRHT for one layer: word i of the stream seeded with
 * `seed` gives D_i = -1 when its top bit is set, +1 otherwise ([MLX] "Walsh-
 * Hadamard Rotation": WalshHadamardRotation(head_dim, seed); [SKL] per-layer
 * seed + i). */
void tqo_signs(int d, uint64_t seed, int8_t *sign) {
    uint64_t s = seed;
    for (int i = 0; i < d; i++) sign[i] = (sm64_next(&s) >> 63) ? -1 : 1;
}

/* IEEE-754 binary16 -> double, written from the format: 1 sign bit, 5 exponent
 * bits (bias 15), 10 fraction bits; exponent 0 is subnormal, 31 is inf/NaN. */
double tqo_half_to_double(uint16_t h) {
    int sgn = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp((double)(1024 + f), e - 25);
    return sgn ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* Rotation y = R x, R = (1/sqrt(d)) D H D ([MLX] "Walsh-Hadamard Rotation").  */
/* ------------------------------------------------------------------------ */

/* binary32 evaluation order (part of the compressed format): sign flip (exact),
 * fast Walsh-Hadamard butterflies with stage widths h = 1, 2, 4, ..., d/2 in that
 * order, each pair (i, i+h) with i & h == 0 becoming (a+b, a-b); output sign flip
 * (exact); then one rounded multiply by c = binary32(1/sqrt(d)). */
void tqo_rotate_f32(int d, const int8_t *sign, const float *x, float *y) {
    float a[TQO_MAX_D];
    const float c = (float)(1.0 / sqrt((double)d));
    for (int i = 0; i < d; i++) a[i] = sign[i] < 0 ? -x[i] : x[i];
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; i++)
            if ((i & h) == 0) {
                float u = a[i], v = a[i + h];
                a[i] = u + v;
                a[i + h] = u - v;
            }
    for (int i = 0; i < d; i++) y[i] = c * (sign[i] < 0 ? -a[i] : a[i]);
}

/* The same transform in binary64 (used for attention and for the original-space
 * view of dequantized vectors).  R is its own inverse. */
void tqo_rotate_f64(int d, const int8_t *sign, const double *x, double *y) {
    double a[TQO_MAX_D];
    const double c = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; i++) a[i] = sign[i] < 0 ? -x[i] : x[i];
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; i++)
            if ((i & h) == 0) {
                double u = a[i], v = a[i + h];
                a[i] = u + v;
                a[i + h] = u - v;
            }
    for (int i = 0; i < d; i++) y[i] = c * (sign[i] < 0 ? -a[i] : a[i]);
}

/* ------------------------------------------------------------------------ */
/* Gaussian Lloyd-Max codebook ([MOQ] "Architecture": values use a Lloyd-Max  */
/* codebook; fitted here in closed form for the N(0,1) law, not on data).     */
/* ------------------------------------------------------------------------ */
/* Dense rotation ("TurboMOQ", "Stable QR Rotation": a Haar-random orthogonal
 * matrix from a QR factorisation): y = Q x with Q a d x d binary32 matrix,
 * row-major.  The binary32 form takes the exact product (binary64 sums of
 * binary32 x binary16 terms, ~1e-16 relative) rounded once to binary32. */
void tqo_rotate_dense_f32(int d, const float *Q, const float *x, float *y) {
    for (int i = 0; i < d; i++) {
        double acc = 0.0;
        for (int j = 0; j < d; j++) acc += (double)Q[(size_t)i * d + j] * (double)x[j];
        y[i] = (float)acc;
    }
}

/* y = Q x (transpose = 0) or y = Q^T x (transpose = 1) in binary64. */
void tqo_rotate_dense_f64(int d, const float *Q, int transpose, const double *x, double *y) {
    for (int i = 0; i < d; i++) {
        double acc = 0.0;
        for (int j = 0; j < d; j++)
            acc += (double)(transpose ? Q[(size_t)j * d + i] : Q[(size_t)i * d + j]) * x[j];
        y[i] = acc;
    }
}

static double std_pdf(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * TQO_PI); }
/* Upper tail Q(x) = P(X > x) = erfc(x / sqrt 2) / 2, accurate for large x. */
static double std_tail(double x) { return 0.5 * erfc(x / sqrt(2.0)); }

/* Inverse of the tail: the x with Q(x) = p, by bisection (slow, but obviously
 * right). */
static double std_tail_inv(double p) {
    double lo = -40.0, hi = 40.0;
    for (int it = 0; it < 200; it++) {
        double mid = 0.5 * (lo + hi);
        if (std_tail(mid) > p) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

/* Lloyd's iteration for n = 2^bits levels: thresholds are midpoints of adjacent
 * centroids; each centroid is the conditional mean of N(0,1) on its cell,
 * (pdf(a) - pdf(b)) / (P(a < X < b)).  The codebook is odd-symmetric, so only the
 * upper half is iterated (cell probabilities from the upper tail, which keeps the
 * outer cells accurate) and the lower half is its mirror; the middle threshold
 * is exactly 0.  Starts from the quantiles (k + 1/2)/n and stops when no
 * centroid moves by more than 1e-13 (or after max_iter sweeps).  Returns the
 * number of sweeps, or -1 on bad arguments. */
int tqo_lloyd_max(int bits, double *centroid, double *threshold, int max_iter) {
    if (bits < 1 || bits > 8) return -1;
    const int n = 1 << bits, half = n / 2;
    double c[256], t[257];
    for (int k = half; k < n; k++) c[k] = std_tail_inv(1.0 - (k + 0.5) / n);
    int it;
    for (it = 1; it <= max_iter; it++) {
        /* t[k] is the boundary between cells k-1 and k, for the upper half. */
        t[half] = 0.0;
        for (int k = half + 1; k < n; k++) t[k] = 0.5 * (c[k - 1] + c[k]);
        double delta = 0.0;
        for (int k = half; k < n; k++) {
            /* pdf(a) - pdf(b) = pdf(a) * (1 - exp(-(b - a)(b + a)/2)), written with
             * expm1 so that narrow cells (8 bits) keep full relative precision. */
            double a = t[k];
            double pa = std_tail(a), pb = 0.0, num = std_pdf(a);
            if (k + 1 < n) {
                double b = t[k + 1];
                pb = std_tail(b);
                num = -std_pdf(a) * expm1(-0.5 * (b - a) * (b + a));
            }
            double nc = num / (pa - pb);
            double dd = fabs(nc - c[k]);
            if (dd > delta) delta = dd;
            c[k] = nc;
        }
        if (delta <= 1e-13) break;
    }
    for (int k = half; k < n; k++) c[n - 1 - k] = -c[k];
    for (int k = 0; k < n; k++) centroid[k] = c[k];
    for (int k = 0; k + 1 < n; k++) threshold[k] = 0.5 * (c[k] + c[k + 1]);
    threshold[half - 1] = 0.0;
    return it;
}

/* ------------------------------------------------------------------------ */
/* Sphere-coordinate Lloyd-Max codebook ("TurboMOQ", "Head-to-Head Comparison":  */
/* a Beta-CDF codebook beside the Lloyd-Max one; "Project Structure": Beta-    */
/* distribution codebooks).  Reading: after a random rotation a coordinate of   */
/* a d-vector, divided by the vector's RMS, is sqrt(d) times a coordinate of a  */
/* uniform unit vector, whose density is proportional to (1 - u^2/d)^((d-3)/2) */
/* on |u| < sqrt(d) (a scaled symmetric Beta((d-1)/2, (d-1)/2) law).  Same     */
/* Lloyd iteration as the Gaussian codebook, with this law.                    */
/* ------------------------------------------------------------------------ */

/* Gauss-Legendre nodes and weights on [-1, 1] (n points), by Newton's method
 * on the Legendre recurrence. */
static void gauss_legendre(int n, double *x, double *w) {
    for (int i = 0; i < (n + 1) / 2; i++) {
        double z = cos(TQO_PI * (i + 0.75) / (n + 0.5)), dp = 1.0;
        for (int it = 0; it < 100; it++) {
            double p0 = 1.0, p1 = 0.0;
            for (int j = 1; j <= n; j++) {
                const double p2 = p1;
                p1 = p0;
                p0 = ((2.0 * j - 1.0) * z * p1 - (j - 1.0) * p2) / j;
            }
            dp = n * (z * p0 - p1) / (z * z - 1.0);
            const double dz = p0 / dp;
            z -= dz;
            if (fabs(dz) < 1e-16) break;
        }
        x[i] = -z;
        x[n - 1 - i] = z;
        w[i] = w[n - 1 - i] = 2.0 / ((1.0 - z * z) * dp * dp);
    }
}

/* integral of (1 - s^2)^a over [s0, s1] within [0, 1]: composite 20-point
 * Gauss-Legendre on `panels` equal panels. */
static double sphere_mass(double a, double s0, double s1, int panels) {
    static double gx[20], gw[20];
    static int ready = 0;
    if (!ready) {
        gauss_legendre(20, gx, gw);
        ready = 1;
    }
    double sum = 0.0;
    const double h = (s1 - s0) / panels;
    for (int p = 0; p < panels; p++) {
        const double lo = s0 + p * h, mid = lo + 0.5 * h;
        for (int i = 0; i < 20; i++) {
            const double s = mid + 0.5 * h * gx[i];
            sum += gw[i] * exp(a * log1p(-s * s));
        }
    }
    return 0.5 * h * sum;
}

int tqo_lloyd_max_sphere(int bits, int d, double *centroid, double *threshold, int max_iter) {
    if (bits < 1 || bits > 8 || d < 4) return -1;
    const int n = 1 << bits, half = n / 2;
    const double a = 0.5 * (d - 3), rd = sqrt((double)d);
    /* upper tail P(U > x) up to the normalisation, as a mass in s = u / sqrt(d) */
    const double total = sphere_mass(a, 0.0, 1.0, 256);  /* half the full mass */
    double c[256], t[257];
    for (int k = half; k < n; k++) {
        /* initial centroid: the quantile (k + 1/2)/n, by bisection on the tail */
        const double p = 1.0 - (k + 0.5) / n;  /* upper tail probability, < 1/2 */
        double lo = 0.0, hi = 1.0;
        for (int it = 0; it < 80; it++) {
            const double mid = 0.5 * (lo + hi);
            if (sphere_mass(a, mid, 1.0, 32) / (2.0 * total) > p) lo = mid; else hi = mid;
        }
        c[k] = rd * 0.5 * (lo + hi);
    }
    int it;
    for (it = 1; it <= max_iter; it++) {
        t[half] = 0.0;
        for (int k = half + 1; k < n; k++) t[k] = 0.5 * (c[k - 1] + c[k]);
        double delta = 0.0;
        for (int k = half; k < n; k++) {
            /* centroid of [x0, x1]: int u f / int f with f = (1 - u^2/d)^a; the
             * numerator is d/(2(a+1)) ((1 - x0^2/d)^(a+1) - (1 - x1^2/d)^(a+1)),
             * written with expm1 for narrow cells */
            const double x0 = t[k], x1 = k + 1 < n ? t[k + 1] : rd;
            const double l0 = log1p(-x0 * x0 / d);
            double num;
            if (k + 1 < n) {
                const double l1 = log1p(-x1 * x1 / d);
                num = -exp((a + 1.0) * l0) * expm1((a + 1.0) * (l1 - l0));
            } else {
                num = exp((a + 1.0) * l0);
            }
            num *= d / (2.0 * (a + 1.0));
            const int panels = k + 1 < n ? 2 : 64;
            const double den = rd * sphere_mass(a, x0 / rd, x1 / rd, panels);
            const double nc = num / den;
            const double dd = fabs(nc - c[k]);
            if (dd > delta) delta = dd;
            c[k] = nc;
        }
        if (delta <= 1e-13) break;
    }
    for (int k = half; k < n; k++) c[n - 1 - k] = -c[k];
    for (int k = 0; k < n; k++) centroid[k] = c[k];
    for (int k = 0; k + 1 < n; k++) threshold[k] = 0.5 * (c[k] + c[k + 1]);
    threshold[half - 1] = 0.0;
    return it;
}

/* ------------------------------------------------------------------------ */
/* Scalar quantizers (binary32 order is part of the format).                  */
/* ------------------------------------------------------------------------ */

/* Keys ([MOQ] "Architecture": rotate -> symmetric quantize, per-head bits):
 * m = max |y_i|; r = binary32(1/m) (r = 0 when m = 0); v = y*r; t = v + 1;
 * code = clamp(floor(t * 2^(b-1)), 0, 2^b - 1).  Dequantized value (cell centre):
 * m * ((code + 1/2) * 2^(1-b) - 1). */
void tqo_quant_key(int d, int b, const float *y, uint8_t *code, float *scale) {
    float m = 0.0f;
    for (int i = 0; i < d; i++) {
        float a = fabsf(y[i]);
        if (a > m) m = a;
    }
    const float r = m > 0.0f ? 1.0f / m : 0.0f;
    const float half_cells = (float)(1 << (b - 1));
    const int top = (1 << b) - 1;
    for (int i = 0; i < d; i++) {
        float v = y[i] * r;
        float t = v + 1.0f;
        float u = t * half_cells;
        int k = (int)floorf(u);
        if (k < 0) k = 0;
        if (k > top) k = top;
        code[i] = (uint8_t)k;
    }
    *scale = m;
}

/* Cell centre of a key code in units of m (exact in binary32). */
double tqo_key_level(int b, int code) {
    return (code + 0.5) * ldexp(1.0, 1 - b) - 1.0;
}

/* Values ([MOQ] "Architecture": Lloyd-Max codebook -> grid quantize):
 * sigma = sqrt(S / d) with S the sum of y_i^2 taken as a pairwise binary tree in
 * index order ((y0^2 + y1^2) + (y2^2 + y3^2)) + ...; r = binary32(1/sigma) (0 when
 * sigma = 0); u = y * r; code = #{k : thr[k] < u} (a tie goes to the lower code).
 * thr holds the 2^b - 1 binary32 thresholds. */
void tqo_quant_value(int d, int b, const float *y, const float *thr, uint8_t *code,
                     float *scale) {
    float p[TQO_MAX_D];
    for (int i = 0; i < d; i++) p[i] = y[i] * y[i];
    for (int len = d; len > 1; len >>= 1)
        for (int j = 0; j < len / 2; j++) p[j] = p[2 * j] + p[2 * j + 1];
    const float sigma = sqrtf(p[0] / (float)d);
    const float r = sigma > 0.0f ? 1.0f / sigma : 0.0f;
    const int nthr = (1 << b) - 1;
    for (int i = 0; i < d; i++) {
        float u = y[i] * r;
        int k = 0;
        for (int j = 0; j < nthr; j++)
            if (thr[j] < u) k++;
        code[i] = (uint8_t)k;
    }
    *scale = sigma;
}

/* ------------------------------------------------------------------------ */
/* Bit packing ([MOQ] "Project Structure": bit packing utilities).             */
/* ------------------------------------------------------------------------ */
void tqo_pack(int d, int b, const uint8_t *code, uint8_t *rec) {
    memset(rec, 0, (size_t)d * b / 8);
    for (int i = 0; i < d; i++)
        for (int j = 0; j < b; j++)
            if ((code[i] >> j) & 1) {
                int bit = i * b + j;
                rec[bit >> 3] |= (uint8_t)(1u << (bit & 7));
            }
}

void tqo_unpack(int d, int b, const uint8_t *rec, uint8_t *code) {
    for (int i = 0; i < d; i++) {
        int v = 0;
        for (int j = 0; j < b; j++) {
            int bit = i * b + j;
            v |= ((rec[bit >> 3] >> (bit & 7)) & 1) << j;
        }
        code[i] = (uint8_t)v;
    }
}

/* ------------------------------------------------------------------------ */
/* QJL 1-bit residual sketch ([MOQ] "QJL residual correction (sub-2-bit)";    */
/* [MLX] "Asymmetric K/V Compression": keys only; "RaBitQ vs QJL correction").*/
/* ------------------------------------------------------------------------ */

/* S (jl x d, row-major) with N(0,1) entries: SplitMix64 words taken in pairs give
 * u1 = ((w1 >> 11) + 1) 2^-53 in (0, 1] and u2 = (w2 >> 11) 2^-53 in [0, 1);
 * Box-Muller in binary64 gives sqrt(-2 ln u1) cos(2 pi u2) and
 * sqrt(-2 ln u1) sin(2 pi u2) for consecutive entries; each is rounded to
 * binary32. */
void tqo_qjl_matrix(int jl, int d, uint64_t seed, float *S) {
    uint64_t s = seed;
    const int n = jl * d;
    for (int i = 0; i < n; i += 2) {
        double u1 = (double)((sm64_next(&s) >> 11) + 1) * 0x1p-53;
        double u2 = (double)(sm64_next(&s) >> 11) * 0x1p-53;
        double rad = sqrt(-2.0 * log(u1));
        S[i] = (float)(rad * cos(2.0 * TQO_PI * u2));
        if (i + 1 < n) S[i + 1] = (float)(rad * sin(2.0 * TQO_PI * u2));
    }
}

/* Projection p = S r in binary64 (the sign decision's argument). */
void tqo_qjl_project(int jl, int d, const float *S, const float *r, double *p) {
    for (int j = 0; j < jl; j++) {
        double acc = 0.0;
        for (int i = 0; i < d; i++) acc += (double)S[(size_t)j * d + i] * (double)r[i];
        p[j] = acc;
    }
}

/* Sketch of the key residual r = y - yhat (binary32 subtraction): bit j of the
 * packed sign record is 1 iff (S r)_j >= 0 (a zero projection counts as +1);
 * rho = ||r||_2 (binary64, rounded to binary32). */
void tqo_qjl_sketch(int jl, int d, const float *S, const float *y, const float *yhat,
                    uint8_t *signs, float *rho) {
    float r[TQO_MAX_D];
    double p[TQO_MAX_D];
    double ss = 0.0;
    for (int i = 0; i < d; i++) {
        r[i] = y[i] - yhat[i];
        ss += (double)r[i] * (double)r[i];
    }
    tqo_qjl_project(jl, d, S, r, p);
    memset(signs, 0, (size_t)jl / 8);
    for (int j = 0; j < jl; j++)
        if (p[j] >= 0.0) signs[j >> 3] |= (uint8_t)(1u << (j & 7));
    *rho = (float)sqrt(ss);
}

/* ------------------------------------------------------------------------ */
/* Packed segment layout (one layer).                                          */
/*   record sizes rk(h) = d*kbits[h]/8, rv(h) = d*vbits[h]/8 bytes              */
/*   kcodes byte offset of (b, h, t): b*cap*sum_h rk + cap*sum_{h'<h} rk(h')      */
/*                                    + t*rk(h)       (vcodes likewise)         */
/*   kscale / vscale float index:     (b*H + h)*cap + t                          */
/*   QJL heads are ranked q(h) = #{h' < h : qjl[h']}, nq of them:               */
/*   qjl_signs byte offset ((b*nq + q(h))*cap + t) * jl/8, qjl_norm float index  */
/*   (b*nq + q(h))*cap + t.                                                      */
/*   fp16 segments: k16 / v16 element offset ((b*H + h)*cap + t)*d.              */
/* ------------------------------------------------------------------------ */
typedef struct {
    int kind;      /* 0 = packed, 1 = fp16 */
    int n_tokens;  /* valid tokens */
    int capacity;  /* layout capacity in tokens */
    const uint8_t *kbits, *vbits, *qjl; /* [H] */
    uint8_t *kcodes, *vcodes;
    float *kscale, *vscale;
    uint8_t *qjl_signs;
    float *qjl_norm;
    uint16_t *k16, *v16;
    int value_law; /* value codebook: 0 Gaussian, 1 sphere coordinate (tables [law * 9 + bits]) */
    /* QJL on values: heads with qjl_v[h] != 0 also sketch the value residual,
     * ranked v(h) = #{h' < h : qjl_v[h']}, nv of them, records at
     * vqjl_signs byte offset ((b*nv + v(h))*cap + t) * jl/8 and norms at
     * vqjl_norm index (b*nv + v(h))*cap + t (NULL qjl_v: none) */
    const uint8_t *qjl_v;
    uint8_t *vqjl_signs;
    float *vqjl_norm;
} tqo_segment;

static size_t off_codes(const uint8_t *bits, int H, int d, int cap, int b, int h, int t) {
    size_t all = 0, before = 0;
    for (int i = 0; i < H; i++) {
        size_t r = (size_t)d * bits[i] / 8;
        all += r;
        if (i < h) before += r;
    }
    return (size_t)b * cap * all + (size_t)cap * before + (size_t)t * ((size_t)d * bits[h] / 8);
}

static int qjl_rank(const uint8_t *qjl, int h) {
    int r = 0;
    for (int i = 0; i < h; i++) r += qjl[i] ? 1 : 0;
    return r;
}

static int vqjl_rank(const tqo_segment *seg, int h) {
    int r = 0;
    for (int i = 0; i < h; i++) r += seg->qjl_v && seg->qjl_v[i] ? 1 : 0;
    return r;
}

/* Compress T tokens of K and V (fp16 bit patterns, element strides sb, sh, st,
 * unit stride along d) into token positions [t_begin, t_begin + T) of a packed
 * segment.  thr[law * 9 + b] points at the 2^b - 1 binary32 value thresholds for
 * b bits of codebook law `law` (0 Gaussian, 1 sphere coordinate).
 * S is the QJL matrix (jl x d) or NULL when no head uses QJL.
 * Q: NULL for the SRHT of `sign`, else the dense rotation (d x d, y = Q x).
 * Value heads with qjl_v set sketch r = y - sigma*cent[code] (binary32 product
 * and difference, cent[law * 9 + b] the binary32 centroids) like the keys. */
void tqo_compress(int B, int H, int d, int T, const uint16_t *K, const uint16_t *V,
                  long long sb, long long sh, long long st, const int8_t *sign,
                  const float *const *thr, const float *S, int jl,
                  const tqo_segment *seg, int t_begin, const float *Q, const float *const *cent) {
    float x[TQO_MAX_D], y[TQO_MAX_D], yhat[TQO_MAX_D];
    uint8_t code[TQO_MAX_D];
    const int nq = qjl_rank(seg->qjl, H);
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++)
            for (int t = 0; t < T; t++) {
                const int pos = t_begin + t;
                const size_t src = (size_t)(b * sb + h * sh + t * st);
                const size_t sidx = ((size_t)b * H + h) * seg->capacity + pos;
                /* keys */
                const int kb = seg->kbits[h];
                for (int i = 0; i < d; i++) x[i] = (float)tqo_half_to_double(K[src + i]);
                if (Q) tqo_rotate_dense_f32(d, Q, x, y);
                else tqo_rotate_f32(d, sign, x, y);
                float m;
                tqo_quant_key(d, kb, y, code, &m);
                tqo_pack(d, kb, code, seg->kcodes + off_codes(seg->kbits, H, d, seg->capacity, b, h, pos));
                seg->kscale[sidx] = m;
                if (seg->qjl[h]) {
                    for (int i = 0; i < d; i++) yhat[i] = m * (float)tqo_key_level(kb, code[i]);
                    const size_t q = ((size_t)b * nq + qjl_rank(seg->qjl, h)) * seg->capacity + pos;
                    tqo_qjl_sketch(jl, d, S, y, yhat, seg->qjl_signs + q * (jl / 8), &seg->qjl_norm[q]);
                }
                /* values */
                const int vb = seg->vbits[h];
                for (int i = 0; i < d; i++) x[i] = (float)tqo_half_to_double(V[src + i]);
                if (Q) tqo_rotate_dense_f32(d, Q, x, y);
                else tqo_rotate_f32(d, sign, x, y);
                float sg;
                tqo_quant_value(d, vb, y, thr[seg->value_law * 9 + vb], code, &sg);
                tqo_pack(d, vb, code, seg->vcodes + off_codes(seg->vbits, H, d, seg->capacity, b, h, pos));
                seg->vscale[sidx] = sg;
                if (seg->qjl_v && seg->qjl_v[h]) {
                    const float *c = cent[seg->value_law * 9 + vb];
                    for (int i = 0; i < d; i++) yhat[i] = sg * c[code[i]];
                    int nv = 0;
                    for (int i = 0; i < H; i++) nv += seg->qjl_v[i] ? 1 : 0;
                    const size_t q = ((size_t)b * nv + vqjl_rank(seg, h)) * seg->capacity + pos;
                    tqo_qjl_sketch(jl, d, S, y, yhat, seg->vqjl_signs + q * (jl / 8), &seg->vqjl_norm[q]);
                }
            }
}

/* Dequantize token positions [t0, t0 + n) of one (b, h) of a packed segment into
 * the rotated space with the binary32 products the format defines:
 * keys m * level(code), values sigma * centroid[code] (cent[law * 9 + b] are binary32
 * centroids).  Outputs are [n][d] floats. */
void tqo_dequant(int H, int d, const tqo_segment *seg, int b, int h, int t0, int n,
                 const float *const *cent, float *khat, float *vhat) {
    uint8_t code[TQO_MAX_D];
    for (int t = 0; t < n; t++) {
        const int pos = t0 + t;
        const size_t sidx = ((size_t)b * H + h) * seg->capacity + pos;
        const int kb = seg->kbits[h], vb = seg->vbits[h];
        tqo_unpack(d, kb, seg->kcodes + off_codes(seg->kbits, H, d, seg->capacity, b, h, pos), code);
        for (int i = 0; i < d; i++) khat[(size_t)t * d + i] = seg->kscale[sidx] * (float)tqo_key_level(kb, code[i]);
        tqo_unpack(d, vb, seg->vcodes + off_codes(seg->vbits, H, d, seg->capacity, b, h, pos), code);
        for (int i = 0; i < d; i++)
            vhat[(size_t)t * d + i] = seg->vscale[sidx] * cent[seg->value_law * 9 + vb][code[i]];
    }
}

/* Tier demotion ("TurboMOQ", "Progressive temporal tiering": tokens move to
 * tiers with fewer bits as they age; "Attention-Weighted Demotion").  Reading:
 * the rotated-space reconstruction of a packed token (keys m*level(code),
 * values sigma*c[code], exactly as tqo_dequant) is compressed again with the
 * destination segment's widths by the same per-vector quantizers, in the
 * rotated space (no rotation either way).  Tokens [src_t0, src_t0 + n) of src
 * go to [dst_t0, dst_t0 + n) of dst; destination heads carry no QJL sketch. */
void tqo_requantize(int B, int H, int d, const tqo_segment *src, int src_t0, int n,
                    const float *const *cent, const float *const *thr, const tqo_segment *dst,
                    int dst_t0) {
    float kh[TQO_MAX_D], vh[TQO_MAX_D];
    uint8_t code[TQO_MAX_D];
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++)
            for (int t = 0; t < n; t++) {
                tqo_dequant(H, d, src, b, h, src_t0 + t, 1, cent, kh, vh);
                const int pos = dst_t0 + t;
                const size_t sidx = ((size_t)b * H + h) * dst->capacity + pos;
                const int kb = dst->kbits[h], vb = dst->vbits[h];
                float m, sg;
                tqo_quant_key(d, kb, kh, code, &m);
                tqo_pack(d, kb, code, dst->kcodes + off_codes(dst->kbits, H, d, dst->capacity, b, h, pos));
                dst->kscale[sidx] = m;
                tqo_quant_value(d, vb, vh, thr[dst->value_law * 9 + vb], code, &sg);
                tqo_pack(d, vb, code, dst->vcodes + off_codes(dst->vbits, H, d, dst->capacity, b, h, pos));
                dst->vscale[sidx] = sg;
            }
}

/* ------------------------------------------------------------------------ */
/* Decode attention over one layer's cache, in binary64.                       */
/*   packed tokens: khat = R (m*level(code) [+ rhat]), vhat = R (sigma*c[code]),  */
/*     rhat = sqrt(pi/2)/jl * rho * S^T s, s_j = +1 for a set sign bit else -1     */
/*     ([MOQ] "QJL residual correction": corrected = quantized + correction);   */
/*   fp16 tokens are used as stored;                                           */
/*   query head j reads KV head j / (Hq/H); scores q.k/sqrt(d); softmax; sum p v. */
/* q: fp16 bit patterns [B][Hq][d]; out: [B][Hq][d] binary64.  An empty cache     */
/* gives a zero output.                                                         */
/* ------------------------------------------------------------------------ */
/* Decode attention in binary64 over a layer's segments.
 *
 * QJL heads: estimator 0 adds the residual estimate sqrt(pi/2)/jl * rho * S^T s
 * to the key ("QJL residual correction (sub-2-bit)", the unbiased estimator);
 * estimator 1 adds instead, to the score, (pi/2)/jl * ||q'|| * rho *
 * <sign(S q'), s> with q' = R q (the sign-pair estimator of "RaBitQ vs QJL
 * correction": pi/2 times the two scales times the mean sign agreement; the
 * query's sign follows the key side's convention, sign(0) = +1).
 *
 * mass (may be NULL): for each (b, KV head h, token n of the segments taken in
 * order), the softmax weight of the token averaged over the g query heads that
 * read h, at mass[(b * H + h) * total + n] (total = the tokens of all segments).
 *
 * Q: NULL for the layer's SRHT (sign), else its dense rotation: packed keys and
 * values return to the original space as Q^T yhat.
 */
void tqo_decode_attention(int B, int H, int Hq, int d, int n_seg, const tqo_segment *segs,
                          const int8_t *sign, const float *const *cent, const float *S,
                          int jl, int estimator, const uint16_t *q, double *out, double *mass,
                          const float *Q) {
    const int g = Hq / H;
    int total = 0;
    for (int s = 0; s < n_seg; s++) total += segs[s].n_tokens;
    double *score = (double *)malloc(sizeof(double) * (total > 0 ? total : 1));
    double *vals = (double *)malloc(sizeof(double) * (size_t)(total > 0 ? total : 1) * d);
    double yk[TQO_MAX_D], yv[TQO_MAX_D], kh[TQO_MAX_D], qq[TQO_MAX_D], qr[TQO_MAX_D];
    double qsgn[1024];
    uint8_t code[TQO_MAX_D];
    if (mass)
        for (size_t i = 0; i < (size_t)B * H * total; i++) mass[i] = 0.0;
    for (int b = 0; b < B; b++)
        for (int j = 0; j < Hq; j++) {
            const int h = j / g;
            for (int i = 0; i < d; i++) qq[i] = tqo_half_to_double(q[((size_t)b * Hq + j) * d + i]);
            double qnorm = 0.0;
            if (estimator == 1 && S) {
                if (Q) tqo_rotate_dense_f64(d, Q, 0, qq, qr);
                else tqo_rotate_f64(d, sign, qq, qr);
                for (int i = 0; i < d; i++) qnorm += qr[i] * qr[i];
                qnorm = sqrt(qnorm);
                for (int jj = 0; jj < jl; jj++) {
                    double t = 0.0;
                    for (int i = 0; i < d; i++) t += (double)S[(size_t)jj * d + i] * qr[i];
                    qsgn[jj] = t >= 0.0 ? 1.0 : -1.0;
                }
            }
            int n = 0;
            for (int s = 0; s < n_seg; s++) {
                const tqo_segment *sg = &segs[s];
                const int nq = sg->kind == 0 ? qjl_rank(sg->qjl, H) : 0;
                for (int t = 0; t < sg->n_tokens; t++, n++) {
                    double *v = vals + (size_t)n * d;
                    double corr = 0.0;  /* sign-pair QJL term of the score */
                    if (sg->kind == 1) {
                        const size_t o = (((size_t)b * H + h) * sg->capacity + t) * d;
                        for (int i = 0; i < d; i++) {
                            kh[i] = tqo_half_to_double(sg->k16[o + i]);
                            v[i] = tqo_half_to_double(sg->v16[o + i]);
                        }
                    } else {
                        const size_t sidx = ((size_t)b * H + h) * sg->capacity + t;
                        const int kb = sg->kbits[h], vb = sg->vbits[h];
                        tqo_unpack(d, kb, sg->kcodes + off_codes(sg->kbits, H, d, sg->capacity, b, h, t), code);
                        for (int i = 0; i < d; i++) yk[i] = (double)sg->kscale[sidx] * tqo_key_level(kb, code[i]);
                        if (sg->qjl[h]) {
                            const size_t qi = ((size_t)b * nq + qjl_rank(sg->qjl, h)) * sg->capacity + t;
                            const uint8_t *sb = sg->qjl_signs + qi * (jl / 8);
                            const double rho = (double)sg->qjl_norm[qi];
                            for (int jj = 0; jj < jl; jj++) {
                                const double sj = ((sb[jj >> 3] >> (jj & 7)) & 1) ? 1.0 : -1.0;
                                if (estimator == 1) {
                                    corr += qsgn[jj] * sj;
                                } else {
                                    const double coef = sqrt(TQO_PI / 2.0) / jl * rho;
                                    for (int i = 0; i < d; i++) yk[i] += coef * sj * (double)S[(size_t)jj * d + i];
                                }
                            }
                            corr *= TQO_PI / 2.0 / jl * qnorm * rho;
                        }
                        if (Q) tqo_rotate_dense_f64(d, Q, 1, yk, kh);
                        else tqo_rotate_f64(d, sign, yk, kh);
                        tqo_unpack(d, vb, sg->vcodes + off_codes(sg->vbits, H, d, sg->capacity, b, h, t), code);
                        for (int i = 0; i < d; i++)
                            yv[i] = (double)sg->vscale[sidx] * (double)cent[sg->value_law * 9 + vb][code[i]];
                        if (sg->qjl_v && sg->qjl_v[h]) {  /* + sqrt(pi/2)/jl rho S^T s (the unbiased estimate of r) */
                            int nv = 0;
                            for (int i = 0; i < H; i++) nv += sg->qjl_v[i] ? 1 : 0;
                            const size_t qi = ((size_t)b * nv + vqjl_rank(sg, h)) * sg->capacity + t;
                            const uint8_t *sb = sg->vqjl_signs + qi * (jl / 8);
                            const double coef = sqrt(TQO_PI / 2.0) / jl * (double)sg->vqjl_norm[qi];
                            for (int jj = 0; jj < jl; jj++) {
                                const double sj = ((sb[jj >> 3] >> (jj & 7)) & 1) ? 1.0 : -1.0;
                                for (int i = 0; i < d; i++) yv[i] += coef * sj * (double)S[(size_t)jj * d + i];
                            }
                        }
                        if (Q) tqo_rotate_dense_f64(d, Q, 1, yv, v);
                        else tqo_rotate_f64(d, sign, yv, v);
                    }
                    double dot = 0.0;
                    for (int i = 0; i < d; i++) dot += qq[i] * kh[i];
                    dot += corr;
                    score[n] = dot / sqrt((double)d);
                }
            }
            double *o = out + ((size_t)b * Hq + j) * d;
            for (int i = 0; i < d; i++) o[i] = 0.0;
            if (total == 0) continue;
            double mx = score[0];
            for (int t = 1; t < total; t++) if (score[t] > mx) mx = score[t];
            double l = 0.0;
            for (int t = 0; t < total; t++) {
                score[t] = exp(score[t] - mx);
                l += score[t];
            }
            for (int t = 0; t < total; t++) {
                const double p = score[t] / l;
                for (int i = 0; i < d; i++) o[i] += p * vals[(size_t)t * d + i];
                if (mass) mass[((size_t)b * H + h) * total + t] += p / g;
            }
        }
    free(score);
    free(vals);
}
