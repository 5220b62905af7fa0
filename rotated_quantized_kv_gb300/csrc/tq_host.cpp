// tq_host.cpp -- host side of the C ABI declared in include/tq.h: argument
// checks, buffer layouts, the codebook fit, the QJL projection, the decode
// planner and the kernel launches.  No device memory is allocated here.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <atomic>
#include <limits>
#include <mutex>
#include <vector>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tq_internal.h"
#include "tq_mass.h"

using namespace tqk;

namespace {

thread_local int g_last_cuda = 0;
thread_local cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;
thread_local int g_last_launches_v = 0;
// polls of a split-K CTA's wait for its own copies (tq_set_decode_wait_polls)
std::atomic<int> g_wait_polls{1 << 20};
struct LaunchCounter {
    void store(int v) { g_last_launches_v = v; }
} g_last_launches;

tq_status cuda_fail(cudaError_t e) {
    g_last_cuda = static_cast<int>(e);
    return TQ_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// SplitMix64 (Steele, Lea, Flood, OOPSLA 2014).
struct SplitMix64 {
    uint64_t state;
    uint64_t next() {
        state += 0x9E3779B97F4A7C15ull;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    }
};

// n N(0,1) binary32 values: Box-Muller pairs on SplitMix64 words
void fill_gaussian(uint64_t seed, int n, float *S) {
    SplitMix64 g{seed};
    const double two_pi = 6.283185307179586476925;
    for (int i = 0; i < n; i += 2) {
        const double u1 = static_cast<double>((g.next() >> 11) + 1) * 0x1p-53;
        const double u2 = static_cast<double>(g.next() >> 11) * 0x1p-53;
        const double rad = std::sqrt(-2.0 * std::log(u1));
        S[i] = static_cast<float>(rad * std::cos(two_pi * u2));
        if (i + 1 < n) S[i + 1] = static_cast<float>(rad * std::sin(two_pi * u2));
    }
}

// ---------------------------------------------------------------- codebook fit
// Gaussian Lloyd-Max quantizer ("TurboMOQ", "Architecture": values go through a
// Lloyd-Max codebook), computed for N(0,1) in binary64.  The codebook is odd
// symmetric, so the upper half is iterated: cell k of the upper half is
// [b_k, b_{k+1}) with b at the midpoints of adjacent levels (b = 0 at the middle,
// +inf at the top); its conditional mean is (phi(b_k) - phi(b_{k+1})) / (Q(b_k) -
// Q(b_{k+1})) with Q the upper tail.  Start: the (k + 1/2)/n quantiles; stop
// when the largest move is at most 1e-13.
double upper_tail(double x) { return 0.5 * std::erfc(x * 0.70710678118654752440); }
double density(double x) { return 0.39894228040143267794 * std::exp(-0.5 * x * x); }

double tail_quantile(double p) {  // x with upper_tail(x) = p, by bisection
    double lo = -40.0, hi = 40.0;
    for (int i = 0; i < 200; ++i) {
        const double mid = 0.5 * (lo + hi);
        (upper_tail(mid) > p ? lo : hi) = mid;
    }
    return 0.5 * (lo + hi);
}

struct FittedCodebook {
    bool ready = false;
    std::vector<double> level, bound;  // full codebook, n levels and n-1 thresholds
};

std::mutex g_cb_mutex;
FittedCodebook g_cb[9];

std::mutex &g_cb_mutex_tables() {
    static std::mutex m;
    return m;
}

const FittedCodebook &fit(int bits) {
    std::lock_guard<std::mutex> lock(g_cb_mutex);
    FittedCodebook &cb = g_cb[bits];
    if (cb.ready) return cb;
    const int n = 1 << bits, half = n / 2;
    std::vector<double> up(half);  // levels half..n-1
    for (int k = 0; k < half; ++k) up[k] = tail_quantile(1.0 - (half + k + 0.5) / n);
    std::vector<double> edge(half + 1);
    for (int sweep = 0; sweep < 1000000; ++sweep) {
        edge[0] = 0.0;
        for (int k = 1; k < half; ++k) edge[k] = 0.5 * (up[k - 1] + up[k]);
        double move = 0.0;
        for (int k = 0; k < half; ++k) {
            const double a = edge[k];
            double num, den;
            if (k + 1 < half) {
                const double b = edge[k + 1];
                // phi(a) - phi(b) without cancellation for narrow cells
                num = -density(a) * std::expm1(-0.5 * (b - a) * (b + a));
                den = upper_tail(a) - upper_tail(b);
            } else {
                num = density(a);
                den = upper_tail(a);
            }
            const double v = num / den;
            move = std::fmax(move, std::fabs(v - up[k]));
            up[k] = v;
        }
        if (move <= 1e-13) break;
    }
    cb.level.assign(n, 0.0);
    for (int k = 0; k < half; ++k) {
        cb.level[half + k] = up[k];
        cb.level[half - 1 - k] = -up[k];
    }
    cb.bound.assign(n - 1, 0.0);
    for (int k = 0; k + 1 < n; ++k) cb.bound[k] = 0.5 * (cb.level[k] + cb.level[k + 1]);
    cb.bound[half - 1] = 0.0;
    cb.ready = true;
    return cb;
}

// ------------------------------------------- sphere-coordinate codebook
// The law of sqrt(d) times a coordinate of a uniform unit d-vector (what a
// rotated coordinate divided by its vector's RMS follows): density
// proportional to (1 - u^2/d)^((d-3)/2) on |u| < sqrt(d).  Lloyd's iteration
// as for the Gaussian law: first moments of a cell in closed form, cell masses
// by composite Gauss-Legendre quadrature in s = u / sqrt(d).
struct GaussRule {
    double x[24], w[24];
    GaussRule() {
        const int n = 24;
        for (int i = 0; i < n / 2; ++i) {
            double z = std::cos(3.14159265358979323846 * (i + 0.75) / (n + 0.5)), d = 1.0;
            for (int it = 0; it < 100; ++it) {
                double p = 1.0, q = 0.0;
                for (int j = 1; j <= n; ++j) {
                    const double r = q;
                    q = p;
                    p = ((2 * j - 1) * z * q - (j - 1) * r) / j;
                }
                d = n * (z * p - q) / (z * z - 1.0);
                const double step = p / d;
                z -= step;
                if (std::fabs(step) < 1e-16) break;
            }
            x[i] = z;
            x[n - 1 - i] = -z;
            w[i] = w[n - 1 - i] = 2.0 / ((1.0 - z * z) * d * d);
        }
    }
};

// mass of (1 - s^2)^e over [s0, s1] (0 <= s0 <= s1 <= 1) on `panels` panels
double sphere_cell_mass(double e, double s0, double s1, int panels) {
    static const GaussRule rule;
    const double h = (s1 - s0) / panels;
    double acc = 0.0;
    for (int p = 0; p < panels; ++p) {
        const double c = s0 + (p + 0.5) * h;
        for (int i = 0; i < 24; ++i) {
            const double s = c + 0.5 * h * rule.x[i];
            acc += rule.w[i] * std::exp(e * std::log1p(-s * s));
        }
    }
    return 0.5 * h * acc;
}

void fit_sphere(int bits, int d, FittedCodebook &cb) {
    const int n = 1 << bits, half = n / 2;
    const double e = 0.5 * (d - 3), sd = std::sqrt(static_cast<double>(d));
    const double half_mass = sphere_cell_mass(e, 0.0, 1.0, 256);
    std::vector<double> up(half);
    for (int k = 0; k < half; ++k) {  // start at the (k + 1/2)/n quantiles
        const double p = 1.0 - (half + k + 0.5) / n;
        double lo = 0.0, hi = 1.0;
        for (int it = 0; it < 80; ++it) {
            const double mid = 0.5 * (lo + hi);
            (sphere_cell_mass(e, mid, 1.0, 32) / (2.0 * half_mass) > p ? lo : hi) = mid;
        }
        up[k] = sd * 0.5 * (lo + hi);
    }
    std::vector<double> edge(half + 1);
    for (int sweep = 0; sweep < 1000000; ++sweep) {
        edge[0] = 0.0;
        for (int k = 1; k < half; ++k) edge[k] = 0.5 * (up[k - 1] + up[k]);
        double move = 0.0;
        for (int k = 0; k < half; ++k) {
            const double a = edge[k], la = std::log1p(-a * a / d);
            double num, b;
            if (k + 1 < half) {
                b = edge[k + 1];
                num = -std::exp((e + 1.0) * la) * std::expm1((e + 1.0) * (std::log1p(-b * b / d) - la));
            } else {
                b = sd;
                num = std::exp((e + 1.0) * la);
            }
            num *= 0.5 * d / (e + 1.0);
            const double den = sd * sphere_cell_mass(e, a / sd, b / sd, k + 1 < half ? 2 : 64);
            const double v = num / den;
            move = std::fmax(move, std::fabs(v - up[k]));
            up[k] = v;
        }
        if (move <= 1e-13) break;
    }
    cb.level.assign(n, 0.0);
    for (int k = 0; k < half; ++k) {
        cb.level[half + k] = up[k];
        cb.level[half - 1 - k] = -up[k];
    }
    cb.bound.assign(n - 1, 0.0);
    for (int k = 0; k + 1 < n; ++k) cb.bound[k] = 0.5 * (cb.level[k] + cb.level[k + 1]);
    cb.bound[half - 1] = 0.0;
    cb.ready = true;
}

FittedCodebook g_cb_sphere[9];  // d = kD

// The value codebook of a law: TQ_VALUE_LAW_GAUSS or TQ_VALUE_LAW_SPHERE (d = 128).
const FittedCodebook &fit(int bits, int law) {
    if (law == TQ_VALUE_LAW_GAUSS) return fit(bits);
    std::lock_guard<std::mutex> lock(g_cb_mutex);
    FittedCodebook &cb = g_cb_sphere[bits];
    if (!cb.ready) fit_sphere(bits, kD, cb);
    return cb;
}

void fill_thresholds(float *flat, const uint8_t *bits, int H, int law) {
    for (int h = 0; h < H; ++h) {
        const FittedCodebook &cb = fit(bits[h], law);
        for (int k = 0; k + 1 < (1 << bits[h]); ++k) flat[cb_off(bits[h]) + k] = static_cast<float>(cb.bound[k]);
    }
}

void fill_centroids(float *flat, const uint8_t *bits, int H, int law) {
    for (int h = 0; h < H; ++h) {
        const FittedCodebook &cb = fit(bits[h], law);
        for (int k = 0; k < (1 << bits[h]); ++k) flat[cb_off(bits[h]) + k] = static_cast<float>(cb.level[k]);
    }
}

// ---------------------------------------------------------------- layouts
tq_status check_layout(const tq_segment_layout *L, bool need_bits) {
    if (!L) return TQ_ERR_ARG;
    if (L->batch < 1 || L->n_heads < 1 || L->n_heads > TQ_MAX_HEADS || L->capacity < 0) return TQ_ERR_ARG;
    if (!pow2(L->head_dim) || L->head_dim < 16 || L->head_dim > TQ_MAX_HEAD_DIM) return TQ_ERR_ARG;
    if (need_bits) {
        bool any_qjl = false;
        for (int h = 0; h < L->n_heads; ++h) {
            if (L->kbits[h] < 1 || L->kbits[h] > 8 || L->vbits[h] < 1 || L->vbits[h] > 8) return TQ_ERR_ARG;
            if (L->qjl[h] > 1 || L->qjl_v[h] > 1) return TQ_ERR_ARG;
            any_qjl |= L->qjl[h] != 0 || L->qjl_v[h] != 0;
        }
        if (any_qjl && (L->jl_dim < 32 || L->jl_dim > 1024 || L->jl_dim % 32)) return TQ_ERR_ARG;
        if (L->value_law != TQ_VALUE_LAW_GAUSS && L->value_law != TQ_VALUE_LAW_SPHERE) return TQ_ERR_ARG;
    }
    return TQ_OK;
}

struct Offsets {
    uint32_t kblock = 0, vblock = 0;
    uint32_t koff[TQ_MAX_HEADS] = {}, voff[TQ_MAX_HEADS] = {};
    int8_t qrank[TQ_MAX_HEADS] = {};
    int nq = 0;
    int8_t vrank[TQ_MAX_HEADS] = {};  // value sketches
    int nv = 0;
};

Offsets offsets(const tq_segment_layout *L) {
    Offsets o;
    size_t k = 0, v = 0;
    for (int h = 0; h < L->n_heads; ++h) {
        o.koff[h] = static_cast<uint32_t>(k);
        o.voff[h] = static_cast<uint32_t>(v);
        k += static_cast<size_t>(L->capacity) * L->head_dim * L->kbits[h] / 8;
        v += static_cast<size_t>(L->capacity) * L->head_dim * L->vbits[h] / 8;
        o.qrank[h] = L->qjl[h] ? static_cast<int8_t>(o.nq++) : static_cast<int8_t>(-1);
        o.vrank[h] = L->qjl_v[h] ? static_cast<int8_t>(o.nv++) : static_cast<int8_t>(-1);
    }
    o.kblock = static_cast<uint32_t>(k);
    o.vblock = static_cast<uint32_t>(v);
    return o;
}

bool fits_u32(const tq_segment_layout *L) {
    size_t k = 0, v = 0;
    for (int h = 0; h < L->n_heads; ++h) {
        k += static_cast<size_t>(L->capacity) * L->head_dim * L->kbits[h] / 8;
        v += static_cast<size_t>(L->capacity) * L->head_dim * L->vbits[h] / 8;
    }
    return k < (1ull << 32) && v < (1ull << 32);
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

float inv_sqrt_f32(int d) { return static_cast<float>(1.0 / std::sqrt(static_cast<double>(d))); }

// Bucket table of a value width <= 3 (RowsParams::bucket): bucket i holds the
// bit patterns [i << 22, (i + 1) << 22), i.e. sign, exponent and one mantissa
// bit of the quotient u; k = the thresholds below every u of the bucket, t = the
// one threshold inside it (+inf if none).  False if a bucket holds two.
bool value_buckets(const float *thr, int nt, RowsParams::Bucket *out) {
    auto as_float = [](uint32_t b) {
        float f;
        std::memcpy(&f, &b, 4);
        return f;
    };
    const float inf = std::numeric_limits<float>::infinity();
    uint32_t inf_bits;
    std::memcpy(&inf_bits, &inf, 4);
    for (int i = 0; i < kRowsBuckets; ++i) {
        const uint32_t m = static_cast<uint32_t>(i & 511);
        if (m >= 510) {  // exponent 255: infinities and NaNs, never a quotient of finite inputs
            out[i].t = inf_bits;
            out[i].k = i < 512 ? static_cast<uint32_t>(nt) : 0u;
            continue;
        }
        const float lo = as_float(m << 22);                                   // magnitude range [lo, hi)
        const float hi = (m + 1) << 22 >= 0x7F800000u ? inf : as_float((m + 1) << 22);
        int k = 0, inside = 0;
        float t_c = inf;
        for (int j = 0; j < nt; ++j) {
            const float t = thr[j];
            if (i < 512) {  // u in [lo, hi)
                if (t < lo) ++k;
                else if (t < hi) { ++inside; t_c = t; }
            } else {  // u in (-hi, -lo]
                if (t <= -hi) ++k;
                else if (t <= -lo) { ++inside; t_c = t; }
            }
        }
        if (inside > 1) return false;
        uint32_t tb;
        std::memcpy(&tb, &t_c, 4);
        out[i].t = tb;
        out[i].k = static_cast<uint32_t>(k);
    }
    return true;
}

// The 4-bit table of compress_rows_kernel (RowsParams::bucket4): buckets of
// the 11 top bits of u, each holding at most one threshold; false if some
// bucket holds two (the kernel then searches the thresholds).
bool value_buckets4(const float *thr, int nt, uint32_t *out) {
    auto as_float = [](uint32_t b) {
        float f;
        std::memcpy(&f, &b, 4);
        return f;
    };
    constexpr uint32_t kLow = (1u << 21) - 1u;
    const float inf = std::numeric_limits<float>::infinity();
    for (int i = 0; i < 2 * kRowsBuckets; ++i) {
        const uint32_t m = static_cast<uint32_t>(i & 1023);
        const bool neg = i >= 1024;
        if (m >= 1020) {  // exponent 255: infinities and NaNs, never a quotient of finite inputs
            out[i] = (static_cast<uint32_t>(neg ? 0 : nt) << 21) | kLow;
            continue;
        }
        const float lo = as_float(m << 21);  // magnitude range [lo, hi)
        const float hi = (m + 1) << 21 >= 0x7F800000u ? inf : as_float((m + 1) << 21);
        int k = 0, inside = 0;
        uint32_t tl = kLow;  // no threshold: [t' < x] never holds
        for (int j = 0; j < nt; ++j) {
            const float t = thr[j];
            bool in;
            if (!neg) {  // u in [lo, hi)
                in = !(t < lo) && t < hi;
                if (t < lo) ++k;
            } else {  // u in (-hi, -lo]
                in = !(t <= -hi) && t <= -lo;
                if (t <= -hi) ++k;
            }
            if (in) {
                // t shares u's top 11 bits, or t = +-0 at lo = 0, whose low bits
                // (0) give [t < u] all the same
                uint32_t tb;
                std::memcpy(&tb, &t, 4);
                tl = (tb & kLow) ^ (neg ? kLow : 0u);
                ++inside;
            }
        }
        if (inside > 1) return false;
        out[i] = (static_cast<uint32_t>(k) << 21) | tl;
    }
    return true;
}

// Launches of the one-thread-per-slice kernels for the heads c.sel[0..n_sel)
// (none of them sketched) at head_dim d = 128, 256 or 512 (sign_bits: the
// rotation's d bits; c supplies the pointers, strides and widths): the keys of
// each distinct key width, then the values of each distinct value width (one
// launch each; uniform layouts take two).  Returns cudaErrorNotSupported,
// before launching anything, if a value width's bucket table does not separate
// its thresholds (the caller then takes another kernel).
cudaError_t launch_rows(const CompressParams &c, const tq_segment_layout *layout, const uint32_t *sign_bits, int d,
                        cudaStream_t s) {
    // head_dim 64: token pairs starting at even positions (whole 16-byte stores)
    if (d != kD && d != 2 * kD && d != 4 * kD && !(d == kD / 2 && c.t_begin % 2 == 0)) return cudaErrorNotSupported;
    bool in_sel[kMaxH] = {};
    for (int i = 0; i < c.n_sel; ++i) in_sel[c.sel[i]] = true;
    for (int h = 0; h < c.H; ++h) {
        if (!in_sel[h] || c.vbits[h] > 3) continue;
        const FittedCodebook &cb = fit(c.vbits[h], layout->value_law);
        float thr[7];
        for (int k = 0; k + 1 < (1 << c.vbits[h]); ++k) thr[k] = static_cast<float>(cb.bound[k]);
        static thread_local RowsParams::Bucket scratch[kRowsBuckets];
        if (!value_buckets(thr, (1 << c.vbits[h]) - 1, scratch)) return cudaErrorNotSupported;
    }
    RowsParams p;
    std::memset(&p, 0, sizeof(p));
    p.sb = c.sb;
    p.sh = c.sh;
    p.st = c.st;
    p.B = c.B;
    p.H = c.H;
    p.T = c.T;
    p.t_begin = c.t_begin;
    p.capacity = c.capacity;
    p.nh = d >= kD ? d / kD : 1;
    p.np = d >= kD ? 1 : kD / d;  // head_dim 64: two tokens per thread, the same signs for both
    const float c_d = inv_sqrt_f32(d);
    for (int i = 0; i < p.nh * kD / 2; ++i) {
        const int j = i % (d / 2);
        const uint32_t s0 = (sign_bits[(2 * j) >> 5] >> ((2 * j) & 31)) & 1u;
        const uint32_t s1 = (sign_bits[(2 * j + 1) >> 5] >> ((2 * j + 1) & 31)) & 1u;
        p.in_mask[i] = (s0 << 15) | (s1 << 31);
    }
    for (int i = 0; i < p.nh * kD; ++i) {
        const int j = i % d;
        p.out_scale[i] = ((sign_bits[j >> 5] >> (j & 31)) & 1u) ? -c_d : c_d;
    }
    for (int values = 0; values < 2; ++values) {
        p.X = values ? c.V : c.K;
        p.codes = values ? c.vcodes : c.kcodes;
        p.scale = values ? c.vscale : c.kscale;
        p.block = values ? c.vblock : c.kblock;
        for (int h = 0; h < c.H; ++h) p.off[h] = values ? c.voff[h] : c.koff[h];
        for (int bits = 1; bits <= 8; ++bits) {
            p.n_heads = 0;
            for (int h = 0; h < c.H; ++h)
                if (in_sel[h] && (values ? c.vbits[h] : c.kbits[h]) == bits) p.head[p.n_heads++] = static_cast<uint8_t>(h);
            if (p.n_heads == 0) continue;
            if (values) {
                const FittedCodebook &cb = fit(bits, layout->value_law);
                for (int k = 0; k + 1 < (1 << bits); ++k) p.thr[k] = static_cast<float>(cb.bound[k]);
                if (bits <= 3 && !value_buckets(p.thr, (1 << bits) - 1, p.bucket)) return cudaErrorNotSupported;
                p.bucket4_ok = bits == 4 && value_buckets4(p.thr, 15, p.bucket4) ? 1 : 0;
            }
            const cudaError_t e = launch_compress_rows(p, bits, values != 0, s);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

// ---------------------------------------------------------------- other head dims
// Compression for head dimensions other than kD (tq_generic.cu): SRHT only,
// no QJL sketches, Gaussian value codebook.
tq_status compress_other_dims(const tq_segment_layout *layout, const tq_rotation *rot, const Offsets &o,
                              const void *K, const void *V, int n_tokens, int64_t stride_b, int64_t stride_h,
                              int64_t stride_t, int t_begin, const tq_packed_bufs *out, cudaStream_t s) {
    const int d = layout->head_dim;
    if (o.nq || o.nv || rot->dense || layout->value_law != TQ_VALUE_LAW_GAUSS) return TQ_ERR_UNSUPPORTED;
    if (!aligned16(K) || !aligned16(V) || !aligned16(out->kcodes) || !aligned16(out->vcodes) ||
        !aligned16(out->kscale) || !aligned16(out->vscale))
        return TQ_ERR_ALIGN;
    if (stride_t < d || stride_h < 0 || stride_b < 0 || (stride_t % 8) || (stride_h % 8) || (stride_b % 8))
        return TQ_ERR_ALIGN;
    if (n_tokens == 0) return TQ_OK;
    if (d == kD / 2 || d == 2 * kD || d == 4 * kD) {  // one thread per 128-dim slice (or per token pair)
        CompressParams c;
        std::memset(&c, 0, sizeof(c));
        c.K = static_cast<const uint16_t *>(K);
        c.V = static_cast<const uint16_t *>(V);
        c.sb = stride_b;
        c.sh = stride_h;
        c.st = stride_t;
        c.B = layout->batch;
        c.H = layout->n_heads;
        c.T = n_tokens;
        c.t_begin = t_begin;
        c.capacity = layout->capacity;
        c.kcodes = static_cast<uint8_t *>(out->kcodes);
        c.vcodes = static_cast<uint8_t *>(out->vcodes);
        c.kscale = out->kscale;
        c.vscale = out->vscale;
        c.kblock = o.kblock;
        c.vblock = o.vblock;
        for (int h = 0; h < c.H; ++h) {
            c.koff[h] = o.koff[h];
            c.voff[h] = o.voff[h];
            c.kbits[h] = layout->kbits[h];
            c.vbits[h] = layout->vbits[h];
            c.sel[c.n_sel++] = static_cast<uint8_t>(h);
        }
        const cudaError_t e = launch_rows(c, layout, rot->sign_bits, d, s);
        if (e != cudaErrorNotSupported) return e == cudaSuccess ? TQ_OK : cuda_fail(e);
    }
    GenCompressParams p;
    std::memset(&p, 0, sizeof(p));
    p.K = static_cast<const uint16_t *>(K);
    p.V = static_cast<const uint16_t *>(V);
    p.sb = stride_b;
    p.sh = stride_h;
    p.st = stride_t;
    p.B = layout->batch;
    p.H = layout->n_heads;
    p.T = n_tokens;
    p.t_begin = t_begin;
    p.capacity = layout->capacity;
    p.kcodes = static_cast<uint8_t *>(out->kcodes);
    p.vcodes = static_cast<uint8_t *>(out->vcodes);
    p.kscale = out->kscale;
    p.vscale = out->vscale;
    p.kblock = o.kblock;
    p.vblock = o.vblock;
    for (int h = 0; h < p.H; ++h) {
        p.koff[h] = o.koff[h];
        p.voff[h] = o.voff[h];
        p.kbits[h] = layout->kbits[h];
        p.vbits[h] = layout->vbits[h];
    }
    std::memcpy(p.sign_bits, rot->sign_bits, sizeof(p.sign_bits));
    p.inv_sqrt_d = inv_sqrt_f32(d);
    fill_thresholds(p.thr, layout->vbits, p.H, layout->value_law);
    const cudaError_t e = launch_gen_compress(p, d, s);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status dequantize_other_dims(const tq_segment_layout *layout, const tq_packed_bufs *bufs, const tq_rotation *rot,
                                const Offsets &o, int t_begin, int n_tokens, float *k_rot, float *v_rot,
                                float *k_orig, float *v_orig, cudaStream_t s) {
    if (rot && rot->dense) return TQ_ERR_UNSUPPORTED;
    if (layout->value_law != TQ_VALUE_LAW_GAUSS) return TQ_ERR_UNSUPPORTED;
    GenDequantParams p;
    std::memset(&p, 0, sizeof(p));
    p.B = layout->batch;
    p.H = layout->n_heads;
    p.t_begin = t_begin;
    p.n = n_tokens;
    p.capacity = layout->capacity;
    p.kcodes = static_cast<const uint8_t *>(bufs->kcodes);
    p.vcodes = static_cast<const uint8_t *>(bufs->vcodes);
    p.kscale = bufs->kscale;
    p.vscale = bufs->vscale;
    p.kblock = o.kblock;
    p.vblock = o.vblock;
    for (int h = 0; h < p.H; ++h) {
        p.koff[h] = o.koff[h];
        p.voff[h] = o.voff[h];
        p.kbits[h] = layout->kbits[h];
        p.vbits[h] = layout->vbits[h];
    }
    if (rot) std::memcpy(p.sign_bits, rot->sign_bits, sizeof(p.sign_bits));
    p.inv_sqrt_d = inv_sqrt_f32(layout->head_dim);
    p.k_rot = k_rot;
    p.v_rot = v_rot;
    p.k_orig = k_orig;
    p.v_orig = v_orig;
    fill_centroids(p.centroid, layout->vbits, p.H, layout->value_law);
    const cudaError_t e = launch_gen_dequant(p, layout->head_dim, s);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- decode plan
struct Plan {
    std::vector<WorkItem> items;      // sorted by class; fp16 items last
    std::vector<LayerPlan> layer;
    std::vector<ClassLaunch> classes;
    DecodeDims dims{};
    bool any_qjl = false;
    int n_parts = 0;
    int mass_ctas = 0;  // CTAs of the attention-mass launch (0: no segment asked for mass)
    int vqjl_ctas = 0;  // CTAs of the value-sketch launch (0: no value sketch)
    int mass_stage = 0, vqjl_stage = 0;  // bytes of one step buffer of each rescoring launch
    // work item of every CTA: the class launches' tables (ClassLaunch::cta_off),
    // then the attention-mass launch's (mass_cta_off), then the value-sketch one's
    std::vector<int> cta_item;
    int mass_cta_off = 0, vqjl_cta_off = 0;
    std::vector<int> grp_part, grp_nparts, lbh_total;
    size_t off_items = 0, off_layer = 0, off_grp_part = 0, off_grp_nparts = 0, off_lbh_total = 0, off_counter = 0;
    size_t off_cta_item = 0;
    size_t off_qrot = 0, off_qjlt = 0, off_qsum = 0, off_part = 0, off_ml = 0, off_z = 0, total = 0;
    // head dimensions other than kD: one CTA per (layer, batch, KV head) over
    // the layer's items, the rotations' sign bits per layer
    bool generic = false;
    std::vector<uint32_t> signs;
    size_t off_signs = 0;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The persistent CTA (of G sharing S stages in equal contiguous ranges
// [i S / G, (i+1) S / G)) that holds stage s; same arithmetic as the kernels.
long long dec_cta_of_stage(long long s, long long S, long long G) { return ((s + 1) * G + S - 1) / S - 1; }
// first stage of CTA i of a packed launch (the kernels' range_begin)
long long dec_range_begin(long long i, long long S, long long G) { return i * S / G; }

// Decode class of an item: one kernel instantiation and one value table each
// (fp16 items form one class after all packed ones).
constexpr int kFp16ClassKey = 1100;
int class_key(const WorkItem &w) {
    return w.kind == TQ_SEG_FP16 ? kFp16ClassKey : ((w.kb * 16 + w.vb) * 2 + w.qjl) * 2 + w.vlaw;
}

// Validate the views and lay out the work: one item per (layer, segment, KV
// head) with tokens, split into chunks of `chunk` tokens (a multiple of 64)
// sized so that each CTA reads a few hundred KB at most while the whole call
// still spans many CTAs per SM.
tq_status build_plan(const tq_layer_view *layers, int n_layers, int B, int H, int Hq, int d,
                     const float *S, int jl, Plan &P, bool check_ptrs) {
    if (!layers || n_layers < 1 || B < 1 || H < 1 || H > TQ_MAX_HEADS || Hq < H || Hq % H) return TQ_ERR_ARG;
    if (!pow2(d) || d < 16 || d > TQ_MAX_HEAD_DIM) return TQ_ERR_ARG;
    const int gqa = Hq / H;
    // head_dim 256 and 512 with GQA 1, 2 or 4 run the split-K kernels on 128-dim
    // sub-records, head_dim 64 on token pairs read as 128-dim records; other
    // head dims the generic kernel (GQA up to 4); none of them takes QJL
    // sketches, dense rotations or attention-mass outputs
    const bool mma_gqa = gqa == 1 || gqa == 2 || gqa == 4;
    const bool wide = (d == 2 * kD || d == 4 * kD) && mma_gqa;
    const bool narrow = d == kD / 2 && mma_gqa;
    const bool generic = d != kD && !wide && !narrow;
    const bool other_dim = d != kD;
    if (!generic && !mma_gqa) return TQ_ERR_UNSUPPORTED;
    if (generic && gqa > kMaxGqa) return TQ_ERR_UNSUPPORTED;
    const int nh = wide ? d / kD : 1;
    const int np = narrow ? 2 : 1;
    for (int l = 0; l < n_layers; ++l) {
        const tq_layer_view &lv = layers[l];
        if (lv.n_segments < 0 || lv.n_segments > TQ_MAX_SEGMENTS || lv.rot.head_dim != d) return TQ_ERR_ARG;
        if (lv.qjl_estimator != TQ_QJL_UNBIASED && lv.qjl_estimator != TQ_QJL_SIGN_PAIR) return TQ_ERR_ARG;
        if (check_ptrs && lv.rot.dense && !aligned16(lv.rot.dense)) return TQ_ERR_ALIGN;
        if (other_dim && lv.rot.dense) return TQ_ERR_UNSUPPORTED;
        for (int s = 0; s < lv.n_segments; ++s) {
            const tq_segment &sg = lv.seg[s];
            const tq_segment_layout &L = sg.layout;
            if (sg.kind != TQ_SEG_PACKED && sg.kind != TQ_SEG_FP16) return TQ_ERR_ARG;
            if (check_ptrs && sg.attn_mass && !aligned16(sg.attn_mass)) return TQ_ERR_ALIGN;
            tq_status st = check_layout(&L, sg.kind == TQ_SEG_PACKED);
            if (st != TQ_OK) return st;
            if (L.batch != B || L.n_heads != H || L.head_dim != d) return TQ_ERR_ARG;
            if (sg.n_tokens < 0 || sg.n_tokens > L.capacity) return TQ_ERR_SIZE;
            if (other_dim && sg.attn_mass) return TQ_ERR_UNSUPPORTED;
            if (sg.kind == TQ_SEG_PACKED) {
                if (L.capacity % 16) return TQ_ERR_ALIGN;
                if (!fits_u32(&L)) return TQ_ERR_UNSUPPORTED;
                bool q = false, qv = false;
                for (int h = 0; h < H; ++h) {
                    q |= L.qjl[h] != 0;
                    qv |= L.qjl_v[h] != 0;
                }
                if (check_ptrs) {
                    const tq_packed_bufs &pb = sg.packed;
                    if (!pb.kcodes || !pb.vcodes || !pb.kscale || !pb.vscale) return TQ_ERR_ARG;
                    if (!aligned16(pb.kcodes) || !aligned16(pb.vcodes) || !aligned16(pb.kscale) ||
                        !aligned16(pb.vscale))
                        return TQ_ERR_ALIGN;
                    if (q) {
                        if (!pb.qjl_signs || !pb.qjl_norm || !S) return TQ_ERR_ARG;
                        if (!aligned16(pb.qjl_signs) || !aligned16(pb.qjl_norm) || !aligned16(S)) return TQ_ERR_ALIGN;
                    }
                    if (qv) {
                        if (!pb.vqjl_signs || !pb.vqjl_norm || !S) return TQ_ERR_ARG;
                        if (!aligned16(pb.vqjl_signs) || !aligned16(pb.vqjl_norm) || !aligned16(S)) return TQ_ERR_ALIGN;
                    }
                }
                if ((q || qv) && (jl != kJl || L.jl_dim != kJl)) return TQ_ERR_UNSUPPORTED;
                if (other_dim && (q || qv || L.value_law != TQ_VALUE_LAW_GAUSS)) return TQ_ERR_UNSUPPORTED;
            } else {
                if (check_ptrs) {
                    if (!sg.k16 || !sg.v16) return TQ_ERR_ARG;
                    if (!aligned16(sg.k16) || !aligned16(sg.v16)) return TQ_ERR_ALIGN;
                }
            }
        }
    }
    P = Plan();
    P.layer.assign(n_layers, LayerPlan{});
    bool any_dense = false;
    {
        size_t n = 0;
        for (int l = 0; l < n_layers; ++l) n += static_cast<size_t>(layers[l].n_segments) * H;
        P.items.reserve(n);
    }
    for (int l = 0; l < n_layers; ++l) {
        const tq_layer_view &lv = layers[l];
        LayerPlan &lp = P.layer[l];
        std::memcpy(lp.sign_bits, lv.rot.sign_bits, sizeof(lp.sign_bits));
        lp.qjl_mode = lv.qjl_estimator;
        lp.dense = lv.rot.dense;
        any_dense |= lv.rot.dense != nullptr;
        for (int s = 0; s < lv.n_segments; ++s) {
            const tq_segment &sg = lv.seg[s];
            if (sg.n_tokens == 0) continue;
            const tq_segment_layout &L = sg.layout;
            const size_t cap = static_cast<size_t>(L.capacity);
            const Offsets o = offsets(&L);
            for (int h = 0; h < H; ++h) {
                WorkItem w;
                std::memset(&w, 0, sizeof(w));
                w.kind = sg.kind;
                w.layer = l;
                w.head = h;
                w.n_tokens = sg.n_tokens;
                w.mass = sg.attn_mass ? sg.attn_mass + h * cap : nullptr;
                w.sstride = static_cast<uint32_t>(H * cap);
                if (sg.kind == TQ_SEG_PACKED) {
                    w.kc = static_cast<const uint8_t *>(sg.packed.kcodes) + o.koff[h];
                    w.vc = static_cast<const uint8_t *>(sg.packed.vcodes) + o.voff[h];
                    w.ks = sg.packed.kscale + h * cap;
                    w.vs = sg.packed.vscale + h * cap;
                    w.kstride = o.kblock;
                    w.vstride = o.vblock;
                    w.kb = L.kbits[h];
                    w.vb = L.vbits[h];
                    w.qjl = L.qjl[h] ? 1 : 0;
                    w.vlaw = L.value_law;
                    if (L.qjl_v[h]) {
                        w.vqs = static_cast<const uint8_t *>(sg.packed.vqjl_signs) + o.vrank[h] * cap * (kJl / 8);
                        w.vqn = sg.packed.vqjl_norm + o.vrank[h] * cap;
                        w.vqstride = static_cast<uint32_t>(o.nv * cap);
                        lp.has_vqjl = 1;
                    }
                    if (w.qjl) {
                        w.qs = static_cast<const uint8_t *>(sg.packed.qjl_signs) + o.qrank[h] * cap * (kJl / 8);
                        w.qn = sg.packed.qjl_norm + o.qrank[h] * cap;
                        w.qstride = static_cast<uint32_t>(o.nq * cap);
                        P.any_qjl = true;
                        lp.has_qjl = 1;
                    }
                } else {
                    const size_t row = cap * d * 2;  // bytes of one (b, h) block
                    w.kc = static_cast<const uint8_t *>(sg.k16) + h * row;
                    w.vc = static_cast<const uint8_t *>(sg.v16) + h * row;
                    w.kstride = w.vstride = H * row;
                    w.kb = w.vb = 16;
                }
                // fp16 segments: one CTA per 64-token chunk (packed segments
                // ignore the chunk: their persistent CTAs split the stages)
                w.chunk = kStageTokens;
                w.n_chunks = (sg.n_tokens + w.chunk - 1) / w.chunk;
                P.items.push_back(w);
            }
        }
    }
    if (generic) {  // each (layer, KV head)'s items, the sign bits, the offsets
        P.generic = true;
        for (size_t i = 0; i < P.items.size(); ++i) {
            LayerPlan &lp = P.layer[P.items[i].layer];
            lp.item[P.items[i].head][lp.n_items[P.items[i].head]++] = static_cast<int>(i);
        }
        P.signs.assign(static_cast<size_t>(n_layers) * (kMaxD / 32), 0u);
        for (int l = 0; l < n_layers; ++l)
            std::memcpy(P.signs.data() + static_cast<size_t>(l) * (kMaxD / 32), layers[l].rot.sign_bits,
                        sizeof(uint32_t) * (kMaxD / 32));
        DecodeDims &D = P.dims;
        D.L = n_layers;
        D.B = B;
        D.H = H;
        D.Hq = Hq;
        D.gqa = gqa;
        D.inv_sqrt_d = inv_sqrt_f32(d);
        D.qk_scale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
        P.off_items = 256;
        size_t off = P.off_items + align256(sizeof(WorkItem) * std::max<size_t>(P.items.size(), 1));
        P.off_layer = off;
        off += align256(sizeof(LayerPlan) * n_layers);
        P.off_signs = off;
        off += align256(sizeof(uint32_t) * P.signs.size());
        P.off_qrot = off;  // the uploaded plan ends here
        P.total = off;
        return TQ_OK;
    }
    {  // stable bucket sort by class (at most 2 * 8 * 8 packed classes, fp16 last)
        std::vector<int> key(P.items.size());
        int nkeys = 0;
        int slot_of[kFp16ClassKey + 1];
        std::fill(std::begin(slot_of), std::end(slot_of), -1);
        int keys[kFp16ClassKey + 1];
        for (size_t i = 0; i < P.items.size(); ++i) {
            const int k = class_key(P.items[i]);
            if (slot_of[k] < 0) {
                slot_of[k] = 0;
                keys[nkeys++] = k;
            }
            key[i] = k;
        }
        std::sort(keys, keys + nkeys);
        std::vector<int> start(nkeys + 1, 0);
        for (int j = 0; j < nkeys; ++j) slot_of[keys[j]] = j;
        for (size_t i = 0; i < P.items.size(); ++i) start[slot_of[key[i]] + 1]++;
        for (int j = 0; j < nkeys; ++j) start[j + 1] += start[j];
        std::vector<WorkItem> sorted(P.items.size());
        for (size_t i = 0; i < P.items.size(); ++i) sorted[start[slot_of[key[i]]]++] = P.items[i];
        P.items.swap(sorted);
    }
    // classes: packed ones run persistent CTAs over their 128-token stages,
    // fp16 runs one CTA per (item, batch element, chunk)
    const int sms = sm_count();
    long long cta = 0, stages = 0;
    for (size_t i = 0; i < P.items.size(); ++i) {
        WorkItem &w = P.items[i];
        if (i == 0 || class_key(w) != class_key(P.items[i - 1])) {
            P.classes.push_back(ClassLaunch{w.kb, w.vb, w.qjl, w.vlaw, static_cast<int>(i), static_cast<int>(i), 0, 0});
            cta = 0;
            stages = 0;
        }
        ClassLaunch &c = P.classes.back();
        c.item_hi = static_cast<int>(i) + 1;
        if (w.kind == TQ_SEG_PACKED) {
            const int pt = packed_stage_tokens(w.kb, w.vb, w.qjl != 0, nh, np);
            w.n_stages = (w.n_tokens + pt - 1) / pt;
            w.stage_begin = stages;
            stages += static_cast<long long>(B) * w.n_stages;
            c.n_stages = stages;
            c.n_ctas = static_cast<int>(std::min<long long>(
                stages, static_cast<long long>(sms) * packed_ctas_per_sm(w.kb, w.vb, w.qjl != 0, nh, np)));
        } else {
            w.cta_begin = static_cast<int>(cta);
            cta += static_cast<long long>(B) * w.n_chunks;
            if (cta > 0x7fffffffLL) return TQ_ERR_UNSUPPORTED;
            c.n_ctas = static_cast<int>(cta);
        }
    }
    // partial records: one per (group, CTA touching it); per (layer, batch, KV
    // head) the total the fused combine waits for
    P.grp_part.assign(P.items.size() * B, 0);
    P.grp_nparts.assign(P.items.size() * B, 0);
    P.lbh_total.assign(static_cast<size_t>(n_layers) * B * H, 0);
    long long part = 0;
    int ci = 0;
    for (size_t i = 0; i < P.items.size(); ++i) {
        WorkItem &w = P.items[i];
        while (static_cast<int>(i) >= P.classes[ci].item_hi) ++ci;
        const ClassLaunch &c = P.classes[ci];
        for (int b = 0; b < B; ++b) {
            int np, portions;
            if (w.kind == TQ_SEG_PACKED) {
                // CTAs touching the group; each writes one record per warp
                const long long gs = w.stage_begin + static_cast<long long>(b) * w.n_stages;
                portions = static_cast<int>(dec_cta_of_stage(gs + w.n_stages - 1, c.n_stages, c.n_ctas) -
                                            dec_cta_of_stage(gs, c.n_stages, c.n_ctas) + 1);
                np = kDecodeWarps * portions;
            } else {
                portions = w.n_chunks;  // one CTA-merged record per chunk and 128-dim block
                np = w.n_chunks * nh;
            }
            P.grp_part[i * B + b] = static_cast<int>(part);
            P.grp_nparts[i * B + b] = np;
            P.lbh_total[(static_cast<size_t>(w.layer) * B + b) * H + w.head] += portions;
            part += np;
        }
        if (part > 0x7fffffffLL) return TQ_ERR_UNSUPPORTED;
        LayerPlan &lp = P.layer[w.layer];
        lp.item[w.head][lp.n_items[w.head]++] = static_cast<int>(i);
    }
    P.n_parts = static_cast<int>(part);
    // attention mass: one CTA per (item with a mass buffer, batch element,
    // kMassTokens tokens); items without one start where the next one does
    {
        long long mc = 0;
        int mkb = 1, vkb = 1;
        bool mq = false, vq = false;
        for (WorkItem &w : P.items) {
            w.mass_cta_begin = static_cast<int>(mc);
            if (w.mass) mc += static_cast<long long>(B) * ((w.n_tokens + kMassTokens - 1) / kMassTokens);
            if (mc > 0x7fffffffLL) return TQ_ERR_UNSUPPORTED;
            if (w.mass && w.kind == TQ_SEG_PACKED) {
                mkb = std::max(mkb, static_cast<int>(w.kb));
                mq |= w.qjl != 0;
            }
        }
        P.mass_ctas = static_cast<int>(mc);
        P.mass_stage = mass_stage_bytes(mkb, mq, false);
        long long vc = 0;  // value sketches: the same split as the mass
        for (WorkItem &w : P.items) {
            w.vqjl_cta_begin = static_cast<int>(vc);
            if (w.vqs) {
                vc += static_cast<long long>(B) * ((w.n_tokens + kMassTokens - 1) / kMassTokens);
                vkb = std::max(vkb, static_cast<int>(w.kb));
                vq |= w.qjl != 0;
            }
            if (vc > 0x7fffffffLL) return TQ_ERR_UNSUPPORTED;
        }
        P.vqjl_ctas = static_cast<int>(vc);
        P.vqjl_stage = mass_stage_bytes(vkb, vq, true);
    }
    {  // per-CTA work items: stage range_begin(i) of a packed launch, chunk CTA i
       // of the fp16 launch, the CTAs of each mass / value-sketch item
        size_t total = static_cast<size_t>(P.mass_ctas) + P.vqjl_ctas;
        for (const ClassLaunch &c : P.classes) total += c.n_ctas;
        P.cta_item.clear();
        P.cta_item.reserve(total);
        for (ClassLaunch &c : P.classes) {
            c.cta_off = static_cast<int>(P.cta_item.size());
            int it = c.item_lo;
            for (int i = 0; i < c.n_ctas; ++i) {
                if (c.kb != 16) {
                    const long long s0 = dec_range_begin(i, c.n_stages, c.n_ctas);
                    while (it + 1 < c.item_hi && P.items[it + 1].stage_begin <= s0) ++it;
                } else {
                    while (it + 1 < c.item_hi && P.items[it + 1].cta_begin <= i) ++it;
                }
                P.cta_item.push_back(it);
            }
        }
        P.mass_cta_off = static_cast<int>(P.cta_item.size());
        for (size_t i = 0; i < P.items.size(); ++i)
            if (P.items[i].mass) {
                const long long n = static_cast<long long>(B) * ((P.items[i].n_tokens + kMassTokens - 1) / kMassTokens);
                P.cta_item.insert(P.cta_item.end(), static_cast<size_t>(n), static_cast<int>(i));
            }
        P.vqjl_cta_off = static_cast<int>(P.cta_item.size());
        for (size_t i = 0; i < P.items.size(); ++i)
            if (P.items[i].vqs) {
                const long long n = static_cast<long long>(B) * ((P.items[i].n_tokens + kMassTokens - 1) / kMassTokens);
                P.cta_item.insert(P.cta_item.end(), static_cast<size_t>(n), static_cast<int>(i));
            }
    }
    DecodeDims &D = P.dims;
    D.L = n_layers;
    D.B = B;
    D.H = H;
    D.Hq = Hq;
    D.gqa = gqa;
    D.any_qjl = P.any_qjl ? 1 : 0;
    // the prep kernel rotates every query once (the packed classes read its
    // output); calls with fp16 segments only skip it
    bool any_packed = false;
    for (const WorkItem &w : P.items) any_packed |= w.kind == TQ_SEG_PACKED;
    D.any_prep = any_packed || P.any_qjl || any_dense ? 1 : 0;
    D.inv_sqrt_d = inv_sqrt_f32(d);
    D.qk_scale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    D.wait_polls = g_wait_polls.load();
    D.nh = nh;
    D.np = np;
    const size_t nq = static_cast<size_t>(n_layers) * B * Hq;
    // offset 0: the error flag (kept in its own 256 bytes so that it has a
    // fixed place), then the work items
    P.off_items = 256;
    size_t off = P.off_items + align256(sizeof(WorkItem) * std::max<size_t>(P.items.size(), 1));
    P.off_layer = off;
    off += align256(sizeof(LayerPlan) * n_layers);
    P.off_grp_part = off;
    off += align256(sizeof(int) * std::max<size_t>(P.grp_part.size(), 1));
    P.off_grp_nparts = off;
    off += align256(sizeof(int) * std::max<size_t>(P.grp_nparts.size(), 1));
    P.off_lbh_total = off;
    off += align256(static_cast<size_t>(n_layers) * B * H * sizeof(int));
    P.off_cta_item = off;
    off += align256(sizeof(int) * std::max<size_t>(P.cta_item.size(), 1));
    P.off_counter = off;
    off += align256(static_cast<size_t>(n_layers) * B * H * sizeof(int));
    P.off_qrot = off;  // the uploaded plan ends here
    if (D.any_prep) {
        off += align256(nq * d * 4);
        P.off_qjlt = off;
        off += align256(nq * d * 4);
        P.off_qsum = off;
        off += align256(nq * 16);
    } else {
        P.off_qjlt = P.off_qsum = off;
    }
    P.off_part = off;
    off += align256(static_cast<size_t>(std::max(P.n_parts, 1)) * kMaxGqa * (4 + kD) * 4);
    P.off_ml = off;
    if (P.mass_ctas > 0 || P.vqjl_ctas > 0) off += align256(nq * 2 * sizeof(float));
    P.off_z = off;
    if (P.vqjl_ctas > 0) off += align256(nq * kD * sizeof(float));
    P.total = off;
    return TQ_OK;
}

}  // namespace

tq_status tqk::record_cuda_error(cudaError_t e) { return cuda_fail(e); }

// =============================================================== C ABI
extern "C" {

const char *tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "TQ_OK";
        case TQ_ERR_ARG: return "TQ_ERR_ARG: invalid argument";
        case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED: shape not implemented by the kernels";
        case TQ_ERR_ALIGN: return "TQ_ERR_ALIGN: pointer, stride or capacity not 16-byte aligned";
        case TQ_ERR_SIZE: return "TQ_ERR_SIZE: buffer or capacity too small";
        case TQ_ERR_CUDA: return "TQ_ERR_CUDA: CUDA runtime error (see tq_last_cuda_error)";
        case TQ_ERR_TIMEOUT: return "TQ_ERR_TIMEOUT: a kernel gave up waiting for its own copies; its output is incomplete";
        default: return "unknown tq_status";
    }
}

int tq_last_cuda_error(void) { return g_last_cuda; }

int tq_version(void) { return 100; }

tq_status tq_make_rotation(int head_dim, uint64_t seed, tq_rotation *rot) {
    if (!rot || !pow2(head_dim) || head_dim < 16 || head_dim > TQ_MAX_HEAD_DIM) return TQ_ERR_ARG;
    std::memset(rot, 0, sizeof(*rot));
    rot->head_dim = head_dim;
    rot->seed = seed;
    SplitMix64 g{seed};
    for (int i = 0; i < head_dim; ++i)
        if (g.next() >> 63) rot->sign_bits[i >> 5] |= 1u << (i & 31);
    return TQ_OK;
}

tq_status tq_fit_codebook(int bits, float *centroids, float *thresholds) {
    if (bits < 1 || bits > 8 || !centroids) return TQ_ERR_ARG;
    const FittedCodebook &cb = fit(bits);
    for (int k = 0; k < (1 << bits); ++k) centroids[k] = static_cast<float>(cb.level[k]);
    if (thresholds)
        for (int k = 0; k + 1 < (1 << bits); ++k) thresholds[k] = static_cast<float>(cb.bound[k]);
    return TQ_OK;
}

tq_status tq_fit_codebook_sphere(int bits, int head_dim, float *centroids, float *thresholds) {
    if (bits < 1 || bits > 8 || !centroids || head_dim < 4 || head_dim > TQ_MAX_HEAD_DIM) return TQ_ERR_ARG;
    FittedCodebook local;
    const FittedCodebook *cb = &local;
    if (head_dim == kD) cb = &fit(bits, TQ_VALUE_LAW_SPHERE);
    else fit_sphere(bits, head_dim, local);
    for (int k = 0; k < (1 << bits); ++k) centroids[k] = static_cast<float>(cb->level[k]);
    if (thresholds)
        for (int k = 0; k + 1 < (1 << bits); ++k) thresholds[k] = static_cast<float>(cb->bound[k]);
    return TQ_OK;
}

tq_status tq_value_code_table(int bits, const float *thresholds, uint32_t *table) {
    if (bits < 1 || bits > 4 || !thresholds || !table) return TQ_ERR_ARG;
    const int nt = (1 << bits) - 1;
    if (bits == 4) return value_buckets4(thresholds, nt, table) ? TQ_OK : TQ_ERR_UNSUPPORTED;
    std::vector<RowsParams::Bucket> b(kRowsBuckets);
    if (!value_buckets(thresholds, nt, b.data())) return TQ_ERR_UNSUPPORTED;
    for (int i = 0; i < kRowsBuckets; ++i) {
        table[2 * i] = b[i].t;
        table[2 * i + 1] = b[i].k;
    }
    return TQ_OK;
}

tq_status tq_make_haar_rotation(int head_dim, uint64_t seed, float *Q) {
    if (!Q || !pow2(head_dim) || head_dim < 16 || head_dim > TQ_MAX_HEAD_DIM) return TQ_ERR_ARG;
    const int d = head_dim;
    std::vector<float> g(static_cast<size_t>(d) * d);
    fill_gaussian(seed, d * d, g.data());  // the matrix tq_make_qjl(d, d, seed) writes
    // Householder QR in binary64: A = G; reflector k maps A[k:, k] onto
    // alpha_k e_1 with alpha_k = -sign(A_kk) ||A[k:, k]||, so R_kk = alpha_k.
    std::vector<double> A(g.begin(), g.end()), V(static_cast<size_t>(d) * d, 0.0), alpha(d);
    auto a = [&](int r, int c) -> double & { return A[static_cast<size_t>(r) * d + c]; };
    for (int k = 0; k < d; ++k) {
        double norm = 0.0;
        for (int r = k; r < d; ++r) norm += a(r, k) * a(r, k);
        norm = std::sqrt(norm);
        alpha[k] = a(k, k) >= 0.0 ? -norm : norm;
        double *v = &V[static_cast<size_t>(k) * d];
        for (int r = k; r < d; ++r) v[r] = a(r, k);
        v[k] -= alpha[k];
        double vn = 0.0;
        for (int r = k; r < d; ++r) vn += v[r] * v[r];
        vn = std::sqrt(vn);
        if (vn == 0.0) continue;  // column already alpha e_1
        for (int r = k; r < d; ++r) v[r] /= vn;
        for (int c = k; c < d; ++c) {
            double dot = 0.0;
            for (int r = k; r < d; ++r) dot += v[r] * a(r, c);
            for (int r = k; r < d; ++r) a(r, c) -= 2.0 * v[r] * dot;
        }
    }
    // Q = H_0 H_1 ... H_{d-1} (applied to I from the last reflector), then
    // column j times sign(R_jj) so that R has a positive diagonal
    std::vector<double> M(static_cast<size_t>(d) * d, 0.0);
    for (int i = 0; i < d; ++i) M[static_cast<size_t>(i) * d + i] = 1.0;
    for (int k = d - 1; k >= 0; --k) {
        const double *v = &V[static_cast<size_t>(k) * d];
        for (int c = 0; c < d; ++c) {
            double dot = 0.0;
            for (int r = k; r < d; ++r) dot += v[r] * M[static_cast<size_t>(r) * d + c];
            for (int r = k; r < d; ++r) M[static_cast<size_t>(r) * d + c] -= 2.0 * v[r] * dot;
        }
    }
    for (int r = 0; r < d; ++r)
        for (int c = 0; c < d; ++c)
            Q[static_cast<size_t>(r) * d + c] =
                static_cast<float>(alpha[c] < 0.0 ? -M[static_cast<size_t>(r) * d + c] : M[static_cast<size_t>(r) * d + c]);
    return TQ_OK;
}

tq_status tq_compress_error_flag(int *flag, int reset) {
    if (!flag) return TQ_ERR_ARG;
    cudaError_t e = read_compress_dense_error(flag);
    if (e == cudaSuccess && reset) e = clear_compress_dense_error();
    if (e != cudaSuccess) return cuda_fail(e);
    return *flag ? TQ_ERR_TIMEOUT : TQ_OK;
}

tq_status tq_make_qjl(int head_dim, int jl_dim, uint64_t seed, float *S) {
    if (!S || !pow2(head_dim) || head_dim < 16 || head_dim > TQ_MAX_HEAD_DIM) return TQ_ERR_ARG;
    if (jl_dim < 32 || jl_dim > 1024 || jl_dim % 32) return TQ_ERR_ARG;
    fill_gaussian(seed, jl_dim * head_dim, S);
    return TQ_OK;
}

tq_status tq_packed_size(const tq_segment_layout *layout, tq_packed_sizes *sizes) {
    tq_status st = check_layout(layout, true);
    if (st != TQ_OK) return st;
    if (!sizes) return TQ_ERR_ARG;
    const Offsets o = offsets(layout);
    const size_t B = layout->batch, cap = layout->capacity;
    size_t k = 0, v = 0;
    for (int h = 0; h < layout->n_heads; ++h) {
        k += cap * layout->head_dim * layout->kbits[h] / 8;
        v += cap * layout->head_dim * layout->vbits[h] / 8;
    }
    sizes->kcode_bytes = B * k;
    sizes->vcode_bytes = B * v;
    sizes->kscale_bytes = B * layout->n_heads * cap * 4;
    sizes->vscale_bytes = sizes->kscale_bytes;
    sizes->qjl_sign_bytes = B * o.nq * cap * (o.nq ? layout->jl_dim / 8 : 0);
    sizes->qjl_norm_bytes = B * o.nq * cap * 4;
    sizes->vqjl_sign_bytes = B * o.nv * cap * (o.nv ? layout->jl_dim / 8 : 0);
    sizes->vqjl_norm_bytes = B * o.nv * cap * 4;
    return TQ_OK;
}

tq_status tq_compress(const tq_segment_layout *layout, const tq_rotation *rot, const float *qjl_S,
                      const void *K, const void *V, int n_tokens, int64_t stride_b, int64_t stride_h,
                      int64_t stride_t, int t_begin, const tq_packed_bufs *out, void *stream) {
    tq_status st = check_layout(layout, true);
    if (st != TQ_OK) return st;
    if (!rot || !K || !V || !out || n_tokens < 0 || t_begin < 0) return TQ_ERR_ARG;
    if (rot->head_dim != layout->head_dim) return TQ_ERR_ARG;
    if (static_cast<int64_t>(t_begin) + n_tokens > layout->capacity) return TQ_ERR_SIZE;
    if (!out->kcodes || !out->vcodes || !out->kscale || !out->vscale) return TQ_ERR_ARG;
    if (!fits_u32(layout)) return TQ_ERR_UNSUPPORTED;
    const Offsets o = offsets(layout);
    if (layout->head_dim != kD)
        return compress_other_dims(layout, rot, o, K, V, n_tokens, stride_b, stride_h, stride_t, t_begin, out,
                                   static_cast<cudaStream_t>(stream));
    if (o.nq) {
        if (!qjl_S || !out->qjl_signs || !out->qjl_norm) return TQ_ERR_ARG;
        if (layout->jl_dim != kJl) return TQ_ERR_UNSUPPORTED;
        if (!aligned16(qjl_S) || !aligned16(out->qjl_signs)) return TQ_ERR_ALIGN;
    }
    if (o.nv) {
        if (!qjl_S || !out->vqjl_signs || !out->vqjl_norm) return TQ_ERR_ARG;
        if (layout->jl_dim != kJl) return TQ_ERR_UNSUPPORTED;
        if (!aligned16(qjl_S) || !aligned16(out->vqjl_signs)) return TQ_ERR_ALIGN;
    }
    if (!aligned16(K) || !aligned16(V) || !aligned16(out->kcodes) || !aligned16(out->vcodes) ||
        !aligned16(out->kscale) || !aligned16(out->vscale))
        return TQ_ERR_ALIGN;
    if (stride_t < kD || stride_h < 0 || stride_b < 0 || (stride_t % 8) || (stride_h % 8) || (stride_b % 8))
        return TQ_ERR_ALIGN;
    if (n_tokens == 0) return TQ_OK;
    CompressParams p;
    std::memset(&p, 0, sizeof(p));
    p.K = static_cast<const uint16_t *>(K);
    p.V = static_cast<const uint16_t *>(V);
    p.sb = stride_b;
    p.sh = stride_h;
    p.st = stride_t;
    p.B = layout->batch;
    p.H = layout->n_heads;
    p.T = n_tokens;
    p.t_begin = t_begin;
    p.capacity = layout->capacity;
    p.kcodes = static_cast<uint8_t *>(out->kcodes);
    p.vcodes = static_cast<uint8_t *>(out->vcodes);
    p.kscale = out->kscale;
    p.vscale = out->vscale;
    p.qjl_signs = static_cast<uint8_t *>(out->qjl_signs);
    p.qjl_norm = out->qjl_norm;
    p.S = qjl_S;
    p.nq = o.nq;
    p.vqjl_signs = static_cast<uint8_t *>(out->vqjl_signs);
    p.vqjl_norm = out->vqjl_norm;
    p.nv = o.nv;
    p.kblock = o.kblock;
    p.vblock = o.vblock;
    for (int h = 0; h < p.H; ++h) {
        p.koff[h] = o.koff[h];
        p.voff[h] = o.voff[h];
        p.kbits[h] = layout->kbits[h];
        p.vbits[h] = layout->vbits[h];
        p.qrank[h] = o.qrank[h];
        p.vrank[h] = o.vrank[h];
        p.sel[h] = static_cast<uint8_t>(h);
    }
    p.n_sel = p.H;
    std::memcpy(p.sign_bits, rot->sign_bits, sizeof(p.sign_bits));
    p.inv_sqrt_d = inv_sqrt_f32(kD);
    p.Q = rot->dense;
    fill_thresholds(p.thr, layout->vbits, p.H, layout->value_law);
    if (o.nv) fill_centroids(p.cent, layout->vbits, p.H, layout->value_law);
    if (p.Q) {  // dense rotation: the tensor-core kernel (no QJL heads)
        if (o.nq || o.nv) return TQ_ERR_UNSUPPORTED;
        if (!aligned16(p.Q)) return TQ_ERR_ALIGN;
        const cudaError_t e = launch_compress_dense(p, static_cast<cudaStream_t>(stream));
        if (e == cudaErrorInvalidValue) {
            cudaGetLastError();
            return TQ_ERR_UNSUPPORTED;  // strides TMA cannot describe
        }
        return e == cudaSuccess ? TQ_OK : cuda_fail(e);
    }
    // heads without sketches: one thread per vector, a launch per width; the
    // sketched heads (all heads if a value width's bucket table does not
    // separate its thresholds): four lanes per vector
    {
        CompressParams plain = p;
        plain.n_sel = 0;
        for (int h = 0; h < p.H; ++h)
            if (p.qrank[h] < 0 && p.vrank[h] < 0) plain.sel[plain.n_sel++] = static_cast<uint8_t>(h);
        if (plain.n_sel > 0) {
            const cudaError_t e = launch_rows(plain, layout, rot->sign_bits, kD, static_cast<cudaStream_t>(stream));
            if (e == cudaSuccess) {
                p.n_sel = 0;
                for (int h = 0; h < p.H; ++h)
                    if (p.qrank[h] >= 0 || p.vrank[h] >= 0) p.sel[p.n_sel++] = static_cast<uint8_t>(h);
                if (p.n_sel == 0) return TQ_OK;
            } else if (e != cudaErrorNotSupported) {
                return cuda_fail(e);
            }
        }
    }
    const cudaError_t e = launch_compress(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_dequantize(const tq_segment_layout *layout, const tq_packed_bufs *bufs, const tq_rotation *rot,
                        int t_begin, int n_tokens, float *k_rot, float *v_rot, float *k_orig, float *v_orig,
                        void *stream) {
    tq_status st = check_layout(layout, true);
    if (st != TQ_OK) return st;
    if (!bufs || !bufs->kcodes || !bufs->vcodes || !bufs->kscale || !bufs->vscale) return TQ_ERR_ARG;
    if (t_begin < 0 || n_tokens < 0) return TQ_ERR_ARG;
    if (static_cast<int64_t>(t_begin) + n_tokens > layout->capacity) return TQ_ERR_SIZE;
    if ((k_orig || v_orig) && !rot) return TQ_ERR_ARG;
    if (rot && rot->head_dim != layout->head_dim) return TQ_ERR_ARG;
    if (!fits_u32(layout)) return TQ_ERR_UNSUPPORTED;
    if (n_tokens == 0) return TQ_OK;
    const Offsets o = offsets(layout);
    if (layout->head_dim != kD)
        return dequantize_other_dims(layout, bufs, rot, o, t_begin, n_tokens, k_rot, v_rot, k_orig, v_orig,
                                     static_cast<cudaStream_t>(stream));
    DequantParams p;
    std::memset(&p, 0, sizeof(p));
    p.B = layout->batch;
    p.H = layout->n_heads;
    p.t_begin = t_begin;
    p.n = n_tokens;
    p.capacity = layout->capacity;
    p.kcodes = static_cast<const uint8_t *>(bufs->kcodes);
    p.vcodes = static_cast<const uint8_t *>(bufs->vcodes);
    p.kscale = bufs->kscale;
    p.vscale = bufs->vscale;
    p.kblock = o.kblock;
    p.vblock = o.vblock;
    for (int h = 0; h < p.H; ++h) {
        p.koff[h] = o.koff[h];
        p.voff[h] = o.voff[h];
        p.kbits[h] = layout->kbits[h];
        p.vbits[h] = layout->vbits[h];
    }
    if (rot) std::memcpy(p.sign_bits, rot->sign_bits, sizeof(p.sign_bits));
    p.Q = rot ? rot->dense : nullptr;
    if (p.Q && !aligned16(p.Q)) return TQ_ERR_ALIGN;
    p.inv_sqrt_d = inv_sqrt_f32(kD);
    p.k_rot = k_rot;
    p.v_rot = v_rot;
    p.k_orig = k_orig;
    p.v_orig = v_orig;
    fill_centroids(p.centroid, layout->vbits, p.H, layout->value_law);
    const cudaError_t e = launch_dequant(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_requantize(const tq_segment_layout *src, const tq_packed_bufs *src_bufs, int src_t_begin,
                        const tq_segment_layout *dst, const tq_packed_bufs *dst_bufs, int dst_t_begin,
                        int n_tokens, void *stream) {
    tq_status st = check_layout(src, true);
    if (st != TQ_OK) return st;
    st = check_layout(dst, true);
    if (st != TQ_OK) return st;
    if (!src_bufs || !dst_bufs || n_tokens < 0 || src_t_begin < 0 || dst_t_begin < 0) return TQ_ERR_ARG;
    if (src->batch != dst->batch || src->n_heads != dst->n_heads || src->head_dim != dst->head_dim)
        return TQ_ERR_ARG;
    if (src->head_dim != kD) return TQ_ERR_UNSUPPORTED;
    for (int h = 0; h < dst->n_heads; ++h)
        if (dst->qjl[h] || dst->qjl_v[h]) return TQ_ERR_UNSUPPORTED;  // demoted tokens carry no sketch
    if (static_cast<int64_t>(src_t_begin) + n_tokens > src->capacity ||
        static_cast<int64_t>(dst_t_begin) + n_tokens > dst->capacity)
        return TQ_ERR_SIZE;
    if (!src_bufs->kcodes || !src_bufs->vcodes || !src_bufs->kscale || !src_bufs->vscale || !dst_bufs->kcodes ||
        !dst_bufs->vcodes || !dst_bufs->kscale || !dst_bufs->vscale)
        return TQ_ERR_ARG;
    if (!aligned16(src_bufs->kcodes) || !aligned16(src_bufs->vcodes) || !aligned16(dst_bufs->kcodes) ||
        !aligned16(dst_bufs->vcodes) || !aligned16(src_bufs->kscale) || !aligned16(src_bufs->vscale) ||
        !aligned16(dst_bufs->kscale) || !aligned16(dst_bufs->vscale))
        return TQ_ERR_ALIGN;
    if (!fits_u32(src) || !fits_u32(dst)) return TQ_ERR_UNSUPPORTED;
    if (n_tokens == 0) return TQ_OK;
    const Offsets so = offsets(src), d_o = offsets(dst);
    RequantParams p;
    std::memset(&p, 0, sizeof(p));
    CompressParams &q = p.dst;
    q.B = dst->batch;
    q.H = dst->n_heads;
    q.T = n_tokens;
    q.t_begin = dst_t_begin;
    q.capacity = dst->capacity;
    q.kcodes = static_cast<uint8_t *>(dst_bufs->kcodes);
    q.vcodes = static_cast<uint8_t *>(dst_bufs->vcodes);
    q.kscale = dst_bufs->kscale;
    q.vscale = dst_bufs->vscale;
    q.kblock = d_o.kblock;
    q.vblock = d_o.vblock;
    for (int h = 0; h < q.H; ++h) {
        q.koff[h] = d_o.koff[h];
        q.voff[h] = d_o.voff[h];
        q.kbits[h] = dst->kbits[h];
        q.vbits[h] = dst->vbits[h];
        q.qrank[h] = -1;
        q.vrank[h] = -1;
        p.skoff[h] = so.koff[h];
        p.svoff[h] = so.voff[h];
        p.skbits[h] = src->kbits[h];
        p.svbits[h] = src->vbits[h];
    }
    fill_thresholds(q.thr, dst->vbits, q.H, dst->value_law);
    p.skcodes = static_cast<const uint8_t *>(src_bufs->kcodes);
    p.svcodes = static_cast<const uint8_t *>(src_bufs->vcodes);
    p.skscale = src_bufs->kscale;
    p.svscale = src_bufs->vscale;
    p.skblock = so.kblock;
    p.svblock = so.vblock;
    p.scapacity = src->capacity;
    p.s_t0 = src_t_begin;
    fill_centroids(p.centroid, src->vbits, src->n_heads, src->value_law);
    const cudaError_t e = launch_requantize(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_age_tiers(int n_tokens, int n_bounds, const int *age_bounds, int *start, int *end) {
    if (n_tokens < 0 || n_bounds < 0 || !start || !end || (n_bounds > 0 && !age_bounds)) return TQ_ERR_ARG;
    for (int i = 0; i < n_bounds; ++i)
        if (age_bounds[i] < 0 || (i > 0 && age_bounds[i] < age_bounds[i - 1])) return TQ_ERR_ARG;
    for (int tier = 0; tier <= n_bounds; ++tier) {
        const long long lo_age = tier == 0 ? 0 : age_bounds[tier - 1];
        // positions with lo_age <= n-1-p < hi_age  <=>  n-hi_age <= p <= n-1-lo_age
        const long long e = std::max<long long>(0, n_tokens - lo_age);
        long long s = 0;
        if (tier < n_bounds) s = std::max<long long>(0, static_cast<long long>(n_tokens) - age_bounds[tier]);
        start[tier] = static_cast<int>(std::min(s, e));
        end[tier] = static_cast<int>(e);
    }
    return TQ_OK;
}

tq_status tq_decode_workspace_size(const tq_layer_view *layers, int n_layers, int batch, int n_heads,
                                   int q_heads, int head_dim, size_t *bytes) {
    if (!bytes) return TQ_ERR_ARG;
    Plan P;
    tq_status st = build_plan(layers, n_layers, batch, n_heads, q_heads, head_dim, nullptr, kJl, P, false);
    if (st != TQ_OK) return st;
    *bytes = P.total;
    return TQ_OK;
}

// Pinned host staging of the per-call plan.  A copy from pageable memory
// synchronises the stream before it starts, which would keep the caller's host
// thread from running ahead of the GPU; slots of pinned memory are reused
// round-robin, each guarded by an event recorded after its copy.
struct PlanStaging {
    static constexpr int kSlots = 8;
    struct Slot {
        void *p = nullptr;
        size_t cap = 0;
        cudaEvent_t ev = nullptr;
        int dev = -1;
    };
    std::mutex mu;
    Slot slot[kSlots];
    int next = 0;
};
PlanStaging &plan_staging() {
    static PlanStaging s;
    return s;
}

tq_status tq_decode_attention(const tq_layer_view *layers, int n_layers, int batch, int n_heads, int q_heads,
                              int head_dim, const float *qjl_S, int jl_dim, const void *q, float *out,
                              void *workspace, size_t ws_bytes, void *stream) {
    if (!q || !out || !workspace) return TQ_ERR_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return TQ_ERR_ALIGN;
    Plan P;
    tq_status st = build_plan(layers, n_layers, batch, n_heads, q_heads, head_dim, qjl_S, jl_dim, P, true);
    if (st != TQ_OK) return st;
    if (ws_bytes < P.total) return TQ_ERR_SIZE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    // upload the plan (error flag, items, tables, zeroed counters) from a pinned slot
    cudaError_t e;
    {
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e);
        PlanStaging &ring = plan_staging();
        std::lock_guard<std::mutex> lock(ring.mu);
        PlanStaging::Slot &sl = ring.slot[ring.next];
        ring.next = (ring.next + 1) % PlanStaging::kSlots;
        if (sl.ev) {  // the slot's previous copy (kSlots calls ago) has normally long finished
            e = cudaEventSynchronize(sl.ev);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        if (sl.cap < P.off_qrot) {
            if (sl.p) cudaFreeHost(sl.p);
            sl.p = nullptr;
            sl.cap = 0;
            const size_t cap = std::max<size_t>(P.off_qrot, 64 * 1024);
            e = cudaHostAlloc(&sl.p, cap, cudaHostAllocPortable);
            if (e != cudaSuccess) return cuda_fail(e);
            sl.cap = cap;
        }
        if (sl.ev == nullptr || sl.dev != dev) {
            if (sl.ev) cudaEventDestroy(sl.ev);
            sl.ev = nullptr;
            e = cudaEventCreateWithFlags(&sl.ev, cudaEventDisableTiming);
            if (e != cudaSuccess) return cuda_fail(e);
            sl.dev = dev;
        }
        uint8_t *host = static_cast<uint8_t *>(sl.p);
        std::memset(host, 0, P.off_qrot);
        if (!P.items.empty())
            std::memcpy(host + P.off_items, P.items.data(), sizeof(WorkItem) * P.items.size());
        std::memcpy(host + P.off_layer, P.layer.data(), sizeof(LayerPlan) * P.layer.size());
        if (!P.grp_part.empty()) {
            std::memcpy(host + P.off_grp_part, P.grp_part.data(), sizeof(int) * P.grp_part.size());
            std::memcpy(host + P.off_grp_nparts, P.grp_nparts.data(), sizeof(int) * P.grp_nparts.size());
        }
        if (!P.lbh_total.empty())
            std::memcpy(host + P.off_lbh_total, P.lbh_total.data(), sizeof(int) * P.lbh_total.size());
        if (!P.signs.empty())
            std::memcpy(host + P.off_signs, P.signs.data(), sizeof(uint32_t) * P.signs.size());
        if (!P.cta_item.empty())
            std::memcpy(host + P.off_cta_item, P.cta_item.data(), sizeof(int) * P.cta_item.size());
        e = cudaMemcpyAsync(ws, host, P.off_qrot, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaEventRecord(sl.ev, s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (P.generic) {  // head dims other than kD: one kernel, one CTA per (layer, batch, KV head)
        GenDecodeParams gp;
        std::memset(&gp, 0, sizeof(gp));
        gp.L = n_layers;
        gp.B = batch;
        gp.H = n_heads;
        gp.Hq = q_heads;
        gp.gqa = P.dims.gqa;
        gp.qk_scale = P.dims.qk_scale;
        gp.inv_sqrt_d = P.dims.inv_sqrt_d;
        gp.items = reinterpret_cast<const WorkItem *>(ws + P.off_items);
        gp.layer = reinterpret_cast<const LayerPlan *>(ws + P.off_layer);
        gp.signs = reinterpret_cast<const uint32_t *>(ws + P.off_signs);
        gp.q = static_cast<const uint16_t *>(q);
        gp.out = out;
        {
            std::lock_guard<std::mutex> lock(g_cb_mutex_tables());
            for (const WorkItem &w : P.items)
                if (w.kind == TQ_SEG_PACKED) {
                    const FittedCodebook &cb = fit(w.vb, TQ_VALUE_LAW_GAUSS);
                    for (int k = 0; k < (1 << w.vb); ++k) gp.centroid[cb_off(w.vb) + k] = static_cast<float>(cb.level[k]);
                }
        }
        if (g_ev_start) {
            e = cudaEventRecord(g_ev_start, s);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        e = launch_gen_decode(gp, head_dim, s);
        if (e != cudaSuccess) return cuda_fail(e);
        if (g_ev_stop) {
            e = cudaEventRecord(g_ev_stop, s);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        g_last_launches.store(1);
        return TQ_OK;
    }
    DecodeWorkspace W;
    W.items = reinterpret_cast<WorkItem *>(ws + P.off_items);
    W.layer = reinterpret_cast<LayerPlan *>(ws + P.off_layer);
    W.grp_part = reinterpret_cast<int *>(ws + P.off_grp_part);
    W.grp_nparts = reinterpret_cast<int *>(ws + P.off_grp_nparts);
    W.lbh_total = reinterpret_cast<int *>(ws + P.off_lbh_total);
    W.counter = reinterpret_cast<int *>(ws + P.off_counter);
    W.cta_item = reinterpret_cast<const int *>(ws + P.off_cta_item);
    W.mass_cta_item = W.cta_item + P.mass_cta_off;
    W.vqjl_cta_item = W.cta_item + P.vqjl_cta_off;
    W.error = reinterpret_cast<int *>(ws);
    W.qrot = reinterpret_cast<uint32_t *>(ws + P.off_qrot);
    W.qjlt = reinterpret_cast<uint32_t *>(ws + P.off_qjlt);
    W.qsum = reinterpret_cast<float *>(ws + P.off_qsum);
    W.part = reinterpret_cast<float *>(ws + P.off_part);
    W.ml = P.mass_ctas > 0 || P.vqjl_ctas > 0 ? reinterpret_cast<float *>(ws + P.off_ml) : nullptr;
    W.z = P.vqjl_ctas > 0 ? reinterpret_cast<float *>(ws + P.off_z) : nullptr;
    W.q = static_cast<const uint16_t *>(q);
    W.out = out;
    // fp16 codebook values (and the 1-bit centroid) of every decode class;
    // 1-bit values decode as c1 * (2 code - 1) since the codebooks are symmetric
    static unsigned short value_half[2][9][256];
    static bool value_ready[2][9] = {};
    std::vector<const unsigned short *> class_half(P.classes.size(), nullptr);
    std::vector<float> class_c1(P.classes.size(), 0.f);
    {
        std::lock_guard<std::mutex> lock(g_cb_mutex_tables());
        for (size_t i = 0; i < P.classes.size(); ++i) {
            const ClassLaunch &c = P.classes[i];
            if (c.kb == 16) continue;
            const FittedCodebook &cb = fit(c.vb, c.law);
            if (!value_ready[c.law][c.vb]) {
                for (int k = 0; k < 256; ++k)
                    value_half[c.law][c.vb][k] =
                        k < (1 << c.vb) ? __half_as_ushort(__float2half_rn(static_cast<float>(cb.level[k]))) : 0;
                value_ready[c.law][c.vb] = true;
            }
            class_half[i] = value_half[c.law][c.vb];
            class_c1[i] = c.vb == 1 ? static_cast<float>(cb.level[1]) : 0.f;
        }
    }
    // (layer, KV head) groups without any token are written by no CTA: their
    // output is zero
    bool empty_group = false;
    for (int l = 0; l < n_layers; ++l)
        for (int h = 0; h < n_heads; ++h) empty_group |= P.layer[l].n_items[h] == 0;
    if (empty_group) {
        e = cudaMemsetAsync(out, 0, static_cast<size_t>(n_layers) * batch * q_heads * head_dim * sizeof(float), s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (P.items.empty()) return TQ_OK;
    int launched = 0;
    if (P.vqjl_ctas > 0) {  // the value-sketch sums accumulate into z
        e = cudaMemsetAsync(W.z, 0, static_cast<size_t>(n_layers) * batch * q_heads * kD * sizeof(float), s);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_decode_kernels(P.dims, W, P.classes.data(), static_cast<int>(P.classes.size()), qjl_S,
                              class_half.data(), class_c1.data(), s, g_ev_start, g_ev_stop, &launched);
    if (e == cudaSuccess && P.mass_ctas > 0) {
        e = launch_attention_mass(P.dims, W, P.mass_ctas, P.mass_stage, s);
        ++launched;
    }
    if (e == cudaSuccess && P.vqjl_ctas > 0) {
        e = launch_value_qjl(P.dims, W, P.vqjl_ctas, P.vqjl_stage, qjl_S, s);
        launched += 2;
    }
    g_last_launches.store(launched);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status tq_decode_error_flag(const void *workspace, int *flag, void *stream) {
    if (!flag) return TQ_ERR_ARG;
    if (!workspace) {  // the static scratch array of this device (tq_decode_attention_static)
        void *ws = nullptr;
        const tq_status st = static_workspace(&ws);
        if (st != TQ_OK) return st;
        workspace = ws;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(flag, workspace, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    return *flag ? TQ_ERR_TIMEOUT : TQ_OK;
}

tq_status tq_set_decode_wait_polls(int polls) {
    if (polls < 0 || polls > (1 << 20)) return TQ_ERR_ARG;
    g_wait_polls.store(polls);
    return TQ_OK;
}

int tq_decode_last_launches(void) { return g_last_launches_v; }

tq_status tq_set_decode_kernel_events(void *start, void *stop) {
    if ((start == nullptr) != (stop == nullptr)) return TQ_ERR_ARG;
    g_ev_start = static_cast<cudaEvent_t>(start);
    g_ev_stop = static_cast<cudaEvent_t>(stop);
    return TQ_OK;
}

}  // extern "C"
