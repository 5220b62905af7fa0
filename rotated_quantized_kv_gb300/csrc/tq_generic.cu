// tq_generic.cu -- compression, dequantization and decode attention for head
// dimensions other than 128: every power of two from 16 to 1024.
//
// Method: the same as the 128-dimension kernels ("turboquant-mlx" (TurboQuant-MLX
// v2.0 README), "Walsh-Hadamard Rotation": WalshHadamardRotation(head_dim, seed),
// the SRHT D H D / sqrt(d) for any power-of-two head_dim; "TurboMOQ",
// "Architecture": keys on a symmetric grid, values through a Gaussian Lloyd-Max
// codebook, 1-8 bits per head; "turboquant-mlx" skill note, "Optimisations
// Metal": attention on the compressed cache with the inverse transform pulled
// out of the value sum).  The format is the one the 128-dimension path writes:
// binary32 arithmetic in a fixed order, so codes and scales are a pure function
// of the fp16 input; code i of a vector at bits [b i, b i + b) of its d*b/8-byte
// record, LSB first.
//
// Rotation layout (GB300): a team of T lanes holds one vector, E = d / T
// coordinates per lane (d <= 64: T = d / 4, E = 4, several vectors per warp;
// d >= 256: one vector per warp, E = d / 32).  The butterfly stages h < E run in
// registers on the lane's contiguous coordinates; for d >= 256 a shared-memory
// stage then transposes the vector so that lane l holds coordinates l + 32 j:
// the stages E <= h < 32 are warp shuffles (partner lane l ^ h) and every stage
// h >= 32 is in registers again.  For d <= 64 the stages h >= E are shuffles
// inside the team.  The stages still run in ascending order, each pair
// (i, i + h) becoming (a + b, a - b) with one IEEE rounding each.
//
// Decode attention runs one CTA per (layer, batch element, KV head): the GQA
// group's queries are rotated once into shared memory, every segment's tokens
// are staged in chunks with cp.async, scored (a warp per token, lanes over the
// coordinates), folded into an online softmax (exp2 with a running max per
// query head) and summed against the values (threads over the coordinates);
// the packed tokens' sum stays in the rotated space and takes one inverse
// rotation at the end.  No QJL sketches, dense rotations or attention-mass
// outputs on this path (the host rejects them).
#include <algorithm>

#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tqk {
namespace {

constexpr int kGenThreads = 256;
constexpr int kGenWarps = kGenThreads / 32;
constexpr int kGenMaxChunk = 256;             // tokens per staged decode chunk
constexpr int kGenStageBytes = 64 * 1024;     // staging buffer of the decode kernel

__device__ __forceinline__ bool neg_coord(const uint32_t *sb, int i) { return (sb[i >> 5] >> (i & 31)) & 1u; }

template <int D>
struct Team {
    static constexpr int T = D >= 128 ? 32 : D / 4;  // lanes per vector
    static constexpr int E = D / T;                  // coordinates per lane
    static constexpr int VPW = 32 / T;               // vectors per warp
    static constexpr bool STAGE = D >= 256;          // shared-memory stage between the in-lane stages
};

// Coordinate held in slot e of team lane lt once the rotation is done.
template <int D>
__device__ __forceinline__ int coord(int lt, int e) {
    return Team<D>::STAGE ? lt + 32 * e : lt * Team<D>::E + e;
}

// The signs a team lane applies, as bit masks over its E slots: in_neg bit e
// for coordinate lt * E + e (the input), out_neg bit e for coord<D>(lt, e).
template <int D>
__device__ __forceinline__ void lane_sign_masks(const uint32_t *sb, int lt, uint32_t &in_neg, uint32_t &out_neg) {
    in_neg = out_neg = 0u;
#pragma unroll
    for (int e = 0; e < Team<D>::E; e++) {
        in_neg |= static_cast<uint32_t>(neg_coord(sb, lt * Team<D>::E + e)) << e;
        out_neg |= static_cast<uint32_t>(neg_coord(sb, coord<D>(lt, e))) << e;
    }
}

// y = c * D H D x in the format's binary32 order: input sign flip (exact),
// butterfly widths h = 1, 2, ..., D/2 ascending with each pair (i, i + h) ->
// (a + b, a - b), output sign flip (exact), one rounded multiply by c.  On
// entry a[e] is coordinate lt * E + e; on return slot e holds coord<D>(lt, e).
// stage: D floats of this warp's shared memory (d >= 256).
template <int D>
__device__ __forceinline__ void rotate_exact(float (&a)[Team<D>::E], int lt, uint32_t in_neg, uint32_t out_neg,
                                             float c, float *stage) {
    constexpr int E = Team<D>::E;
#pragma unroll
    for (int e = 0; e < E; e++)
        if ((in_neg >> e) & 1u) a[e] = -a[e];
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int i = 0; i < E; i++) {
            if ((i & h) == 0) {
                const float u = a[i], v = a[i + h];
                a[i] = __fadd_rn(u, v);
                a[i + h] = __fsub_rn(u, v);
            }
        }
    }
    if constexpr (!Team<D>::STAGE) {
        // stages h >= E: partner lane lt ^ (h / E) inside the team; the lower
        // lane keeps a + o, the upper one o - a
#pragma unroll
        for (int h = E; h < D; h <<= 1) {
            const int x = h / E;
            const bool up = (lt & x) != 0;
#pragma unroll
            for (int e = 0; e < E; e++) {
                const float o = __shfl_xor_sync(0xffffffffu, a[e], x);
                a[e] = up ? __fsub_rn(o, a[e]) : __fadd_rn(a[e], o);
            }
        }
    } else {
        // shared-memory stage: contiguous -> strided (lane l: coordinates l + 32 j)
#pragma unroll
        for (int e = 0; e < E; e += 4)
            *reinterpret_cast<float4 *>(stage + lt * E + e) = make_float4(a[e], a[e + 1], a[e + 2], a[e + 3]);
        __syncwarp();
#pragma unroll
        for (int j = 0; j < E; j++) a[j] = stage[lt + 32 * j];
        __syncwarp();
#pragma unroll
        for (int h = E; h < 32; h <<= 1) {  // partner lane lt ^ h, same slot
            const bool up = (lt & h) != 0;
#pragma unroll
            for (int j = 0; j < E; j++) {
                const float o = __shfl_xor_sync(0xffffffffu, a[j], h);
                a[j] = up ? __fsub_rn(o, a[j]) : __fadd_rn(a[j], o);
            }
        }
#pragma unroll
        for (int h = 32; h < D; h <<= 1) {  // slots j, j + h / 32 of the lane
            const int hj = h / 32;
#pragma unroll
            for (int j = 0; j < E; j++) {
                if ((j & hj) == 0) {
                    const float u = a[j], v = a[j + hj];
                    a[j] = __fadd_rn(u, v);
                    a[j + hj] = __fsub_rn(u, v);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < E; e++) a[e] = __fmul_rn(c, ((out_neg >> e) & 1u) ? -a[e] : a[e]);
}

// sum_i y_i^2 as a pairwise binary tree in index order, each square and sum
// rounded once; every lane of the team returns the root.  The lane's squares
// of E consecutive indices lt * E + e (for d >= 256 the rotated vector is
// strided, so the squares go through the warp's stage first) sum in-lane for
// the blocks up to E, then across lanes (partner lt ^ x: the two add the same
// pair, and IEEE addition commutes).
template <int D>
__device__ __forceinline__ float tree_sum_squares(const float (&a)[Team<D>::E], int lt, float *stage) {
    constexpr int E = Team<D>::E, T = Team<D>::T;
    float p[E];
    if constexpr (!Team<D>::STAGE) {
#pragma unroll
        for (int e = 0; e < E; e++) p[e] = __fmul_rn(a[e], a[e]);
    } else {
#pragma unroll
        for (int j = 0; j < E; j++) stage[lt + 32 * j] = __fmul_rn(a[j], a[j]);
        __syncwarp();
#pragma unroll
        for (int e = 0; e < E; e += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(stage + lt * E + e);
            p[e] = v.x;
            p[e + 1] = v.y;
            p[e + 2] = v.z;
            p[e + 3] = v.w;
        }
    }
#pragma unroll
    for (int len = E; len > 1; len >>= 1) {
#pragma unroll
        for (int j = 0; j < len / 2; j++) p[j] = __fadd_rn(p[2 * j], p[2 * j + 1]);
    }
    float s = p[0];
#pragma unroll
    for (int x = 1; x < T; x <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, x));
    return s;
}

// Bits [32 w, 32 w + 32) of a record from its code bytes (LSB-first stream).
__device__ __forceinline__ uint32_t record_word(const uint8_t *cw, int bits, int d, int w) {
    const int lo = 32 * w;
    uint32_t x = 0;
    for (int i = lo / bits; i < d && i * bits < lo + 32; i++) {
        const int off = i * bits - lo;
        const uint32_t k = cw[i];
        x |= off >= 0 ? (k << off) : (k >> -off);
    }
    return x;
}

// Store the d*bits/8-byte record built from the code bytes: each team lane
// assembles whole 32-bit words (coalesced 4-byte stores); records of d = 16 at
// an odd width in 2-byte halves.
template <int D>
__device__ __forceinline__ void store_record(const uint8_t *cw, int bits, uint8_t *dst, int lt) {
    constexpr int T = Team<D>::T;
    const int rk = D * bits / 8;
    if (rk % 4 == 0) {
        for (int c = lt; c < rk / 4; c += T) reinterpret_cast<uint32_t *>(dst)[c] = record_word(cw, bits, D, c);
    } else {  // d = 16 and an odd width: 2-byte halves
        for (int c = lt; c < rk / 2; c += T) {
            const uint32_t w = record_word(cw, bits, D, c >> 1);
            reinterpret_cast<uint16_t *>(dst)[c] = static_cast<uint16_t>((c & 1) ? (w >> 16) : (w & 0xFFFFu));
        }
    }
}

// Load the lane's E contiguous fp16 coordinates (16- or 8-byte loads).
template <int E>
__device__ __forceinline__ void load_coords(const uint16_t *src, float (&a)[E]) {
    if constexpr (E % 8 == 0) {
#pragma unroll
        for (int c = 0; c < E / 8; c++) {
            const uint4 v = reinterpret_cast<const uint4 *>(src)[c];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[q]));
                a[8 * c + 2 * q] = f.x;
                a[8 * c + 2 * q + 1] = f.y;
            }
        }
    } else {
        static_assert(E == 4, "four coordinates per lane below 256 dimensions");
        const uint2 v = *reinterpret_cast<const uint2 *>(src);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
        a[0] = f0.x;
        a[1] = f0.y;
        a[2] = f1.x;
        a[3] = f1.y;
    }
}

// ------------------------------------------------------------------ compress
// Rows (kv, b, h) of T vectors: blockIdx.y strides over the 2 B H rows (kv
// slowest), blockIdx.x over each row's tokens; warp teams take consecutive
// tokens of a row.
template <int D>
__global__ void __launch_bounds__(kGenThreads) gen_compress_kernel(const __grid_constant__ GenCompressParams p) {
    using TM = Team<D>;
    constexpr int E = TM::E, T = TM::T, VPW = TM::VPW;
    __shared__ float thr[kCbTotal];
    __shared__ __align__(16) float stage[TM::STAGE ? kGenWarps * D : 4];
    __shared__ __align__(16) uint8_t codes[kGenWarps][VPW * D];
    for (int j = threadIdx.x; j < kCbTotal; j += kGenThreads) thr[j] = p.thr[j];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v = lane / T, lt = lane % T;
    uint32_t in_neg, out_neg;
    lane_sign_masks<D>(p.sign_bits, lt, in_neg, out_neg);
    const int rows = 2 * p.B * p.H;
    for (int row = blockIdx.y; row < rows; row += gridDim.y)
    for (int t0 = (blockIdx.x * kGenWarps + warp) * VPW; t0 < p.T; t0 += gridDim.x * kGenWarps * VPW) {
        const int t = t0 + v;
        const bool valid = t < p.T;
        const int h = row % p.H;
        const int b = (row / p.H) % p.B;
        const int kv = row / (p.H * p.B);
        float a[E];
        if (valid) {
            load_coords<E>((kv ? p.V : p.K) + b * p.sb + h * p.sh + static_cast<int64_t>(t) * p.st + lt * E, a);
        } else {
#pragma unroll
            for (int e = 0; e < E; e++) a[e] = 0.0f;
        }
        rotate_exact<D>(a, lt, in_neg, out_neg, p.inv_sqrt_d, stage + (TM::STAGE ? warp * D : 0));
        // both per-vector statistics for every team, so that the exchanges stay uniform
        float m = 0.0f;
#pragma unroll
        for (int e = 0; e < E; e++) m = fmaxf(m, fabsf(a[e]));
#pragma unroll
        for (int x = 1; x < T; x <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, x));
        const float S = tree_sum_squares<D>(a, lt, stage + (TM::STAGE ? warp * D : 0));
        const int bits = kv ? p.vbits[h] : p.kbits[h];
        uint8_t *cw = codes[warp] + v * D;
        float scale;
        if (kv == 0) {  // keys: midrise grid on [-m, m]
            scale = m;
            const float rr = m > 0.0f ? __frcp_rn(m) : 0.0f;
            const float hc = static_cast<float>(1 << (bits - 1)), top = static_cast<float>((1 << bits) - 1);
#pragma unroll
            for (int e = 0; e < E; e++) {
                // round(v + 1) 2^(b-1) as one FMA (scaling by a power of two commutes with the rounding)
                float u = __fmaf_rn(__fmul_rn(a[e], rr), hc, hc);
                u = fminf(fmaxf(u, 0.0f), top);
                cw[coord<D>(lt, e)] = static_cast<uint8_t>(__float_as_uint(__fadd_rd(u, 8388608.0f)) & 0xFFu);
            }
        } else {  // values: #{k : thr_k < y / sigma}
            const float sigma = __fsqrt_rn(__fmul_rn(S, 1.0f / D));  // / d exact (a power of two)
            scale = sigma;
            const float rr = sigma > 0.0f ? __frcp_rn(sigma) : 0.0f;
            const float *th = thr + cb_off(bits);
#pragma unroll
            for (int e = 0; e < E; e++) {
                const float u = __fmul_rn(a[e], rr);
                int k = 0;
                for (int s = 1 << (bits - 1); s >= 1; s >>= 1)
                    if (th[k + s - 1] < u) k += s;
                cw[coord<D>(lt, e)] = static_cast<uint8_t>(k);
            }
        }
        __syncwarp();
        if (valid) {
            const int pos = p.t_begin + t;
            uint8_t *dst = (kv ? p.vcodes : p.kcodes) + static_cast<size_t>(b) * (kv ? p.vblock : p.kblock) +
                           (kv ? p.voff[h] : p.koff[h]) + static_cast<size_t>(pos) * (D * bits / 8);
            store_record<D>(cw, bits, dst, lt);
            if (lt == 0) (kv ? p.vscale : p.kscale)[(static_cast<size_t>(b) * p.H + h) * p.capacity + pos] = scale;
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------------ dequant
__device__ __forceinline__ uint32_t code_at(const uint8_t *rec, int i, int bits) {
    const int bit = i * bits, by = bit >> 3, sh = bit & 7;
    uint32_t v = rec[by];
    if (sh + bits > 8) v |= static_cast<uint32_t>(rec[by + 1]) << 8;
    return (v >> sh) & ((1u << bits) - 1u);
}

// One team per (b, h, t, K|V) vector: the rotated values m * level(code) or
// sigma * centroid[code] in binary32, then optionally R applied to them.
template <int D>
__global__ void __launch_bounds__(kGenThreads) gen_dequant_kernel(const __grid_constant__ GenDequantParams p) {
    using TM = Team<D>;
    constexpr int E = TM::E, T = TM::T, VPW = TM::VPW;
    __shared__ float cent[kCbTotal];
    __shared__ __align__(16) float stage[TM::STAGE ? kGenWarps * D : 4];
    for (int j = threadIdx.x; j < kCbTotal; j += kGenThreads) cent[j] = p.centroid[j];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v = lane / T, lt = lane % T;
    uint32_t in_neg, out_neg;
    lane_sign_masks<D>(p.sign_bits, lt, in_neg, out_neg);
    const long long NV = 2LL * p.B * p.H * p.n;
    const long long nwarps = static_cast<long long>(gridDim.x) * kGenWarps;
    for (long long base = (static_cast<long long>(blockIdx.x) * kGenWarps + warp) * VPW; base < NV;
         base += nwarps * VPW) {
        const long long f = base + v;
        const bool valid = f < NV;
        long long r = valid ? f : 0;
        const int t = static_cast<int>(r % p.n);
        r /= p.n;
        const int h = static_cast<int>(r % p.H);
        r /= p.H;
        const int b = static_cast<int>(r % p.B);
        const int kv = static_cast<int>(r / p.B);
        const int bits = kv ? p.vbits[h] : p.kbits[h];
        const int pos = p.t_begin + t;
        const uint8_t *rec = (kv ? p.vcodes : p.kcodes) + static_cast<size_t>(b) * (kv ? p.vblock : p.kblock) +
                             (kv ? p.voff[h] : p.koff[h]) + static_cast<size_t>(pos) * (D * bits / 8);
        const float sc = valid ? (kv ? p.vscale : p.kscale)[(static_cast<size_t>(b) * p.H + h) * p.capacity + pos] : 0.f;
        const float inv_cells = __uint_as_float(static_cast<uint32_t>(127 - bits) << 23);  // 2^-b
        float a[E];
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int i = lt * E + e;
            const uint32_t k = valid ? code_at(rec, i, bits) : 0u;
            a[e] = kv ? __fmul_rn(sc, cent[cb_off(bits) + k])
                      : __fmul_rn(sc, __fadd_rn(__fmul_rn(static_cast<float>(2 * k + 1), inv_cells), -1.0f));
        }
        const size_t row = ((static_cast<size_t>(b) * p.H + h) * p.n + t) * D;
        float *rot_out = kv ? p.v_rot : p.k_rot;
        if (valid && rot_out) {
#pragma unroll
            for (int e = 0; e < E; e++) rot_out[row + lt * E + e] = a[e];
        }
        float *orig_out = kv ? p.v_orig : p.k_orig;
        if (p.k_orig || p.v_orig) {  // uniform across the warp: every team rotates
            rotate_exact<D>(a, lt, in_neg, out_neg, p.inv_sqrt_d, stage + (TM::STAGE ? warp * D : 0));
            if (valid && orig_out) {
#pragma unroll
                for (int e = 0; e < E; e++) orig_out[row + coord<D>(lt, e)] = a[e];
            }
        }
    }
}

// ------------------------------------------------------------------ decode
// R x for a vector held by one warp with lane l owning coordinates l + 32 j
// (j < ceil(D/32); for D < 32 lanes >= D hold zeros): sign flip, butterflies
// (shuffles for h < 32, in-lane for h >= 32), sign flip, scale.  Attention
// arithmetic: any order within its tolerance.
template <int D>
__device__ __forceinline__ void warp_rotate_strided(float (&x)[(D + 31) / 32], const uint32_t *sb, float c,
                                                    int lane) {
    constexpr int J = (D + 31) / 32;
#pragma unroll
    for (int j = 0; j < J; j++) {
        const int i = lane + 32 * j;
        if (i < D && neg_coord(sb, i)) x[j] = -x[j];
    }
#pragma unroll
    for (int h = 1; h < (D < 32 ? D : 32); h <<= 1) {
        const bool up = (lane & h) != 0;
#pragma unroll
        for (int j = 0; j < J; j++) {
            const float o = __shfl_xor_sync(0xffffffffu, x[j], h);
            x[j] = up ? o - x[j] : x[j] + o;
        }
    }
#pragma unroll
    for (int h = 32; h < D; h <<= 1) {
        const int hj = h / 32;
#pragma unroll
        for (int j = 0; j < J; j++) {
            if ((j & hj) == 0) {
                const float u = x[j], v = x[j + hj];
                x[j] = u + v;
                x[j + hj] = u - v;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < J; j++) {
        const int i = lane + 32 * j;
        x[j] = (i < D && neg_coord(sb, i)) ? -c * x[j] : c * x[j];
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}

// bytes rounded up to 16 from a 16-byte aligned source (rows hold a multiple
// of 16 tokens, so the rounded run stays inside the row)
__device__ __forceinline__ void stage_run(uint8_t *dst, const uint8_t *src, int bytes) {
    for (int o = threadIdx.x * 16; o < bytes; o += kGenThreads * 16) cp_async16(dst + o, src + o);
}

template <int D>
constexpr size_t gen_decode_smem() {
    // queries (rotated, plain), scores, statistics, centroids, the two sums, staging
    return static_cast<size_t>(8 * D + 4 * kGenMaxChunk + 16 + 512 + 8 * D) * 4 + kGenStageBytes;
}

template <int D>
__global__ void __launch_bounds__(kGenThreads) gen_decode_kernel(const __grid_constant__ GenDecodeParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int J = (D + 31) / 32;
    float *qr = reinterpret_cast<float *>(smem);  // [4][D] R q of the group's query heads
    float *qo = qr + 4 * D;                       // [4][D] q
    float *sc = qo + 4 * D;                       // [4][kGenMaxChunk] scores, then weights
    float *st = sc + 4 * kGenMaxChunk;            // [0,4) running max, [4,8) sum, [8,12) correction
    float *cent = st + 16;                        // [512] value centroids, flat by width
    float *red = cent + 512;                      // [2][4][D] packed (rotated) and fp16 sums
    uint8_t *stg = reinterpret_cast<uint8_t *>(red + 8 * D);
    const int g = p.gqa;
    const int h = blockIdx.x % p.H;
    const int b = (blockIdx.x / p.H) % p.B;
    const int l = blockIdx.x / (p.H * p.B);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t *sgn = p.signs + static_cast<size_t>(l) * (kMaxD / 32);

    for (int j = threadIdx.x; j < kCbTotal; j += kGenThreads) cent[j] = p.centroid[j];
    for (int j = threadIdx.x; j < 8 * D; j += kGenThreads) red[j] = 0.0f;
    if (threadIdx.x < 4) {
        st[threadIdx.x] = -__builtin_huge_valf();
        st[4 + threadIdx.x] = 0.0f;
        st[8 + threadIdx.x] = 1.0f;
    }
    if (warp < g) {  // warp w rotates query head h g + w once
        const uint16_t *qp = p.q + ((static_cast<size_t>(l) * p.B + b) * p.Hq + h * g + warp) * D;
        float x[J];
#pragma unroll
        for (int j = 0; j < J; j++) {
            const int i = lane + 32 * j;
            x[j] = i < D ? __half2float(__ushort_as_half(qp[i])) : 0.0f;
            if (i < D) qo[warp * D + i] = x[j];
        }
        warp_rotate_strided<D>(x, sgn, p.inv_sqrt_d, lane);
#pragma unroll
        for (int j = 0; j < J; j++) {
            const int i = lane + 32 * j;
            if (i < D) qr[warp * D + i] = x[j];
        }
    }
    __syncthreads();

    // value sums: thread (dim lane vd, token phase ph), EV dims each
    constexpr int DT = D < kGenThreads ? D : kGenThreads;
    constexpr int NPH = kGenThreads / DT;
    constexpr int EV = D / DT;
    const int vd = threadIdx.x % DT, ph = threadIdx.x / DT;
    float accr[4][EV], acco[4][EV];
#pragma unroll
    for (int w = 0; w < 4; w++)
#pragma unroll
        for (int e = 0; e < EV; e++) accr[w][e] = acco[w][e] = 0.0f;

    const LayerPlan &lp = p.layer[l];
    for (int ii = 0; ii < lp.n_items[h]; ii++) {
        const WorkItem &it = p.items[lp.item[h][ii]];
        const bool packed = it.kind == TQ_SEG_PACKED;
        const int kb = packed ? it.kb : 16, vb = packed ? it.vb : 16;
        const int rk = D * kb / 8, rv = D * vb / 8;
        const int bpt = rk + rv + (packed ? 8 : 0);
        const int C = max(16, min(kGenMaxChunk, (kGenStageBytes / bpt) & ~15));
        const uint8_t *kc = it.kc + b * it.kstride, *vc = it.vc + b * it.vstride;
        const float *ks = packed ? it.ks + static_cast<size_t>(b) * it.sstride : nullptr;
        const float *vs = packed ? it.vs + static_cast<size_t>(b) * it.sstride : nullptr;
        uint8_t *sk = stg, *sv = stg + C * rk;
        float *sks = reinterpret_cast<float *>(sv + C * rv), *svs = sks + C;
        const float inv_cells = __uint_as_float(static_cast<uint32_t>(127 - (packed ? kb : 1)) << 23);
        const float *cv = cent + cb_off(packed ? vb : 1);
        for (int t0 = 0; t0 < it.n_tokens; t0 += C) {
            const int n = min(C, it.n_tokens - t0);
            stage_run(sk, kc + static_cast<size_t>(t0) * rk, (n * rk + 15) & ~15);
            stage_run(sv, vc + static_cast<size_t>(t0) * rv, (n * rv + 15) & ~15);
            if (packed) {
                stage_run(reinterpret_cast<uint8_t *>(sks), reinterpret_cast<const uint8_t *>(ks + t0), (n * 4 + 15) & ~15);
                stage_run(reinterpret_cast<uint8_t *>(svs), reinterpret_cast<const uint8_t *>(vs + t0), (n * 4 + 15) & ~15);
            }
            asm volatile("cp.async.commit_group;\n" ::);
            asm volatile("cp.async.wait_group 0;\n" ::: "memory");
            __syncthreads();
            // scores: a warp per token, lanes over the coordinates
            for (int t = warp; t < n; t += kGenWarps) {
                float dq[4] = {0.f, 0.f, 0.f, 0.f};
                if (packed) {
                    const uint8_t *rec = sk + t * rk;
#pragma unroll
                    for (int j = 0; j < J; j++) {
                        const int i = lane + 32 * j;
                        if (i < D) {
                            const uint32_t k = code_at(rec, i, kb);
                            const float lev = __fmaf_rn(static_cast<float>(2 * k + 1), inv_cells, -1.0f);
#pragma unroll
                            for (int w = 0; w < 4; w++)
                                if (w < g) dq[w] = fmaf(qr[w * D + i], lev, dq[w]);
                        }
                    }
                } else {
                    const __half *kr = reinterpret_cast<const __half *>(sk + t * rk);
#pragma unroll
                    for (int j = 0; j < J; j++) {
                        const int i = lane + 32 * j;
                        if (i < D) {
                            const float kx = __half2float(kr[i]);
#pragma unroll
                            for (int w = 0; w < 4; w++)
                                if (w < g) dq[w] = fmaf(qo[w * D + i], kx, dq[w]);
                        }
                    }
                }
                const float m = packed ? sks[t] : 1.0f;
#pragma unroll
                for (int w = 0; w < 4; w++) {
                    if (w < g) {
                        const float s = warp_sum(dq[w]);
                        if (lane == 0) sc[w * kGenMaxChunk + t] = m * s * p.qk_scale;
                    }
                }
            }
            __syncthreads();
            // online softmax in base 2: warp w handles query head w
            if (warp < g) {
                float mx = -__builtin_huge_valf();
                for (int t = lane; t < n; t += 32) mx = fmaxf(mx, sc[warp * kGenMaxChunk + t]);
                mx = warp_max(mx);
                const float mold = st[warp];
                const float mnew = fmaxf(mold, mx);
                const float corr = mold == -__builtin_huge_valf() ? 0.0f : exp2f(mold - mnew);
                float sum = 0.0f;
                for (int t = lane; t < n; t += 32) {
                    const float w = exp2f(sc[warp * kGenMaxChunk + t] - mnew);
                    sc[warp * kGenMaxChunk + t] = w;
                    sum += w;
                }
                sum = warp_sum(sum);
                __syncwarp();
                if (lane == 0) {
                    st[warp] = mnew;
                    st[4 + warp] = st[4 + warp] * corr + sum;
                    st[8 + warp] = corr;
                }
            }
            __syncthreads();
            // values: thread (vd, ph) over dims vd + DT e and tokens ph, ph + NPH, ...
#pragma unroll
            for (int w = 0; w < 4; w++) {
                if (w < g) {
                    const float cw = st[8 + w];
#pragma unroll
                    for (int e = 0; e < EV; e++) {
                        accr[w][e] *= cw;
                        acco[w][e] *= cw;
                    }
                }
            }
            for (int t = ph; t < n; t += NPH) {
                float wt[4];
#pragma unroll
                for (int w = 0; w < 4; w++) wt[w] = w < g ? sc[w * kGenMaxChunk + t] : 0.0f;
                if (packed) {
                    const uint8_t *rec = sv + t * rv;
                    const float sig = svs[t];
#pragma unroll
                    for (int e = 0; e < EV; e++) {
                        const float val = sig * cv[code_at(rec, vd + DT * e, vb)];
#pragma unroll
                        for (int w = 0; w < 4; w++) accr[w][e] = fmaf(wt[w], val, accr[w][e]);
                    }
                } else {
                    const __half *vr = reinterpret_cast<const __half *>(sv + t * rv);
#pragma unroll
                    for (int e = 0; e < EV; e++) {
                        const float val = __half2float(vr[vd + DT * e]);
#pragma unroll
                        for (int w = 0; w < 4; w++) acco[w][e] = fmaf(wt[w], val, acco[w][e]);
                    }
                }
            }
            __syncthreads();  // before the next chunk is staged over this one
        }
    }
    // combine the token phases, rotate the packed (rotated-space) sum back once,
    // normalise and store
#pragma unroll
    for (int w = 0; w < 4; w++) {
        if (w < g) {
#pragma unroll
            for (int e = 0; e < EV; e++) {
                const int d = vd + DT * e;
                if (NPH == 1) {
                    red[w * D + d] = accr[w][e];
                    red[4 * D + w * D + d] = acco[w][e];
                } else {
                    atomicAdd(&red[w * D + d], accr[w][e]);
                    atomicAdd(&red[4 * D + w * D + d], acco[w][e]);
                }
            }
        }
    }
    __syncthreads();
    if (warp < g) {
        float x[J];
#pragma unroll
        for (int j = 0; j < J; j++) {
            const int i = lane + 32 * j;
            x[j] = i < D ? red[warp * D + i] : 0.0f;
        }
        warp_rotate_strided<D>(x, sgn, p.inv_sqrt_d, lane);
        const float L = st[4 + warp];
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
        float *op = p.out + ((static_cast<size_t>(l) * p.B + b) * p.Hq + h * g + warp) * D;
#pragma unroll
        for (int j = 0; j < J; j++) {
            const int i = lane + 32 * j;
            if (i < D) op[i] = (x[j] + red[4 * D + warp * D + i]) * inv;
        }
    }
}

template <int D>
cudaError_t gen_compress_launch(const GenCompressParams &p, cudaStream_t s) {
    const int rows = 2 * p.B * p.H;
    const long long per_block = static_cast<long long>(kGenWarps) * Team<D>::VPW;
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // about 8 resident blocks per SM in all, each block a strided share of one row
    const long long want_x = std::max<long long>(1, static_cast<long long>(sms) * 8 / std::max(rows, 1));
    const long long bx = std::min<long long>((p.T + per_block - 1) / per_block, want_x);
    const int by = std::min(rows, 65535);
    gen_compress_kernel<D><<<dim3(static_cast<unsigned>(bx), static_cast<unsigned>(by)), kGenThreads, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t gen_dequant_launch(const GenDequantParams &p, cudaStream_t s) {
    const long long vecs = 2LL * p.B * p.H * p.n;
    const long long per_block = static_cast<long long>(kGenWarps) * Team<D>::VPW;
    const long long blocks = std::min<long long>((vecs + per_block - 1) / per_block, 1LL << 20);
    gen_dequant_kernel<D><<<static_cast<unsigned>(blocks), kGenThreads, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t gen_decode_launch(const GenDecodeParams &p, cudaStream_t s) {
    constexpr size_t smem = gen_decode_smem<D>();
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(gen_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const long long blocks = static_cast<long long>(p.L) * p.B * p.H;
    gen_decode_kernel<D><<<static_cast<unsigned>(blocks), kGenThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

#define TQ_GEN_DISPATCH(FN, d, ...)                   \
    switch (d) {                                       \
        case 16: return FN<16>(__VA_ARGS__);           \
        case 32: return FN<32>(__VA_ARGS__);           \
        case 64: return FN<64>(__VA_ARGS__);           \
        case 256: return FN<256>(__VA_ARGS__);         \
        case 512: return FN<512>(__VA_ARGS__);         \
        case 1024: return FN<1024>(__VA_ARGS__);       \
        default: return cudaErrorInvalidValue;         \
    }

cudaError_t launch_gen_compress(const GenCompressParams &p, int d, cudaStream_t s) {
    TQ_GEN_DISPATCH(gen_compress_launch, d, p, s)
}
cudaError_t launch_gen_dequant(const GenDequantParams &p, int d, cudaStream_t s) {
    TQ_GEN_DISPATCH(gen_dequant_launch, d, p, s)
}
cudaError_t launch_gen_decode(const GenDecodeParams &p, int d, cudaStream_t s) {
    TQ_GEN_DISPATCH(gen_decode_launch, d, p, s)
}

}  // namespace tqk
