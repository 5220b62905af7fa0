// tq_compress.cu -- rotation + per-vector scale + scalar quantization + bit
// packing (+ QJL residual sketch) of fp16 KV head vectors, and the parity-only
// dequantizer.
//
// Method: "turboquant-mlx" (TurboQuant-MLX v2.0 README), "Walsh-Hadamard
// Rotation" (SRHT D H D, O(d log d)) and "Asymmetric K/V Compression" (QJL on
// keys only); "TurboMOQ", "Architecture" (keys: symmetric quantize, values:
// Lloyd-Max grid quantize, per-head 1-8 bits) and "QJL residual correction".
//
// Design (GB300): one CTA per (batch, head, 64-token block); warps 0-1 take the
// 64 key vectors, warps 2-3 the 64 value vectors, one vector per thread so the
// whole Walsh-Hadamard transform stays in registers with no shuffles.  The
// block is staged with coalesced 16-byte cp.async copies into shared rows padded
// to 272 bytes, which makes each thread's 16-byte row reads bank-conflict free.
// Every rounding step is an explicit IEEE binary32 intrinsic (__fadd_rn,
// __fmul_rn, __frcp_rn, __fsqrt_rn): no contraction into FMA, so the codes are
// the same bits the fixed-order format defines.
#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tqk {
namespace {

constexpr int kTok = 64;         // tokens per CTA
constexpr int kRow = 272;        // padded shared row: 256 B of fp16 + 16 B
constexpr int kThreads = 128;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

// y = R x for one 128-vector: input sign flip applied to the fp16 bits, the
// seven butterfly stages h = 1..64 in ascending order, then one rounded
// multiply by +-binary32(1/sqrt(d)) (the output sign folded into the factor).
__device__ __forceinline__ void load_rotate(const uint8_t *row, const uint32_t *in_mask,
                                            const float *out_scale, float (&a)[kD]) {
#pragma unroll
    for (int c = 0; c < 16; c++) {
        uint4 v = *reinterpret_cast<const uint4 *>(row + c * 16);
        const uint4 mk = *reinterpret_cast<const uint4 *>(in_mask + c * 4);
        v.x ^= mk.x; v.y ^= mk.y; v.z ^= mk.z; v.w ^= mk.w;
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
            a[8 * c + 2 * e] = f.x;
            a[8 * c + 2 * e + 1] = f.y;
        }
    }
#pragma unroll
    for (int h = 1; h < kD; h <<= 1) {
#pragma unroll
        for (int i = 0; i < kD; i++) {
            if ((i & h) == 0) {
                const float u = a[i], v = a[i + h];
                a[i] = __fadd_rn(u, v);
                a[i + h] = __fsub_rn(u, v);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < kD / 4; c++) {
        const float4 s = *reinterpret_cast<const float4 *>(out_scale + 4 * c);
        a[4 * c] = __fmul_rn(a[4 * c], s.x);
        a[4 * c + 1] = __fmul_rn(a[4 * c + 1], s.y);
        a[4 * c + 2] = __fmul_rn(a[4 * c + 2], s.z);
        a[4 * c + 3] = __fmul_rn(a[4 * c + 3], s.w);
    }
}

// Code i occupies bits [B*i, B*i + B) of the record (LSB first).
template <int B>
__device__ __forceinline__ void put_code(uint32_t (&w)[4 * B], int i, uint32_t k) {
    const int bit = i * B, wi = bit >> 5, sh = bit & 31;
    w[wi] |= k << sh;
    if (sh + B > 32) w[wi + 1] |= k >> (32 - sh);
}

template <int B>
__device__ __forceinline__ void store_record(uint8_t *dst, const uint32_t (&w)[4 * B]) {
#pragma unroll
    for (int j = 0; j < B; j++)
        reinterpret_cast<uint4 *>(dst)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

// Select t[k*STRIDE] for a runtime k < N from a register-resident table (a
// binary tree of selects: no dynamic register indexing).
template <int N, int STRIDE>
__device__ __forceinline__ float select_tree(const float *t, uint32_t k) {
    if constexpr (N == 1) {
        return t[0];
    } else {
        constexpr int H = N / 2;
        const float lo = select_tree<H, STRIDE>(t, k);
        const float hi = select_tree<H, STRIDE>(t + H * STRIDE, k);
        return (k & H) ? hi : lo;
    }
}

// #{j : t[j] < u} for 2^VB - 1 sorted thresholds held in registers: VB levels
// of a binary search, each level choosing its threshold with a select tree.
template <int VB, int LEV = 0>
__device__ __forceinline__ uint32_t search_reg(float u, const float *t, uint32_t k) {
    if constexpr (LEV == VB) {
        return k;
    } else {
        constexpr int step = 1 << (VB - 1 - LEV);
        const float th = select_tree<(1 << LEV), 2 * step>(t + step - 1, k);
        return search_reg<VB, LEV + 1>(u, t, (k << 1) | (th < u ? 1u : 0u));
    }
}

// Same count with the thresholds in shared memory (wide codebooks).
template <int VB>
__device__ __forceinline__ uint32_t search_smem(float u, const float *t) {
    uint32_t k = 0;
#pragma unroll
    for (int s = 1 << (VB - 1); s >= 1; s >>= 1)
        if (t[k + s - 1] < u) k += s;
    return k;
}

template <int KB, bool QJL>
__device__ __noinline__ void key_vector(const CompressParams &p, const uint8_t *row,
                                        const uint32_t *in_mask, const float *out_scale, int b,
                                        int h, int pos) {
    float y[kD];
    load_rotate(row, in_mask, out_scale, y);
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kD; i++) m = fmaxf(m, fabsf(y[i]));
    const float r = m > 0.0f ? __frcp_rn(m) : 0.0f;
    constexpr float half_cells = static_cast<float>(1 << (KB - 1));
    constexpr float top = static_cast<float>((1 << KB) - 1);
    uint32_t w[4 * KB];
#pragma unroll
    for (int j = 0; j < 4 * KB; j++) w[j] = 0;
#pragma unroll
    for (int i = 0; i < kD; i++) {
        const float v = __fmul_rn(y[i], r);
        const float t = __fadd_rn(v, 1.0f);
        float u = __fmul_rn(t, half_cells);  // exact: power of two
        u = fminf(fmaxf(u, 0.0f), top);
        // floor(u) for u in [0, 255]: 2^23 + u rounded toward -inf is 2^23 + floor(u)
        const uint32_t k = __float_as_uint(__fadd_rd(u, 8388608.0f)) & 0xFFu;
        put_code<KB>(w, i, k);
        if constexpr (QJL) {
            // residual against the cell centre m * ((2k+1) 2^-KB - 1) (exact level)
            const float lev = __fadd_rn(__fmul_rn(static_cast<float>(2 * k + 1),
                                                  1.0f / static_cast<float>(1 << KB)), -1.0f);
            y[i] = __fsub_rn(y[i], __fmul_rn(m, lev));
        }
    }
    const size_t sidx = (static_cast<size_t>(b) * p.H + h) * p.capacity + pos;
    store_record<KB>(p.kcodes + static_cast<size_t>(b) * p.kblock + p.koff[h] +
                         static_cast<size_t>(pos) * (16 * KB), w);
    p.kscale[sidx] = m;
    if constexpr (QJL) {
        // p_j = sum_i S[j][i] r_i in binary32 (any order: the only decision is the
        // sign); bit j = (p_j >= 0).  rho = ||r||_2.
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < kD; i++) ss = fmaf(y[i], y[i], ss);
        uint32_t sb[4];
#pragma unroll
        for (int jw = 0; jw < 4; jw++) {
            uint32_t word = 0;
            for (int jj = 0; jj < 32; jj++) {
                const float4 *Sj = reinterpret_cast<const float4 *>(p.S + (jw * 32 + jj) * kD);
                float acc = 0.0f;
#pragma unroll
                for (int i4 = 0; i4 < kD / 4; i4++) {
                    const float4 s = __ldg(Sj + i4);
                    acc = fmaf(s.x, y[4 * i4], acc);
                    acc = fmaf(s.y, y[4 * i4 + 1], acc);
                    acc = fmaf(s.z, y[4 * i4 + 2], acc);
                    acc = fmaf(s.w, y[4 * i4 + 3], acc);
                }
                word |= (acc >= 0.0f ? 1u : 0u) << jj;
            }
            sb[jw] = word;
        }
        const size_t q = (static_cast<size_t>(b) * p.nq + p.qrank[h]) * p.capacity + pos;
        *reinterpret_cast<uint4 *>(p.qjl_signs + q * (kJl / 8)) = make_uint4(sb[0], sb[1], sb[2], sb[3]);
        p.qjl_norm[q] = sqrtf(ss);
    }
}

template <int VB>
__device__ __noinline__ void value_vector(const CompressParams &p, const uint8_t *row,
                                          const uint32_t *in_mask, const float *out_scale,
                                          const float *thr_smem, int b, int h, int pos) {
    float y[kD];
    load_rotate(row, in_mask, out_scale, y);
    // pairwise tree of squares in index order
    float s[kD / 2];
#pragma unroll
    for (int j = 0; j < kD / 2; j++)
        s[j] = __fadd_rn(__fmul_rn(y[2 * j], y[2 * j]), __fmul_rn(y[2 * j + 1], y[2 * j + 1]));
#pragma unroll
    for (int len = kD / 2; len > 1; len >>= 1) {
#pragma unroll
        for (int j = 0; j < len / 2; j++) s[j] = __fadd_rn(s[2 * j], s[2 * j + 1]);
    }
    const float sigma = __fsqrt_rn(__fmul_rn(s[0], 1.0f / kD));  // /d exact (power of two)
    const float r = sigma > 0.0f ? __frcp_rn(sigma) : 0.0f;
    uint32_t w[4 * VB];
#pragma unroll
    for (int j = 0; j < 4 * VB; j++) w[j] = 0;
    if constexpr (VB <= 4) {
        float t[(1 << VB) - 1];
#pragma unroll
        for (int j = 0; j < (1 << VB) - 1; j++) t[j] = p.thr[cb_off(VB) + j];
#pragma unroll
        for (int i = 0; i < kD; i++) {
            const float u = __fmul_rn(y[i], r);
            put_code<VB>(w, i, search_reg<VB>(u, t, 0u));
        }
    } else {
#pragma unroll
        for (int i = 0; i < kD; i++) {
            const float u = __fmul_rn(y[i], r);
            put_code<VB>(w, i, search_smem<VB>(u, thr_smem));
        }
    }
    const size_t sidx = (static_cast<size_t>(b) * p.H + h) * p.capacity + pos;
    store_record<VB>(p.vcodes + static_cast<size_t>(b) * p.vblock + p.voff[h] +
                         static_cast<size_t>(pos) * (16 * VB), w);
    p.vscale[sidx] = sigma;
}

__global__ void __launch_bounds__(kThreads, 2)
    compress_kernel(const __grid_constant__ CompressParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *rows = smem;                                            // [2][64][272]
    uint32_t *in_mask = reinterpret_cast<uint32_t *>(smem + 2 * kTok * kRow);  // [64]
    float *out_scale = reinterpret_cast<float *>(in_mask + kD / 2);             // [128]
    float *thr = out_scale + kD;                                                 // [255]

    const int h = blockIdx.y, b = blockIdx.z;
    const int t0 = blockIdx.x * kTok;
    const int nt = min(kTok, p.T - t0);
    const uint16_t *srcK = p.K + b * p.sb + h * p.sh;
    const uint16_t *srcV = p.V + b * p.sb + h * p.sh;
    for (int idx = threadIdx.x; idx < 2 * kTok * 16; idx += kThreads) {
        const int which = idx / (kTok * 16), r = (idx >> 4) % kTok, ch = idx & 15;
        if (r < nt) {
            const uint16_t *src = (which ? srcV : srcK) + static_cast<int64_t>(t0 + r) * p.st + ch * 8;
            cp_async16(rows + (which * kTok + r) * kRow + ch * 16, src);
        }
    }
    cp_async_commit();
    if (threadIdx.x < kD / 2) {
        const int i = 2 * threadIdx.x;
        const uint32_t s0 = (p.sign_bits[i >> 5] >> (i & 31)) & 1u;
        const uint32_t s1 = (p.sign_bits[(i + 1) >> 5] >> ((i + 1) & 31)) & 1u;
        in_mask[threadIdx.x] = (s0 << 15) | (s1 << 31);
    }
    {
        const int i = threadIdx.x;
        const uint32_t s = (p.sign_bits[i >> 5] >> (i & 31)) & 1u;
        out_scale[i] = s ? -p.inv_sqrt_d : p.inv_sqrt_d;
    }
    const int vb = p.vbits[h];
    for (int j = threadIdx.x; j < (1 << vb) - 1; j += kThreads) thr[j] = p.thr[cb_off(vb) + j];
    cp_async_wait_all();
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = (warp & 1) * 32 + lane;
    if (r >= nt) return;  // no barrier follows
    const int pos = p.t_begin + t0 + r;
    if (warp < 2) {
        const uint8_t *row = rows + r * kRow;
        const bool q = p.qrank[h] >= 0;
        switch (p.kbits[h] * 2 + (q ? 1 : 0)) {
#define TQ_KEY_CASE(KB)                                                                     \
    case 2 * KB: key_vector<KB, false>(p, row, in_mask, out_scale, b, h, pos); break;      \
    case 2 * KB + 1: key_vector<KB, true>(p, row, in_mask, out_scale, b, h, pos); break;
            TQ_KEY_CASE(1) TQ_KEY_CASE(2) TQ_KEY_CASE(3) TQ_KEY_CASE(4)
            TQ_KEY_CASE(5) TQ_KEY_CASE(6) TQ_KEY_CASE(7) TQ_KEY_CASE(8)
#undef TQ_KEY_CASE
            default: break;
        }
    } else {
        const uint8_t *row = rows + (kTok + r) * kRow;
        switch (vb) {
#define TQ_VAL_CASE(VB) \
    case VB: value_vector<VB>(p, row, in_mask, out_scale, thr, b, h, pos); break;
            TQ_VAL_CASE(1) TQ_VAL_CASE(2) TQ_VAL_CASE(3) TQ_VAL_CASE(4)
            TQ_VAL_CASE(5) TQ_VAL_CASE(6) TQ_VAL_CASE(7) TQ_VAL_CASE(8)
#undef TQ_VAL_CASE
            default: break;
        }
    }
}

constexpr size_t compress_smem() {
    return 2 * kTok * kRow + (kD / 2) * 4 + kD * 4 + 256 * 4;
}

// ------------------------------------------------------------------ dequant
// One thread per (b, h, token, K|V) vector: unpack, scale in binary32 and
// optionally rotate back to the original space.
__global__ void dequant_kernel(const __grid_constant__ DequantParams p) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t total = static_cast<int64_t>(p.B) * p.H * p.n * 2;
    if (idx >= total) return;
    const int which = static_cast<int>(idx & 1);
    int64_t v = idx >> 1;
    const int t = static_cast<int>(v % p.n);
    v /= p.n;
    const int h = static_cast<int>(v % p.H);
    const int b = static_cast<int>(v / p.H);
    const int pos = p.t_begin + t;
    const int bits = which ? p.vbits[h] : p.kbits[h];
    const uint8_t *rec = (which ? p.vcodes + static_cast<size_t>(b) * p.vblock + p.voff[h]
                                : p.kcodes + static_cast<size_t>(b) * p.kblock + p.koff[h]) +
                         static_cast<size_t>(pos) * (16 * bits);
    const size_t sidx = (static_cast<size_t>(b) * p.H + h) * p.capacity + pos;
    const float scale = which ? p.vscale[sidx] : p.kscale[sidx];
    const uint32_t mask = (1u << bits) - 1u;
    float y[kD];
#pragma unroll
    for (int i = 0; i < kD; i++) {
        const int bit = i * bits, by = bit >> 3;
        uint32_t word = rec[by];
        if ((bit & 7) + bits > 8) word |= static_cast<uint32_t>(rec[by + 1]) << 8;
        const uint32_t k = (word >> (bit & 7)) & mask;
        float lev;
        if (which) {
            lev = p.centroid[cb_off(bits) + k];
        } else {
            lev = __fadd_rn(__fmul_rn(static_cast<float>(2 * k + 1),
                                      __frcp_rn(static_cast<float>(1 << bits))), -1.0f);
        }
        y[i] = __fmul_rn(scale, lev);
    }
    const size_t o = ((static_cast<size_t>(b) * p.H + h) * p.n + t) * kD;
    float *rot = which ? p.v_rot : p.k_rot;
    if (rot) {
#pragma unroll
        for (int i = 0; i < kD; i++) rot[o + i] = y[i];
    }
    float *orig = which ? p.v_orig : p.k_orig;
    if (orig) {
#pragma unroll
        for (int i = 0; i < kD; i++)
            if ((p.sign_bits[i >> 5] >> (i & 31)) & 1u) y[i] = -y[i];
#pragma unroll
        for (int hh = 1; hh < kD; hh <<= 1) {
#pragma unroll
            for (int i = 0; i < kD; i++) {
                if ((i & hh) == 0) {
                    const float u = y[i], w = y[i + hh];
                    y[i] = u + w;
                    y[i + hh] = u - w;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kD; i++) {
            const float s = ((p.sign_bits[i >> 5] >> (i & 31)) & 1u) ? -p.inv_sqrt_d : p.inv_sqrt_d;
            orig[o + i] = y[i] * s;
        }
    }
}

}  // namespace

cudaError_t launch_compress(const CompressParams &p, cudaStream_t s) {
    static bool configured = false;
    const size_t smem = compress_smem();
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const dim3 grid((p.T + kTok - 1) / kTok, p.H, p.B);
    compress_kernel<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantParams &p, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(p.B) * p.H * p.n * 2;
    const int threads = 128;
    const int64_t blocks = (total + threads - 1) / threads;
    dequant_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace tqk
