// tq_compress.cu -- rotation + per-vector scale + scalar quantization + bit
// packing (+ QJL residual sketch) of fp16 KV head vectors, and the parity-only
// dequantizer.
//
// Method: "turboquant-mlx" (TurboQuant-MLX v2.0 README), "Walsh-Hadamard
// Rotation" (SRHT D H D, O(d log d)) and "Asymmetric K/V Compression" (QJL on
// keys only); "TurboMOQ", "Architecture" (keys: symmetric quantize, values:
// Lloyd-Max grid quantize, per-head 1-8 bits) and "QJL residual correction".
//
// Design (GB300): four lanes per vector, each holding 32 of its coordinates in
// registers: butterfly stages h = 1..16 stay in registers, stages h = 32 and
// h = 64 are exchanges with the partner lanes (xor 1, xor 2), and every later
// reduction (absmax, the pairwise sum of squares) finishes with exchanges in the
// same fixed order.  A CTA of 8 warps runs two independent groups: warps 0-3
// compress key vectors, warps 4-7 value vectors, 32 vectors per pass.  Each
// group loops over 32-token blocks of (batch, head) on its own, over the heads
// the launch selects (the host sends heads without sketches to the
// one-thread-per-vector kernels) (persistent
// CTAs, three per SM), double-buffers its rows with coalesced 16-byte cp.async
// copies and synchronises on its own named barrier, so the lighter key path
// never waits for the value path.  Shared rows are laid out as four 80-byte
// quarters (64 B of coordinates + 16 B pad) so that the eight 16-byte reads of
// a load phase fall in eight different bank groups.  Every rounding step is an
// explicit IEEE binary32 intrinsic (__fadd_rn, __fmul_rn, __frcp_rn,
// __fsqrt_rn): no contraction into FMA, so the codes are the same bits the
// fixed-order format defines.
#include <algorithm>

#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tqk {
namespace {

constexpr int kTok = 32;          // tokens per block
constexpr int kQuarter = 80;      // 64 B of coordinates + 16 B pad
constexpr int kRow = 4 * kQuarter;
constexpr int kThreads = 256;     // two groups of 4 warps (keys, values); 4 lanes per vector
constexpr int kQ = kD / 4;        // coordinates per lane
constexpr int kGroupBuf = kTok * kRow;  // one staged block of one group

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// barrier of one 128-thread group (ids 1, 2; 0 is __syncthreads)
__device__ __forceinline__ void group_sync(int group) {
    if (group == 0) asm volatile("bar.sync 1, 128;" ::: "memory");
    else asm volatile("bar.sync 2, 128;" ::: "memory");
}

// y = R x for one 128-vector held by four lanes: this lane's coordinates
// [32 q, 32 q + 32) in a[0..31].  Input sign flip on the fp16 bits, the seven
// butterfly stages h = 1..64 in ascending order (h = 32: lanes q, q^1; h = 64:
// lanes q, q^2; the lower lane keeps a_i + a_{i+h}, the upper one
// a_i - a_{i+h}), then one rounded multiply by +-binary32(1/sqrt(d)) (the
// output sign folded in).
__device__ __forceinline__ void load_rotate(const uint8_t *qrow, const uint32_t *in_mask, const float *out_scale,
                                            int q, float (&a)[kQ]) {
#pragma unroll
    for (int c = 0; c < 4; c++) {
        uint4 v = *reinterpret_cast<const uint4 *>(qrow + c * 16);
        const uint4 mk = *reinterpret_cast<const uint4 *>(in_mask + (c * 4 + q) * 4);
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
    for (int h = 1; h < kQ; h <<= 1) {
#pragma unroll
        for (int i = 0; i < kQ; i++) {
            if ((i & h) == 0) {
                const float u = a[i], v = a[i + h];
                a[i] = __fadd_rn(u, v);
                a[i + h] = __fsub_rn(u, v);
            }
        }
    }
    // the upper lane's o - a is fma(-1, a, o) and the lower lane's a + o is
    // fma(1, a, o): one rounding of an exact product, the same bits (signed
    // zeros included) as the subtraction or addition
#pragma unroll
    for (int x = 1; x <= 2; x <<= 1) {
        const float sgn = (q & x) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < kQ; i++) {
            const float o = __shfl_xor_sync(0xffffffffu, a[i], x);
            a[i] = __fmaf_rn(sgn, a[i], o);
        }
    }
#pragma unroll
    for (int c = 0; c < kQ / 4; c++) {
        const float4 s = *reinterpret_cast<const float4 *>(out_scale + (c * 4 + q) * 4);
        a[4 * c] = __fmul_rn(a[4 * c], s.x);
        a[4 * c + 1] = __fmul_rn(a[4 * c + 1], s.y);
        a[4 * c + 2] = __fmul_rn(a[4 * c + 2], s.z);
        a[4 * c + 3] = __fmul_rn(a[4 * c + 3], s.w);
    }
}

// Code i of this lane's 32 occupies bits [B*i, B*i + B) of its quarter record
// (the record's bytes [4 B q, 4 B q + 4 B)), LSB first.
template <int B>
__device__ __forceinline__ void put_code(uint32_t (&w)[B], int i, uint32_t k) {
    const int bit = i * B, wi = bit >> 5, sh = bit & 31;
    w[wi] |= k << sh;
    if (sh + B > 32) w[wi + 1] |= k >> (32 - sh);
}

template <int B>
__device__ __forceinline__ void store_quarter_record(uint8_t *dst, const uint32_t (&w)[B]) {
#pragma unroll
    for (int j = 0; j < B; j++) reinterpret_cast<uint32_t *>(dst)[j] = w[j];
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

// ------------------------------------------------------------------ QJL sketch
// Residuals of a 32-token block in shared memory, [32 rows][kRStride] binary32:
// 16 floats of pad per row put the eight rows a quarter-warp reads with one
// 16-byte load (rows g and g + 1 of a lane pair, four chunks each) in eight
// different bank groups.
constexpr int kRStride = kD + 16;
constexpr int kRSmem = kTok * kRStride * 4;

// This lane's quarter of a residual into row `row` of the block buffer, and
// the residual's squared norm (binary32, any order) for rho = ||r||_2.
__device__ __forceinline__ float residual_to_smem(float *R, const float (&y)[kQ], int row, int q) {
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < kQ; i++) ss = fmaf(y[i], y[i], ss);
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    float *dst = R + row * kRStride + kQ * q;
#pragma unroll
    for (int i = 0; i < kQ; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(y[i], y[i + 1], y[i + 2], y[i + 3]);
    return ss;
}

__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// x = hi + lo to 2^-22 relative: hi = tf32(x), lo = tf32(x - hi) (x - hi is exact)
__device__ __forceinline__ void tf32_split(float x, uint32_t &hi, uint32_t &lo) {
    hi = tf32_rna(x);
    lo = tf32_rna(x - __uint_as_float(hi));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float f4at(const float4 &v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

// Signs of P = R S^T for the block's 32 residual rows, projections [32 wq,
// 32 wq + 32) on this warp (wq: the warp within its group), on the tensor
// cores: mma.m16n8k8 in tf32 with every operand split as hi + lo and the
// products hi hi + hi lo + lo hi accumulated in binary32.  Each dropped or
// rounded part is below 2^-22 of |S_ji r_i|, so |P - S r| stays below
// 7.2e-7 ||S_j|| ||r|| besides the accumulation rounding (the plain binary32
// sum has the same kind of bound); only the sign of P is kept, bit j = (P_j >=
// 0).  Within a pair of k-steps lane c takes dims 16 kp + 4 c .. + 3 of both
// operands (any dim order is the same sum).  Row t's 16-byte record at rec0 +
// 16 t receives word wq, for t < n_valid.
__device__ __noinline__ void block_sketch(const float *R, const float *S, int wq, int lane, uint8_t *rec0,
                                          int n_valid) {
    const int g = lane >> 2, c = lane & 3;
    uint32_t word[2][2] = {{0u, 0u}, {0u, 0u}};  // [m-tile][row g | g + 8]
#pragma unroll 1
    for (int nh = 0; nh < 2; nh++) {  // n-tiles 2 nh, 2 nh + 1
        float acc[2][2][4];
#pragma unroll
        for (int mt = 0; mt < 2; mt++)
#pragma unroll
            for (int nt = 0; nt < 2; nt++)
#pragma unroll
                for (int e = 0; e < 4; e++) acc[mt][nt][e] = 0.0f;
#pragma unroll 2
        for (int kp = 0; kp < kD / 16; kp++) {
            float4 ra[2][2], sb[2];
#pragma unroll
            for (int mt = 0; mt < 2; mt++)
#pragma unroll
                for (int hf = 0; hf < 2; hf++)
                    ra[mt][hf] = *reinterpret_cast<const float4 *>(R + (16 * mt + 8 * hf + g) * kRStride + 16 * kp + 4 * c);
#pragma unroll
            for (int nt = 0; nt < 2; nt++)
                sb[nt] = __ldg(reinterpret_cast<const float4 *>(S + (32 * wq + 8 * (2 * nh + nt) + g) * kD + 16 * kp + 4 * c));
#pragma unroll
            for (int ks = 0; ks < 2; ks++) {
                uint32_t ah[2][4], al[2][4], bh[2][2], bl[2][2];
#pragma unroll
                for (int mt = 0; mt < 2; mt++) {
                    // a0: (row g, k c), a1: (row g + 8, k c), a2: (row g, k c + 4), a3: (row g + 8, k c + 4)
                    tf32_split(f4at(ra[mt][0], 2 * ks), ah[mt][0], al[mt][0]);
                    tf32_split(f4at(ra[mt][1], 2 * ks), ah[mt][1], al[mt][1]);
                    tf32_split(f4at(ra[mt][0], 2 * ks + 1), ah[mt][2], al[mt][2]);
                    tf32_split(f4at(ra[mt][1], 2 * ks + 1), ah[mt][3], al[mt][3]);
                }
#pragma unroll
                for (int nt = 0; nt < 2; nt++) {  // b0: (k c, n g), b1: (k c + 4, n g)
                    tf32_split(f4at(sb[nt], 2 * ks), bh[nt][0], bl[nt][0]);
                    tf32_split(f4at(sb[nt], 2 * ks + 1), bh[nt][1], bl[nt][1]);
                }
#pragma unroll
                for (int mt = 0; mt < 2; mt++)
#pragma unroll
                    for (int nt = 0; nt < 2; nt++) {
                        mma_tf32(acc[mt][nt], al[mt], bh[nt][0], bh[nt][1]);
                        mma_tf32(acc[mt][nt], ah[mt], bl[nt][0], bl[nt][1]);
                        mma_tf32(acc[mt][nt], ah[mt], bh[nt][0], bh[nt][1]);
                    }
            }
        }
        // accumulator e of (mt, nt): row g (+8 for e >= 2), projection 8 (2 nh + nt) + 2 c + (e & 1)
#pragma unroll
        for (int mt = 0; mt < 2; mt++)
#pragma unroll
            for (int nt = 0; nt < 2; nt++)
#pragma unroll
                for (int e = 0; e < 4; e++)
                    word[mt][e >> 1] |= (acc[mt][nt][e] >= 0.0f ? 1u : 0u) << (8 * (2 * nh + nt) + 2 * c + (e & 1));
    }
    // the four lanes of a quad hold disjoint bits of the same rows
#pragma unroll
    for (int mt = 0; mt < 2; mt++)
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
            word[mt][hf] |= __shfl_xor_sync(0xffffffffu, word[mt][hf], 1);
            word[mt][hf] |= __shfl_xor_sync(0xffffffffu, word[mt][hf], 2);
        }
    const int mt = c >> 1, hf = c & 1, row = 16 * mt + 8 * hf + g;
    const uint32_t w = c == 0 ? word[0][0] : c == 1 ? word[0][1] : c == 2 ? word[1][0] : word[1][1];
    if (row < n_valid) reinterpret_cast<uint32_t *>(rec0 + static_cast<size_t>(row) * (kJl / 8))[wq] = w;
}

// Quantize and store one key vector held by four lanes (this lane's rotated
// coordinates [32 q, 32 q + 32) in y); `store` is false for rows past the
// block's end (the lanes still run so that their exchanges stay warp-uniform).
template <int KB, bool QJL>
__device__ __forceinline__ void key_tail(const CompressParams &p, float (&y)[kQ], int q, int b, int h, int pos,
                                         bool store, float *Rsm = nullptr, int row = 0) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kQ; i++) m = fmaxf(m, fabsf(y[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const float r = m > 0.0f ? __frcp_rn(m) : 0.0f;
    constexpr float half_cells = static_cast<float>(1 << (KB - 1));
    constexpr float top = static_cast<float>((1 << KB) - 1);
    uint32_t w[KB];
#pragma unroll
    for (int j = 0; j < KB; j++) w[j] = 0;
#pragma unroll
    for (int i = 0; i < kQ; i++) {
        const float v = __fmul_rn(y[i], r);
        // round(v + 1) 2^(KB-1) = round(v 2^(KB-1) + 2^(KB-1)): scaling by a
        // power of two commutes with the rounding (v + 1 is never subnormal)
        float u = __fmaf_rn(v, half_cells, half_cells);
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
    if (store) {
        store_quarter_record<KB>(p.kcodes + static_cast<size_t>(b) * p.kblock + p.koff[h] +
                                     static_cast<size_t>(pos) * (16 * KB) + q * (4 * KB), w);
        if (q == 0) p.kscale[(static_cast<size_t>(b) * p.H + h) * p.capacity + pos] = m;
    }
    if constexpr (QJL) {  // the residual for the block's sketch (block_sketch), and rho
        const float ss = residual_to_smem(Rsm, y, row, q);
        if (store && q == 0) p.qjl_norm[(static_cast<size_t>(b) * p.nq + p.qrank[h]) * p.capacity + pos] = sqrtf(ss);
    }
}

// Quantize and store one value vector held by four lanes (as key_tail); with
// QJLV also the sketch of the residual y - sigma c[code] (binary32 product and
// difference, c the centroids in cent_smem).
template <int VB, bool QJLV = false>
__device__ __forceinline__ void value_tail(const CompressParams &p, float (&y)[kQ], const float *thr_smem, int q,
                                           int b, int h, int pos, bool store, const float *cent_smem = nullptr,
                                           float *Rsm = nullptr, int row = 0) {
    // pairwise tree of squares in index order: this lane's 32 give one of the
    // four subtrees two levels under the root; the root adds
    // (q0 + q1) + (q2 + q3)
    float s[kQ / 2];
#pragma unroll
    for (int j = 0; j < kQ / 2; j++)
        s[j] = __fadd_rn(__fmul_rn(y[2 * j], y[2 * j]), __fmul_rn(y[2 * j + 1], y[2 * j + 1]));
#pragma unroll
    for (int len = kQ / 2; len > 1; len >>= 1) {
#pragma unroll
        for (int j = 0; j < len / 2; j++) s[j] = __fadd_rn(s[2 * j], s[2 * j + 1]);
    }
    float t = s[0];
#pragma unroll
    for (int x = 1; x <= 2; x <<= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, t, x);
        t = (q & x) ? __fadd_rn(o, t) : __fadd_rn(t, o);
    }
    const float sigma = __fsqrt_rn(__fmul_rn(t, 1.0f / kD));  // /d exact (power of two)
    const float r = sigma > 0.0f ? __frcp_rn(sigma) : 0.0f;
    uint32_t w[VB];
#pragma unroll
    for (int j = 0; j < VB; j++) w[j] = 0;
    if constexpr (VB <= 4) {
        float th[(1 << VB) - 1];
#pragma unroll
        for (int j = 0; j < (1 << VB) - 1; j++) th[j] = thr_smem[j];
#pragma unroll
        for (int i = 0; i < kQ; i++) {
            const float u = __fmul_rn(y[i], r);
            const uint32_t k = search_reg<VB>(u, th, 0u);
            put_code<VB>(w, i, k);
            if constexpr (QJLV) y[i] = __fsub_rn(y[i], __fmul_rn(sigma, cent_smem[k]));
        }
    } else {
#pragma unroll
        for (int i = 0; i < kQ; i++) {
            const float u = __fmul_rn(y[i], r);
            const uint32_t k = search_smem<VB>(u, thr_smem);
            put_code<VB>(w, i, k);
            if constexpr (QJLV) y[i] = __fsub_rn(y[i], __fmul_rn(sigma, cent_smem[k]));
        }
    }
    if (store) {
        store_quarter_record<VB>(p.vcodes + static_cast<size_t>(b) * p.vblock + p.voff[h] +
                                     static_cast<size_t>(pos) * (16 * VB) + q * (4 * VB), w);
        if (q == 0) p.vscale[(static_cast<size_t>(b) * p.H + h) * p.capacity + pos] = sigma;
    }
    if constexpr (QJLV) {
        const float ss = residual_to_smem(Rsm, y, row, q);
        if (store && q == 0) p.vqjl_norm[(static_cast<size_t>(b) * p.nv + p.vrank[h]) * p.capacity + pos] = sqrtf(ss);
    }
}

// One key vector of the compress path: rotate, then quantize.
template <int KB, bool QJL>
__device__ __noinline__ void key_vector(const CompressParams &p, const uint8_t *qrow, const uint32_t *in_mask,
                                        const float *out_scale, int q, int b, int h, int pos, bool store,
                                        float *Rsm, int row) {
    float y[kQ];
    load_rotate(qrow, in_mask, out_scale, q, y);
    key_tail<KB, QJL>(p, y, q, b, h, pos, store, Rsm, row);
}

template <int VB, bool QJLV>
__device__ __noinline__ void value_vector(const CompressParams &p, const uint8_t *qrow, const uint32_t *in_mask,
                                          const float *out_scale, const float *thr_smem, const float *cent_smem,
                                          int q, int b, int h, int pos, bool store, float *Rsm, int row) {
    float y[kQ];
    load_rotate(qrow, in_mask, out_scale, q, y);
    value_tail<VB, QJLV>(p, y, thr_smem, q, b, h, pos, store, cent_smem, Rsm, row);
}

// Stage the rows of block `blk` (t-block fastest, then selected head, then
// batch) of one group (0: K, 1: V) into `dst`, by the group's 128 threads.
__device__ __forceinline__ void stage_block(const CompressParams &p, int n_tblk, int blk, int group, int gtid,
                                            uint8_t *dst) {
    const int tb = blk % n_tblk, rest = blk / n_tblk;
    const int h = p.sel[rest % p.n_sel], b = rest / p.n_sel;
    const int t0 = tb * kTok, nt = min(kTok, p.T - t0);
    const uint16_t *src = (group ? p.V : p.K) + b * p.sb + h * p.sh;
#pragma unroll
    for (int i = 0; i < kTok * 16 / 128; i++) {
        const int idx = gtid + 128 * i, r = idx >> 4, ch = idx & 15;
        if (r < nt)
            cp_async16(dst + r * kRow + (ch >> 2) * kQuarter + (ch & 3) * 16,
                       src + static_cast<int64_t>(t0 + r) * p.st + ch * 8);
    }
}

__global__ void __launch_bounds__(kThreads, 3)
    compress_kernel(const __grid_constant__ CompressParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    // sign masks and output scales, 16-byte chunk c of quarter q at chunk
    // 4 c + q: the four quarters a warp reads together sit in four bank groups
    uint32_t *in_mask = reinterpret_cast<uint32_t *>(smem + 4 * kGroupBuf);  // [64]
    float *out_scale = reinterpret_cast<float *>(in_mask + kD / 2);          // [128]
    float *thr = out_scale + kD;                                             // [kCbTotal]
    float *cent = thr + kCbTotal;                                            // [kCbTotal]
    // residual rows of the current block, keys then values, when the launch sketches them
    float *R_key = cent + kCbTotal;
    float *R_val = R_key + (p.nq > 0 ? kTok * kRStride : 0);

    const int n_tblk = (p.T + kTok - 1) / kTok;
    const int n_blk = n_tblk * p.n_sel * p.B;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = warp >> 2, gtid = threadIdx.x & 127, q = lane & 3;
    const int r = (warp & 3) * 8 + (lane >> 2);  // this vector's row in the block
    uint8_t *bufs = smem + group * 2 * kGroupBuf;
    int blk = blockIdx.x;
    if (blk < n_blk) stage_block(p, n_tblk, blk, group, gtid, bufs);
    cp_async_commit();
    if (threadIdx.x < kD / 2) {
        const int i = 2 * threadIdx.x;
        const uint32_t s0 = (p.sign_bits[i >> 5] >> (i & 31)) & 1u;
        const uint32_t s1 = (p.sign_bits[(i + 1) >> 5] >> ((i + 1) & 31)) & 1u;
        const int t = threadIdx.x;  // coordinates 2t, 2t + 1: quarter t / 16, chunk (t / 4) % 4
        in_mask[((((t >> 2) & 3) * 4) + (t >> 4)) * 4 + (t & 3)] = (s0 << 15) | (s1 << 31);
    }
    if (threadIdx.x < kD) {
        const int i = threadIdx.x;
        const uint32_t s = (p.sign_bits[i >> 5] >> (i & 31)) & 1u;
        out_scale[((((i >> 2) & 7) * 4) + (i >> 5)) * 4 + (i & 3)] = s ? -p.inv_sqrt_d : p.inv_sqrt_d;
    }
    for (int j = threadIdx.x; j < kCbTotal; j += kThreads) {
        thr[j] = p.thr[j];
        cent[j] = p.cent[j];
    }
    __syncthreads();  // tables written

    for (int it = 0; blk < n_blk; blk += gridDim.x, it++) {
        const int next = blk + gridDim.x;
        if (next < n_blk) stage_block(p, n_tblk, next, group, gtid, bufs + ((it + 1) & 1) * kGroupBuf);
        cp_async_commit();
        cp_async_wait<1>();
        group_sync(group);  // block `blk` staged and visible to the group

        const int tb = blk % n_tblk, rest = blk / n_tblk;
        const int h = p.sel[rest % p.n_sel], b = rest / p.n_sel;
        const int t0 = tb * kTok, nt = min(kTok, p.T - t0);
        const bool store = r < nt;
        const int pos = p.t_begin + t0 + r;
        const uint8_t *qrow = bufs + (it & 1) * kGroupBuf + r * kRow + q * kQuarter;
        if (group == 0) {
            const bool qj = p.qrank[h] >= 0;
            switch (p.kbits[h] * 2 + (qj ? 1 : 0)) {
#define TQ_KEY_CASE(KB)                                                                                 \
    case 2 * KB: key_vector<KB, false>(p, qrow, in_mask, out_scale, q, b, h, pos, store, R_key, r); break;   \
    case 2 * KB + 1: key_vector<KB, true>(p, qrow, in_mask, out_scale, q, b, h, pos, store, R_key, r); break;
                TQ_KEY_CASE(1) TQ_KEY_CASE(2) TQ_KEY_CASE(3) TQ_KEY_CASE(4)
                TQ_KEY_CASE(5) TQ_KEY_CASE(6) TQ_KEY_CASE(7) TQ_KEY_CASE(8)
#undef TQ_KEY_CASE
                default: break;
            }
        } else {
            const int vb = p.vbits[h];
            const float *t = thr + cb_off(vb), *c = cent + cb_off(vb);
            const bool qv = p.vrank[h] >= 0;
            switch (vb * 2 + (qv ? 1 : 0)) {
#define TQ_VAL_CASE(VB)                                                                                         \
    case 2 * VB: value_vector<VB, false>(p, qrow, in_mask, out_scale, t, c, q, b, h, pos, store, R_val, r); break;   \
    case 2 * VB + 1: value_vector<VB, true>(p, qrow, in_mask, out_scale, t, c, q, b, h, pos, store, R_val, r); break;
                TQ_VAL_CASE(1) TQ_VAL_CASE(2) TQ_VAL_CASE(3) TQ_VAL_CASE(4)
                TQ_VAL_CASE(5) TQ_VAL_CASE(6) TQ_VAL_CASE(7) TQ_VAL_CASE(8)
#undef TQ_VAL_CASE
                default: break;
            }
        }
        // sketched heads: the group's four warps project the block's 32
        // residuals (rows in R_key / R_val), 32 projections each
        const int rank = group == 0 ? p.qrank[h] : p.vrank[h];
        if (rank >= 0) {
            group_sync(group);  // every residual row written
            const size_t rec = (static_cast<size_t>(b) * (group == 0 ? p.nq : p.nv) + rank) * p.capacity +
                               p.t_begin + t0;
            block_sketch(group == 0 ? R_key : R_val, p.S, warp & 3, lane,
                         (group == 0 ? p.qjl_signs : p.vqjl_signs) + rec * (kJl / 8), nt);
        }
        group_sync(group);  // the group is done with this buffer (and its residual rows) before they are restaged
    }
}

// ------------------------------------------------------------------ requantize
// Code i (0..31) of a lane's quarter record, runtime width: byte loads so that
// nothing past the quarter is read.
__device__ __forceinline__ uint32_t quarter_code(const uint8_t *rec, int i, int bits) {
    const int bit = i * bits, by = bit >> 3, sh = bit & 7;
    uint32_t v = __ldg(rec + by);
    if (sh + bits > 8) v |= static_cast<uint32_t>(__ldg(rec + by + 1)) << 8;
    return (v >> sh) & ((1u << bits) - 1u);
}

// One demoted key vector (four lanes): the source record's reconstruction
// m * level(code) in binary32 (level = (2 code + 1) 2^-b - 1, exact), then the
// destination width's quantizer.
template <int KB>
__device__ __noinline__ void key_requant(const RequantParams &p, int q, int b, int h, int sp, int dp, bool store) {
    const int sb = p.skbits[h];
    const uint8_t *rec = p.skcodes + static_cast<size_t>(b) * p.skblock + p.skoff[h] +
                         static_cast<size_t>(sp) * (16 * sb) + q * (4 * sb);
    const float m = __ldg(p.skscale + (static_cast<size_t>(b) * p.dst.H + h) * p.scapacity + sp);
    const float inv_cells = __uint_as_float(static_cast<uint32_t>(127 - sb) << 23);  // 2^-b
    float y[kQ];
#pragma unroll
    for (int i = 0; i < kQ; i++) {
        const float lev = __fadd_rn(__fmul_rn(static_cast<float>(2 * quarter_code(rec, i, sb) + 1), inv_cells), -1.0f);
        y[i] = __fmul_rn(m, lev);
    }
    key_tail<KB, false>(p.dst, y, q, b, h, dp, store);
}

// One demoted value vector: sigma * centroid[code] in binary32, then the
// destination width's quantizer.
template <int VB>
__device__ __noinline__ void value_requant(const RequantParams &p, const float *cent, const float *thr_smem, int q,
                                           int b, int h, int sp, int dp, bool store) {
    const int sb = p.svbits[h];
    const uint8_t *rec = p.svcodes + static_cast<size_t>(b) * p.svblock + p.svoff[h] +
                         static_cast<size_t>(sp) * (16 * sb) + q * (4 * sb);
    const float sg = __ldg(p.svscale + (static_cast<size_t>(b) * p.dst.H + h) * p.scapacity + sp);
    const float *c = cent + cb_off(sb);
    float y[kQ];
#pragma unroll
    for (int i = 0; i < kQ; i++) y[i] = __fmul_rn(sg, c[quarter_code(rec, i, sb)]);
    value_tail<VB>(p.dst, y, thr_smem, q, b, h, dp, store);
}

// One CTA per 32-token block of (batch, head): warps 0-3 keys, 4-7 values,
// four lanes per vector (the compress kernel's layout and quantizers).
__global__ void __launch_bounds__(kThreads) requantize_kernel(const __grid_constant__ RequantParams p) {
    __shared__ float cent[kCbTotal], thr[kCbTotal];
    for (int j = threadIdx.x; j < kCbTotal; j += kThreads) {
        cent[j] = p.centroid[j];
        thr[j] = p.dst.thr[j];
    }
    __syncthreads();
    const int n_tblk = (p.dst.T + kTok - 1) / kTok;
    const int blk = blockIdx.x;
    const int tb = blk % n_tblk, rest = blk / n_tblk;
    const int h = rest % p.dst.H, b = rest / p.dst.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = warp >> 2, q = lane & 3;
    const int r = (warp & 3) * 8 + (lane >> 2);
    const int t = tb * kTok + r;
    const bool store = t < p.dst.T;
    const int sp = p.s_t0 + min(t, p.dst.T - 1);  // rows past the end re-read the last token
    const int dp = p.dst.t_begin + t;
    if (group == 0) {
        switch (p.dst.kbits[h]) {
#define TQ_RQ_KEY(KB) \
    case KB: key_requant<KB>(p, q, b, h, sp, dp, store); break;
            TQ_RQ_KEY(1) TQ_RQ_KEY(2) TQ_RQ_KEY(3) TQ_RQ_KEY(4) TQ_RQ_KEY(5) TQ_RQ_KEY(6) TQ_RQ_KEY(7) TQ_RQ_KEY(8)
#undef TQ_RQ_KEY
            default: break;
        }
    } else {
        const int vb = p.dst.vbits[h];
        const float *tv = thr + cb_off(vb);
        switch (vb) {
#define TQ_RQ_VAL(VB) \
    case VB: value_requant<VB>(p, cent, tv, q, b, h, sp, dp, store); break;
            TQ_RQ_VAL(1) TQ_RQ_VAL(2) TQ_RQ_VAL(3) TQ_RQ_VAL(4) TQ_RQ_VAL(5) TQ_RQ_VAL(6) TQ_RQ_VAL(7) TQ_RQ_VAL(8)
#undef TQ_RQ_VAL
            default: break;
        }
    }
}

constexpr size_t compress_smem() { return 4 * kGroupBuf + (kD / 2) * 4 + kD * 4 + 2 * kCbTotal * 4; }

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
    if (orig && p.Q) {  // x = Q^T y, binary32 products in index order
        for (int j = 0; j < kD; j++) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kD; i++) acc = fmaf(__ldg(p.Q + static_cast<size_t>(i) * kD + j), y[i], acc);
            orig[o + j] = acc;
        }
    } else if (orig) {
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
    // launches with sketched keys (values) also hold the block's key (value)
    // residuals: three CTAs per SM with one of the two, two with both
    const size_t smem = compress_smem() + (p.nq > 0 ? kRSmem : 0) + (p.nv > 0 ? kRSmem : 0);
    const bool sketch = p.nq > 0 && p.nv > 0;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(compress_smem() + 2 * kRSmem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // persistent: three (two) CTAs per SM, each group looping over 32-token blocks
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long n_blk = static_cast<long long>((p.T + kTok - 1) / kTok) * p.n_sel * p.B;
    if (n_blk == 0) return cudaSuccess;
    const int grid = static_cast<int>(std::min<long long>(n_blk, (sketch ? 2LL : 3LL) * sms));
    compress_kernel<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_requantize(const RequantParams &p, cudaStream_t s) {
    const long long n_blk = static_cast<long long>((p.dst.T + kTok - 1) / kTok) * p.dst.H * p.dst.B;
    if (n_blk == 0) return cudaSuccess;
    if (n_blk > 0x7fffffffLL) return cudaErrorInvalidValue;
    requantize_kernel<<<static_cast<unsigned>(n_blk), kThreads, 0, s>>>(p);
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
