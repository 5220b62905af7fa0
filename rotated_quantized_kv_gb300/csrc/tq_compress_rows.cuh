// tq_compress_rows.cuh -- compression of key or value vectors with one thread
// per 128-dimension slice, for launches without QJL sketches (head_dim 128,
// and 256 / 512 as NH = 2 / 4 slices); instantiated per NH by
// tq_compress_rows*.cu.
//
// Method and format: as compress_kernel (tq_compress.cu): "turboquant-mlx"
// (TurboQuant-MLX v2.0 README), "Walsh-Hadamard Rotation" (SRHT D H D / sqrt(d));
// "TurboMOQ", "Architecture" (keys: symmetric grid, values: Gaussian Lloyd-Max
// codebook, 1-8 bits per head) and "Project Structure" (bit packing).  Every
// rounding step is the format's IEEE binary32 operation, so the codes are the
// same bits as the oracle's.
//
// Design (GB300): a thread holds its whole vector in 64 float2 registers, pair
// m = (coordinate m, coordinate m + 64).  Butterfly stages h = 1..32 pair
// registers m and m + h, so one packed f32x2 add and one packed f32x2
// subtract (Blackwell's add/sub.rn.f32x2: two independent IEEE operations)
// do two butterflies each; stage 64 pairs the two halves of each register.
// The output scale, the key grid arithmetic and the value quotient y / sigma
// are packed f32x2 operations too, and the pairwise sum of squares runs as
// two index-order trees of 64 (packed) joined at the root.  No exchanges
// between lanes.  A warp compresses 32 consecutive tokens of one (batch,
// head): their fp16 rows are staged in shared memory with 16-byte cp.async
// copies (chunk c of row r at 16 (c ^ (r & 7)), so that the eight rows one
// 16-byte load phase reads fall in eight bank groups), double-buffered per
// warp, and each thread stores its record with 16-byte stores (16 b bytes per
// vector).  Kernels are specialised by the width of the heads they carry
// (keys and values launched separately), so each holds one quantizer.
//
// Head_dim 128 NH (NH = 2, 4): the NH threads of a vector sit 32 / NH lanes
// apart in one warp (lane = slice j * 32 / NH + token), each holding slice j
// (coordinates 128 j .. 128 j + 127) in the same register layout.  After the
// in-register stages h = 1..64, stage h = 128 (and 256) pairs slice j with
// slice j ^ 1 (j ^ 2): each thread takes its partner's register by a shuffle
// and forms fma(s, own, other) with s = +1 (lower slice: own + other) or -1
// (upper slice: other - own), which is the butterfly's one IEEE rounding.  The
// absmax and the last levels of the sum-of-squares tree (slices 2i + 1 onto
// 2i, then 4i + 2 onto 4i) go through the same shuffles, each pair added in
// the same order on both sides.  A d-dim record is the NH 128-dim records of
// the slices one after another (the LSB-first stream cut at dims 128 j falls on
// a byte boundary), so each thread stores its slice's 16 b bytes.
//
// Head_dim 64 (NP = 2): a thread takes two consecutive tokens, the first in
// the low halves of its 64 register pairs and the second in the high halves
// (the staged row is the two tokens' 64-dim vectors one after the other).  The
// stages h = 1..32 run as at 128 dims on both at once; stage 64 and the root of
// the sum-of-squares tree, which would join the halves, are left out, and each
// half gets its own absmax or sigma.  The two 64-dim records are adjacent in
// the segment, so the thread's 128 codes are both records in order (one
// 16 b-byte store when both tokens exist and the first position is even).
#pragma once

#include <algorithm>

#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tqk {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kRowBytes = 256;            // 128 fp16 coordinates
constexpr int kWarpBuf = 32 * kRowBytes;  // one staged block of 32 rows
constexpr int kMaskStride = 68;           // words per slice of the input sign masks (64 + pad)
constexpr int kPairStride = 132;          // floats per slice of the output scales (128 + pad)

// Packed binary32 pairs: two independent IEEE operations per instruction.
// A packed product that feeds a packed sum can still be fused into one packed
// multiply-add by the compiler (measured: the explicit rounding modifier does
// not prevent it), so no product below ever feeds a sum directly: every chain
// is add/sub only, or multiply then multiply / fma / compare.
#define TQ_F32X2_BINARY(NAME, OP)                                                              \
    __device__ __forceinline__ float2 NAME(float2 a, float2 b) {                               \
        float2 r;                                                                              \
        asm("{.reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n" OP \
            " rr, ra, rb;\n mov.b64 {%0, %1}, rr;}"                                          \
            : "=f"(r.x), "=f"(r.y)                                                             \
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                         \
        return r;                                                                              \
    }
TQ_F32X2_BINARY(fadd2, " add.rn.f32x2")
TQ_F32X2_BINARY(fsub2, " sub.rn.f32x2")
TQ_F32X2_BINARY(fmul2, " mul.rn.f32x2")
TQ_F32X2_BINARY(fadd2_rm, " add.rm.f32x2")
#undef TQ_F32X2_BINARY

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{.reg .b64 ra, rb, rc, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rr, ra, rb, rc;\n mov.b64 {%0, %1}, rr;}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// max(a, b, c) in one instruction (order-free: the absmax needs no fixed order)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t lds32r(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
// #{k : thr_k < u} from the 4-bit table (RowsParams::bucket4)
__device__ __forceinline__ uint32_t bucket4_code(uint32_t tab, float u) {
    const uint32_t ub = __float_as_uint(u);
    const uint32_t e = lds32r(tab + ((ub >> 21) << 2));
    const uint32_t x = (ub ^ static_cast<uint32_t>(static_cast<int32_t>(ub) >> 31)) & 0x1FFFFFu;
    return (e >> 21) + ((e & 0x1FFFFFu) < x ? 1u : 0u);
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}

// Stage the fp16 rows of block `blk` ((b, head of the list, block of tokens),
// token block fastest) into this warp's buffer: row r is slice r / (32 / NH)
// of token r mod (32 / NH) of the block (NP = 2: tokens 2 r, 2 r + 1).
template <int NH, int NP>
__device__ __forceinline__ void stage_rows(const RowsParams &p, int n_tblk, int blk, uint8_t *buf, int lane) {
    constexpr int TPW = 32 * NP / NH;
    const int tb = blk % n_tblk, rest = blk / n_tblk;
    const int h = p.head[rest % p.n_heads], b = rest / p.n_heads;
    const int t0 = tb * TPW, nt = min(TPW, p.T - t0);
    const uint16_t *src = p.X + b * p.sb + h * p.sh + static_cast<int64_t>(t0) * p.st;
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const int idx = lane + 32 * i, r = idx >> 4, c = idx & 15;
        if constexpr (NP == 2) {
            const int tok = 2 * r + (c >> 3);
            if (tok < nt)
                cp_async16(buf + r * kRowBytes + 16 * (c ^ (r & 7)),
                           src + static_cast<int64_t>(tok) * p.st + 8 * (c & 7));
        } else {
            const int tok = r % TPW, sl = r / TPW;
            if (tok < nt)
                cp_async16(buf + r * kRowBytes + 16 * (c ^ (r & 7)),
                           src + static_cast<int64_t>(tok) * p.st + kD * sl + 8 * c);
        }
    }
}

// Code i (0..127) at bits [B i, B i + B) of the record's 4 B words.
template <int B>
__device__ __forceinline__ void put(uint32_t (&w)[4 * B], int i, uint32_t k) {
    const int bit = i * B, wi = bit >> 5, sh = bit & 31;
    w[wi] += k << sh;  // codes never overlap: an add (one shift-and-add instruction) is the or
    if (sh + B > 32) w[wi + 1] += k >> (32 - sh);
}

// Key codes are put as kKeyLo + code (a float bit pattern, see the key
// quantizer); word j of the record then holds the sum of the kKeyLo parts of
// its codes on top of the codes, modulo 2^32.  kKeyLo + code carries nothing
// out of its low 10 bits (code < 512), so the parts shifted out of a word
// (sh + B > 32, a right shift by less than B <= 8) are kKeyLo >> s exactly.
constexpr uint32_t kKeyLo = 0x4B000000u + 512u;
template <int B>
__host__ __device__ constexpr uint32_t key_offset_word(int j) {
    uint32_t c = 0;
    for (int i = 0; i < 128; i++) {
        const int bit = i * B, wi = bit >> 5, sh = bit & 31;
        if (wi == j) c += kKeyLo << sh;
        if (sh + B > 32 && wi + 1 == j) c += kKeyLo >> (32 - sh);
    }
    return c;
}

template <int NH>
__host__ __device__ constexpr size_t rows_smem_bytes(bool val_table) {
    return kWarps * 2 * kWarpBuf + NH * kMaskStride * 4 + NH * kPairStride * 4 + 256 * 4 +
           (val_table ? kRowsBuckets * 8 : 0);
}

template <int BITS, bool VAL, int NH, int NP = 1>
__global__ void __launch_bounds__(kThreads, 3) compress_rows_kernel(const __grid_constant__ RowsParams p) {
    static_assert(NP == 1 || NH == 1, "token pairs: head_dim 64");
    constexpr int TPW = 32 * NP / NH;  // tokens of a warp block
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t *in_mask = reinterpret_cast<uint32_t *>(smem + kWarps * 2 * kWarpBuf);  // [NH][kMaskStride]
    float *out_pair = reinterpret_cast<float *>(in_mask + NH * kMaskStride);         // [NH][kPairStride]
    float *thr = out_pair + NH * kPairStride;                                        // [255]
    uint2 *vtab = reinterpret_cast<uint2 *>(thr + 256);                             // [1024] (values, <= 3 bits)
    for (int i = threadIdx.x; i < NH * 64; i += kThreads) in_mask[(i >> 6) * kMaskStride + (i & 63)] = p.in_mask[i];
    for (int i = threadIdx.x; i < NH * kD; i += kThreads) {
        const int sl = i >> 7, k = i & 127;  // slice, then pairs (m, m + 64) of its scales
        out_pair[sl * kPairStride + k] = p.out_scale[kD * sl + (k >> 1) + 64 * (k & 1)];
    }
    for (int i = threadIdx.x; i < 255; i += kThreads) thr[i] = p.thr[i];
    if constexpr (VAL && BITS <= 3)
        for (int i = threadIdx.x; i < kRowsBuckets; i += kThreads) vtab[i] = make_uint2(p.bucket[i].t, p.bucket[i].k);
    if constexpr (VAL && BITS == 4)
        if (p.bucket4_ok)
            for (int i = threadIdx.x; i < kRowsBuckets; i += kThreads)
                vtab[i] = make_uint2(p.bucket4[2 * i], p.bucket4[2 * i + 1]);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sl = lane / TPW;  // this thread's slice
    const uint32_t *im = in_mask + sl * kMaskStride;
    const float *op = out_pair + sl * kPairStride;
    uint8_t *bufs = smem + warp * 2 * kWarpBuf;
    const int n_tblk = (p.T + TPW - 1) / TPW;
    const int n_blk = n_tblk * p.n_heads * p.B;
    const int gw = blockIdx.x * kWarps + warp, nw = gridDim.x * kWarps;
    if (gw < n_blk) stage_rows<NH, NP>(p, n_tblk, gw, bufs, lane);
    asm volatile("cp.async.commit_group;\n" ::);

    for (int blk = gw, it = 0; blk < n_blk; blk += nw, it++) {
        const int next = blk + nw;
        if (next < n_blk) stage_rows<NH, NP>(p, n_tblk, next, bufs + ((it + 1) & 1) * kWarpBuf, lane);
        asm volatile("cp.async.commit_group;\n" ::);
        asm volatile("cp.async.wait_group 1;\n" ::: "memory");
        __syncwarp();
        const int tb = blk % n_tblk, rest = blk / n_tblk;
        const int h = p.head[rest % p.n_heads], b = rest / p.n_heads;
        const int t = NP == 2 ? tb * TPW + 2 * lane : tb * TPW + lane % TPW;  // (the first token of the pair)
        const uint8_t *row = bufs + (it & 1) * kWarpBuf + lane * kRowBytes;

        // ---- load, input sign flip on the fp16 bits, widen: chunks c and
        // c + 8 (coordinates 8c.. and 64 + 8c..) are permuted into half2 pairs
        // (m, m + 64) that widen straight into the register pairs
        float2 a[64];
#pragma unroll
        for (int c = 0; c < 8; c++) {
            const uint4 v0 = *reinterpret_cast<const uint4 *>(row + 16 * (c ^ (lane & 7)));
            const uint4 v1 = *reinterpret_cast<const uint4 *>(row + 16 * ((c + 8) ^ (lane & 7)));
            const uint4 m0 = *reinterpret_cast<const uint4 *>(im + 4 * c);
            const uint4 m1 = *reinterpret_cast<const uint4 *>(im + 4 * (c + 8));
            const uint32_t w0[4] = {v0.x ^ m0.x, v0.y ^ m0.y, v0.z ^ m0.z, v0.w ^ m0.w};
            const uint32_t w1[4] = {v1.x ^ m1.x, v1.y ^ m1.y, v1.z ^ m1.z, v1.w ^ m1.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int i = 8 * c + 2 * e;  // pairs (i, i + 64) and (i + 1, i + 65)
                const uint32_t lo = prmt(w0[e], w1[e], 0x5410u), hi = prmt(w0[e], w1[e], 0x7632u);
                a[i] = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
                a[i + 1] = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
            }
        }
        __syncwarp();  // every lane has read its row: the buffer may be restaged

        // ---- butterflies h = 1..32 on register pairs (packed), then h = 64
#pragma unroll
        for (int hh = 1; hh < 64; hh <<= 1) {
#pragma unroll
            for (int m = 0; m < 64; m++) {
                if ((m & hh) == 0) {
                    const float2 u = a[m], v = a[m + hh];
                    a[m] = fadd2(u, v);
                    a[m + hh] = fsub2(u, v);
                }
            }
        }
        if constexpr (NP == 1) {
#pragma unroll
            for (int m = 0; m < 64; m++) {
                const float u = a[m].x, v = a[m].y;
                a[m].x = __fadd_rn(u, v);
                a[m].y = __fsub_rn(u, v);
            }
        }
        // h = 128 (256): the same register of slice sl ^ x, x = 1 (2), from
        // lane ^ x TPW; fma(+-1, own, other) rounds the exact sum once
#pragma unroll
        for (int x = 1; x < NH; x <<= 1) {
            const float sg = (sl & x) ? -1.0f : 1.0f;
#pragma unroll
            for (int m = 0; m < 64; m++) {
                const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, a[m].x, x * TPW),
                                             __shfl_xor_sync(0xffffffffu, a[m].y, x * TPW));
                a[m] = ffma2(a[m], make_float2(sg, sg), o);
            }
        }
        // output sign flip and binary32(1/sqrt(d)): one rounded multiply each
        // (op[m] = the scales of coordinates m and m + 64 of the slice)
#pragma unroll
        for (int m = 0; m < 64; m += 2) {
            const float4 sc = *reinterpret_cast<const float4 *>(op + 2 * m);
            a[m] = fmul2(a[m], make_float2(sc.x, sc.y));
            a[m + 1] = fmul2(a[m + 1], make_float2(sc.z, sc.w));
        }

        uint32_t w[4 * BITS];
#pragma unroll
        for (int j = 0; j < 4 * BITS; j++) w[j] = 0u;
        float scale, scale_b = 0.0f;  // scale_b: the pair's second token (NP = 2)
        if constexpr (!VAL) {
            // ---- keys: m = max |y|, v = y * binary32(1/m), u = round(v + 1) 2^(b-1),
            // code = clamp(floor(u), 0, 2^b - 1)
            float mx = 0.0f, mxb = 0.0f;
            if constexpr (NP == 2) {
#pragma unroll
                for (int m = 0; m < 64; m += 2) {
                    mx = fmax3(mx, fabsf(a[m].x), fabsf(a[m + 1].x));
                    mxb = fmax3(mxb, fabsf(a[m].y), fabsf(a[m + 1].y));
                }
            } else {
#pragma unroll
                for (int m = 0; m < 64; m++) mx = fmax3(mx, fabsf(a[m].x), fabsf(a[m].y));
            }
#pragma unroll
            for (int x = 1; x < NH; x <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, x * TPW));
            scale = mx;
            scale_b = mxb;
            const float r = mx > 0.0f ? __frcp_rn(mx) : 0.0f;
            const float rb = NP == 2 ? (mxb > 0.0f ? __frcp_rn(mxb) : 0.0f) : r;
            constexpr float hc = static_cast<float>(1 << (BITS - 1));
            // v = y r lies in [-1, 1]: r = binary32(1/m) is within 2^-24 of 1/m
            // and |y| <= m, so |y r| <= 1 + 2^-24 rounds to at most 1.  Hence
            // u = round(v + 1) 2^(b-1) >= 0 and only the top clamp can act (at
            // v = 1).  floor(u): the round-down of u + 2^23 + 512 has the exponent
            // of 2^23, so its bit pattern is kLo + floor(u).
            constexpr float kMagic = 8388608.0f + 512.0f;
            constexpr uint32_t kHi = kKeyLo + (1u << BITS) - 1u;
#pragma unroll
            for (int m = 0; m < 64; m++) {
                const float2 v = fmul2(a[m], make_float2(r, rb));
                // fma(v, 2^(b-1), 2^(b-1)) is round(v + 1) 2^(b-1): scaling by a
                // power of two commutes with the rounding
                const float2 u = ffma2(v, make_float2(hc, hc), make_float2(hc, hc));
                const float2 f = fadd2_rm(u, make_float2(kMagic, kMagic));
                // kLo + code, placed as is: the words take off the kLo parts below
                put<BITS>(w, m, min(__float_as_uint(f.x), kHi));
                put<BITS>(w, m + 64, min(__float_as_uint(f.y), kHi));
            }
#pragma unroll
            for (int j = 0; j < 4 * BITS; j++) w[j] -= key_offset_word<BITS>(j);
        } else {
            // ---- values: sigma = sqrt(pairwise-tree sum of y^2 in index order / d),
            // u = y * binary32(1/sigma), code = #{k : thr_k < u}
            // first level scalar: the compiler fuses a packed multiply into a
            // packed add (one rounding instead of two), which the scalar _rn
            // intrinsics rule out; the later levels are additions only
            float2 s[32];
#pragma unroll
            for (int j = 0; j < 32; j++) {
                s[j].x = __fadd_rn(__fmul_rn(a[2 * j].x, a[2 * j].x), __fmul_rn(a[2 * j + 1].x, a[2 * j + 1].x));
                s[j].y = __fadd_rn(__fmul_rn(a[2 * j].y, a[2 * j].y), __fmul_rn(a[2 * j + 1].y, a[2 * j + 1].y));
            }
#pragma unroll
            for (int len = 32; len > 1; len >>= 1) {
#pragma unroll
                for (int j = 0; j < len / 2; j++) s[j] = fadd2(s[2 * j], s[2 * j + 1]);
            }
            // NP = 2: the two halves' trees are the two tokens' sums (no root join)
            float tot = NP == 2 ? s[0].x : __fadd_rn(s[0].x, s[0].y);
            // blocks of 256 (512) coordinates: slices (2i, 2i + 1), then (4i, 4i + 2)
#pragma unroll
            for (int x = 1; x < NH; x <<= 1) tot = __fadd_rn(tot, __shfl_xor_sync(0xffffffffu, tot, x * TPW));
            constexpr float inv_d = 1.0f / (kD * NH / NP);  // exact (a power of two)
            const float sigma = __fsqrt_rn(__fmul_rn(tot, inv_d));
            const float sigma_b = NP == 2 ? __fsqrt_rn(__fmul_rn(s[0].y, inv_d)) : sigma;
            scale = sigma;
            scale_b = sigma_b;
            const float r = sigma > 0.0f ? __frcp_rn(sigma) : 0.0f;
            const float rb = NP == 2 ? (sigma_b > 0.0f ? __frcp_rn(sigma_b) : 0.0f) : r;
            constexpr int NT = (1 << BITS) - 1;
            if constexpr (BITS <= 3) {
                // #{k : thr_k < u} from the bucket of u's top ten bits (sign,
                // exponent, one mantissa bit): every u in a bucket exceeds the
                // same k_base thresholds, and at most one threshold t_c lies in
                // the bucket (the host checks), so the count is k_base + [t_c < u]
                const uint32_t tab = static_cast<uint32_t>(__cvta_generic_to_shared(vtab));
#pragma unroll
                for (int m = 0; m < 64; m++) {
                    const float2 u = fmul2(a[m], make_float2(r, rb));
                    const uint2 e0 = lds64(tab + ((__float_as_uint(u.x) >> 22) << 3));
                    const uint2 e1 = lds64(tab + ((__float_as_uint(u.y) >> 22) << 3));
                    put<BITS>(w, m, e0.y + (__uint_as_float(e0.x) < u.x ? 1u : 0u));
                    put<BITS>(w, m + 64, e1.y + (__uint_as_float(e1.x) < u.y ? 1u : 0u));
                }
            } else if constexpr (BITS == 4) {
              if (p.bucket4_ok) {
                const uint32_t tab = static_cast<uint32_t>(__cvta_generic_to_shared(vtab));
#pragma unroll
                for (int m = 0; m < 64; m++) {
                    const float2 u = fmul2(a[m], make_float2(r, rb));
                    put<BITS>(w, m, bucket4_code(tab, u.x));
                    put<BITS>(w, m + 64, bucket4_code(tab, u.y));
                }
              } else {
                float th[NT];
#pragma unroll
                for (int j = 0; j < NT; j++) th[j] = thr[j];
#pragma unroll
                for (int m = 0; m < 64; m++) {
                    const float2 u = fmul2(a[m], make_float2(r, rb));
                    uint32_t k0 = 0, k1 = 0;
#pragma unroll
                    for (int st = 1 << (BITS - 1); st >= 1; st >>= 1) {
                        // threshold k + st - 1 for the current prefix k: a select
                        // tree over the candidates of this level
                        float t0 = th[st - 1], t1 = th[st - 1];
#pragma unroll
                        for (int c = 2 * st; c < (1 << BITS); c += 2 * st) {
                            t0 = (k0 >= static_cast<uint32_t>(c)) ? th[c + st - 1] : t0;
                            t1 = (k1 >= static_cast<uint32_t>(c)) ? th[c + st - 1] : t1;
                        }
                        k0 += (t0 < u.x) ? st : 0;
                        k1 += (t1 < u.y) ? st : 0;
                    }
                    put<BITS>(w, m, k0);
                    put<BITS>(w, m + 64, k1);
                }
              }
            } else {
#pragma unroll
                for (int m = 0; m < 64; m++) {
                    const float2 u = fmul2(a[m], make_float2(r, rb));
                    uint32_t k0 = 0, k1 = 0;
#pragma unroll
                    for (int st = 1 << (BITS - 1); st >= 1; st >>= 1) {
                        if (thr[k0 + st - 1] < u.x) k0 += st;
                        if (thr[k1 + st - 1] < u.y) k1 += st;
                    }
                    put<BITS>(w, m, k0);
                    put<BITS>(w, m + 64, k1);
                }
            }
        }
        if constexpr (NP == 2) {
            // the pair's two 8 b-byte records (t_begin even: 16-byte aligned)
            const int pos = p.t_begin + t;
            uint8_t *dst = p.codes + static_cast<size_t>(b) * p.block + p.off[h] + static_cast<size_t>(pos) * (8 * BITS);
            float *sc = p.scale + (static_cast<size_t>(b) * p.H + h) * p.capacity + pos;
            if (t + 1 < p.T) {
#pragma unroll
                for (int j = 0; j < BITS; j++)
                    reinterpret_cast<uint4 *>(dst)[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                sc[0] = scale;
                sc[1] = scale_b;
            } else if (t < p.T) {  // an unpaired last token
#pragma unroll
                for (int j = 0; j < BITS; j++) reinterpret_cast<uint2 *>(dst)[j] = make_uint2(w[2 * j], w[2 * j + 1]);
                sc[0] = scale;
            }
        } else if (t < p.T) {
            const int pos = p.t_begin + t;
            uint4 *dst = reinterpret_cast<uint4 *>(p.codes + static_cast<size_t>(b) * p.block + p.off[h] +
                                                   static_cast<size_t>(pos) * (16 * BITS * NH) + 16 * BITS * sl);
#pragma unroll
            for (int j = 0; j < BITS; j++) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
            if (sl == 0) p.scale[(static_cast<size_t>(b) * p.H + h) * p.capacity + pos] = scale;
        }
    }
}

template <int BITS, bool VAL, int NH, int NP = 1>
cudaError_t rows_launch(const RowsParams &p, cudaStream_t s) {
    constexpr size_t smem = rows_smem_bytes<NH>(VAL && BITS <= 4);
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(compress_rows_kernel<BITS, VAL, NH, NP>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    constexpr int TPW = 32 * NP / NH;
    const long long blocks = (static_cast<long long>((p.T + TPW - 1) / TPW) * p.n_heads * p.B + kWarps - 1) / kWarps;
    const long long grid = std::min<long long>(blocks, static_cast<long long>(sms) * 3);
    compress_rows_kernel<BITS, VAL, NH, NP><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

// The launch of one width, keys or values.
template <int NH, int NP = 1>
cudaError_t rows_dispatch(const RowsParams &p, int bits, bool values, cudaStream_t s) {
    switch (bits * 2 + (values ? 1 : 0)) {
        case 2: return rows_launch<1, false, NH, NP>(p, s);
        case 3: return rows_launch<1, true, NH, NP>(p, s);
        case 4: return rows_launch<2, false, NH, NP>(p, s);
        case 5: return rows_launch<2, true, NH, NP>(p, s);
        case 6: return rows_launch<3, false, NH, NP>(p, s);
        case 7: return rows_launch<3, true, NH, NP>(p, s);
        case 8: return rows_launch<4, false, NH, NP>(p, s);
        case 9: return rows_launch<4, true, NH, NP>(p, s);
        case 10: return rows_launch<5, false, NH, NP>(p, s);
        case 11: return rows_launch<5, true, NH, NP>(p, s);
        case 12: return rows_launch<6, false, NH, NP>(p, s);
        case 13: return rows_launch<6, true, NH, NP>(p, s);
        case 14: return rows_launch<7, false, NH, NP>(p, s);
        case 15: return rows_launch<7, true, NH, NP>(p, s);
        case 16: return rows_launch<8, false, NH, NP>(p, s);
        case 17: return rows_launch<8, true, NH, NP>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace tqk
