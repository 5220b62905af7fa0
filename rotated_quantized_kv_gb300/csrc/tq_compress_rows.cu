// tq_compress_rows.cu -- compression of 128-dimension key or value vectors
// with one thread per vector, for launches without QJL sketches.
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
#include <algorithm>

#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tqk {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kRowBytes = 256;            // 128 fp16 coordinates
constexpr int kWarpBuf = 32 * kRowBytes;  // one staged block of 32 rows

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

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}

// Stage the fp16 rows of block `blk` ((b, head of the list, 32-token block),
// token block fastest) into this warp's buffer.
__device__ __forceinline__ void stage_rows(const RowsParams &p, int n_tblk, int blk, uint8_t *buf, int lane) {
    const int tb = blk % n_tblk, rest = blk / n_tblk;
    const int h = p.head[rest % p.n_heads], b = rest / p.n_heads;
    const int t0 = tb * 32, nt = min(32, p.T - t0);
    const uint16_t *src = p.X + b * p.sb + h * p.sh + static_cast<int64_t>(t0) * p.st;
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const int idx = lane + 32 * i, r = idx >> 4, c = idx & 15;
        if (r < nt) cp_async16(buf + r * kRowBytes + 16 * (c ^ (r & 7)), src + static_cast<int64_t>(r) * p.st + 8 * c);
    }
}

// Code i (0..127) at bits [B i, B i + B) of the record's 4 B words.
template <int B>
__device__ __forceinline__ void put(uint32_t (&w)[4 * B], int i, uint32_t k) {
    const int bit = i * B, wi = bit >> 5, sh = bit & 31;
    w[wi] += k << sh;  // codes never overlap: an add (one shift-and-add instruction) is the or
    if (sh + B > 32) w[wi + 1] += k >> (32 - sh);
}

template <int BITS, bool VAL>
__global__ void __launch_bounds__(kThreads, 3) compress_rows_kernel(const __grid_constant__ RowsParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t *in_mask = reinterpret_cast<uint32_t *>(smem + kWarps * 2 * kWarpBuf);  // [64]
    float *out_scale = reinterpret_cast<float *>(in_mask + 64);                      // [128]
    float *thr = out_scale + kD;                                                     // [255]
    for (int i = threadIdx.x; i < 64; i += kThreads) in_mask[i] = p.in_mask[i];
    for (int i = threadIdx.x; i < kD; i += kThreads) out_scale[i] = p.out_scale[i];
    for (int i = threadIdx.x; i < 255; i += kThreads) thr[i] = p.thr[i];
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *bufs = smem + warp * 2 * kWarpBuf;
    const int n_tblk = (p.T + 31) / 32;
    const int n_blk = n_tblk * p.n_heads * p.B;
    const int gw = blockIdx.x * kWarps + warp, nw = gridDim.x * kWarps;
    if (gw < n_blk) stage_rows(p, n_tblk, gw, bufs, lane);
    asm volatile("cp.async.commit_group;\n" ::);

    for (int blk = gw, it = 0; blk < n_blk; blk += nw, it++) {
        const int next = blk + nw;
        if (next < n_blk) stage_rows(p, n_tblk, next, bufs + ((it + 1) & 1) * kWarpBuf, lane);
        asm volatile("cp.async.commit_group;\n" ::);
        asm volatile("cp.async.wait_group 1;\n" ::: "memory");
        __syncwarp();
        const int tb = blk % n_tblk, rest = blk / n_tblk;
        const int h = p.head[rest % p.n_heads], b = rest / p.n_heads;
        const int t = tb * 32 + lane;
        const uint8_t *row = bufs + (it & 1) * kWarpBuf + lane * kRowBytes;

        // ---- load, input sign flip on the fp16 bits, widen
        float2 a[64];
#pragma unroll
        for (int c = 0; c < 16; c++) {
            uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * (c ^ (lane & 7)));
            const uint4 mk = *reinterpret_cast<const uint4 *>(in_mask + 4 * c);
            v.x ^= mk.x;
            v.y ^= mk.y;
            v.z ^= mk.z;
            v.w ^= mk.w;
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&wv[e]));
                const int i = 8 * c + 2 * e;  // coordinates i, i + 1
                if (c < 8) {
                    a[i].x = f.x;
                    a[i + 1].x = f.y;
                } else {
                    a[i - 64].y = f.x;
                    a[i - 63].y = f.y;
                }
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
#pragma unroll
        for (int m = 0; m < 64; m++) {
            const float u = a[m].x, v = a[m].y;
            a[m].x = __fadd_rn(u, v);
            a[m].y = __fsub_rn(u, v);
        }
        // output sign flip and binary32(1/sqrt(d)): one rounded multiply each
#pragma unroll
        for (int m = 0; m < 64; m++) a[m] = fmul2(a[m], make_float2(out_scale[m], out_scale[m + 64]));

        uint32_t w[4 * BITS];
#pragma unroll
        for (int j = 0; j < 4 * BITS; j++) w[j] = 0u;
        float scale;
        if constexpr (!VAL) {
            // ---- keys: m = max |y|, v = y * binary32(1/m), u = round(v + 1) 2^(b-1),
            // code = clamp(floor(u), 0, 2^b - 1)
            float mx = 0.0f;
#pragma unroll
            for (int m = 0; m < 64; m++) mx = fmaxf(mx, fmaxf(fabsf(a[m].x), fabsf(a[m].y)));
            scale = mx;
            const float r = mx > 0.0f ? __frcp_rn(mx) : 0.0f;
            constexpr float hc = static_cast<float>(1 << (BITS - 1));
            // floor(u) for u in [-1, 2^b]: round-down of u + 2^23 + 512 has the
            // exponent of 2^23, so its low bits are 512 + floor(u)
            constexpr float kMagic = 8388608.0f + 512.0f;
            constexpr int kLo = 0x4B000000 + 512, kHi = kLo + (1 << BITS) - 1;
#pragma unroll
            for (int m = 0; m < 64; m++) {
                const float2 v = fmul2(a[m], make_float2(r, r));
                // fma(v, 2^(b-1), 2^(b-1)) is round(v + 1) 2^(b-1): scaling by a
                // power of two commutes with the rounding
                const float2 u = ffma2(v, make_float2(hc, hc), make_float2(hc, hc));
                const float2 f = fadd2_rm(u, make_float2(kMagic, kMagic));
                const int k0 = min(max(__float_as_int(f.x), kLo), kHi) - kLo;
                const int k1 = min(max(__float_as_int(f.y), kLo), kHi) - kLo;
                put<BITS>(w, m, static_cast<uint32_t>(k0));
                put<BITS>(w, m + 64, static_cast<uint32_t>(k1));
            }
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
            const float tot = __fadd_rn(s[0].x, s[0].y);
            const float sigma = __fsqrt_rn(__fmul_rn(tot, 1.0f / kD));  // / d exact (a power of two)
            scale = sigma;
            const float r = sigma > 0.0f ? __frcp_rn(sigma) : 0.0f;
            constexpr int NT = (1 << BITS) - 1;
            if constexpr (BITS <= 4) {
                float th[NT];
#pragma unroll
                for (int j = 0; j < NT; j++) th[j] = thr[j];
#pragma unroll
                for (int m = 0; m < 64; m++) {
                    const float2 u = fmul2(a[m], make_float2(r, r));
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
            } else {
#pragma unroll
                for (int m = 0; m < 64; m++) {
                    const float2 u = fmul2(a[m], make_float2(r, r));
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
        if (t < p.T) {
            const int pos = p.t_begin + t;
            uint4 *dst = reinterpret_cast<uint4 *>(p.codes + static_cast<size_t>(b) * p.block + p.off[h] +
                                                   static_cast<size_t>(pos) * (16 * BITS));
#pragma unroll
            for (int j = 0; j < BITS; j++) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
            p.scale[(static_cast<size_t>(b) * p.H + h) * p.capacity + pos] = scale;
        }
    }
}

template <int BITS, bool VAL>
cudaError_t rows_launch(const RowsParams &p, cudaStream_t s) {
    constexpr size_t smem = kWarps * 2 * kWarpBuf + 64 * 4 + kD * 4 + 255 * 4;
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(compress_rows_kernel<BITS, VAL>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long blocks = (static_cast<long long>((p.T + 31) / 32) * p.n_heads * p.B + kWarps - 1) / kWarps;
    const long long grid = std::min<long long>(blocks, static_cast<long long>(sms) * 3);
    compress_rows_kernel<BITS, VAL><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress_rows(const RowsParams &p, int bits, bool values, cudaStream_t s) {
    switch (bits * 2 + (values ? 1 : 0)) {
        case 2: return rows_launch<1, false>(p, s);
        case 3: return rows_launch<1, true>(p, s);
        case 4: return rows_launch<2, false>(p, s);
        case 5: return rows_launch<2, true>(p, s);
        case 6: return rows_launch<3, false>(p, s);
        case 7: return rows_launch<3, true>(p, s);
        case 8: return rows_launch<4, false>(p, s);
        case 9: return rows_launch<4, true>(p, s);
        case 10: return rows_launch<5, false>(p, s);
        case 11: return rows_launch<5, true>(p, s);
        case 12: return rows_launch<6, false>(p, s);
        case 13: return rows_launch<6, true>(p, s);
        case 14: return rows_launch<7, false>(p, s);
        case 15: return rows_launch<7, true>(p, s);
        case 16: return rows_launch<8, false>(p, s);
        case 17: return rows_launch<8, true>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tqk
