// tq_compress_dense.cu -- compression with a dense rotation y = Q x on the
// fifth-generation tensor cores.
//
// Method: "TurboMOQ", "Stable QR Rotation" (a Haar-random orthogonal Q from a
// QR factorisation) with the same per-vector scales, quantizers and bit
// packing as the SRHT path ("TurboMOQ", "Architecture").
//
// The rotation of a 128-token tile of one (batch, head, K|V) is the GEMM
// Y[128 tok][128] = X[128 tok][128] Q^T.  X (fp16, exact) arrives by TMA with
// the 128-byte swizzle; Q is held in shared memory for the whole kernel as two
// fp16 matrices, hi = fp16(16 Q) and lo = fp16(16 Q - hi), so that
// X (hi + lo)^T / 16 carries Q to ~2^-22 (the factor 16 keeps lo out of the
// fp16 subnormal range).  One thread issues the 16 tcgen05.mma (M = N = 128,
// K = 16) of a tile into a TMEM accumulator; each epilogue thread then owns
// one token: it reads its 128 accumulator columns with tcgen05.ld and
// quantizes, packs and stores the vector with the binary32 steps of the SRHT
// path.  The accumulation order of the tensor cores is not the oracle's, so a
// code can differ where y lies within ~1e-6 of a decision boundary.
//
// Roles (576 threads, one CTA per SM, persistent over tiles):
//   warps 0-15 four epilogue warpgroups; warpgroup e takes the CTA's tiles
//              e, e + 4, ... and TMEM accumulator e
//   warp 16    TMA producer: 3 stages of 32 KB (two 64-column boxes per tile)
//   warp 17    TMEM allocation (all 512 columns) and the MMA issue
// Every wait is bounded; on a timeout the kernel sets the compress error flag,
// lets its own copies and MMAs finish (bounded again), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "tq_internal.h"

namespace tqk {
namespace dense {
namespace {

constexpr int kTile = 128;                    // tokens per tile (MMA M)
constexpr int kStagesA = 3;
constexpr int kGroups = 4;                    // epilogue warpgroups = TMEM accumulators
constexpr int kEpiWarps = 4 * kGroups;
constexpr int kWarpTma = kEpiWarps, kWarpMma = kEpiWarps + 1;
constexpr int kThreadsDense = 32 * (kEpiWarps + 2);
constexpr int kBoxBytes = kTile * 64 * 2;     // one 64-column box: 16 KB
constexpr int kTileBytes = 2 * kBoxBytes;     // 32 KB
constexpr int kBBytes = 2 * 2 * kBoxBytes;    // hi and lo, two K halves each: 64 KB
constexpr int kTmemCols = 128 * kGroups;      // one 128-column fp32 accumulator per warpgroup
constexpr int kOffA = kBBytes;
constexpr int kOffThr = kOffA + kStagesA * kTileBytes;
constexpr int kOffBar = kOffThr + kCbTotal * 4 + 8;  // 8-byte aligned
constexpr int kSmemBytes = kOffBar + 16 * 8 + 16 + 1024;  // + alignment slack
static_assert(2 * kStagesA + 2 * kGroups <= 16, "barrier slots");
// instruction descriptor of kind::f16: D f32 (bits 4-5 = 1), A = B = f16,
// both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(128 >> 3) << 17) |
                            (static_cast<uint32_t>(128 >> 4) << 24);

__device__ int g_error;

__device__ __forceinline__ unsigned su32(const void *p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void bar_init(unsigned bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(unsigned bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(unsigned bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool bar_try(unsigned bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded: gives up after 2^20 polls (each may suspend for a while)
__device__ __forceinline__ bool bar_wait(unsigned bar, unsigned parity) {
    for (int i = 0; i < (1 << 20); i++)
        if (bar_try(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void tma_load_box(unsigned dst, const CUtensorMap *map, int x, int t, int h, int b,
                                             unsigned bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(t), "r"(h), "r"(b), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), leading offset unused (1), descriptor version 1
__device__ __forceinline__ uint64_t smem_desc(unsigned addr) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void mma_f16(unsigned tmem_d, uint64_t a, uint64_t b, unsigned accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(unsigned bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive accumulator columns of this thread's TMEM lane, times 1/16
// (the factor of the B operand, exact).  The wait is in the same asm statement
// so that no use of the registers can be scheduled before the load completes.
__device__ __forceinline__ void tmem_ld32(unsigned taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]) * 0.0625f;
}

// ---------------------------------------------------------------- epilogues
// Each epilogue thread owns one token's accumulator row and reads it twice,
// 32 columns at a time: first for the scale, then for the codes (the row stays
// in TMEM, so no thread holds all 128 values).

// sum of squares as the pairwise tree of the format: ((y0^2 + y1^2) + (y2^2 + y3^2)) + ...
template <int N, int OFF>
__device__ __forceinline__ float tree_sumsq(const float (&y)[32]) {
    if constexpr (N == 1) return __fmul_rn(y[OFF], y[OFF]);
    else return __fadd_rn(tree_sumsq<N / 2, OFF>(y), tree_sumsq<N / 2, OFF + N / 2>(y));
}

// Codes of coordinates [32 j, 32 j + 32) as BITS LSB-first words (the record's
// bytes [4 BITS j, 4 BITS (j + 1))), stored at once: the four chunks of a
// record run as a loop, so each width's code is one 32-code body (a quarter
// of the instructions to cache, and BITS words live instead of 4 BITS).
template <int BITS, typename CodeOf>
__device__ __forceinline__ void pack_store_chunk(uint8_t *rec, int j, bool store, CodeOf code_of) {
    uint32_t w[BITS];
#pragma unroll
    for (int i = 0; i < BITS; i++) w[i] = 0u;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        const uint32_t c = code_of(i);
        const int bit = BITS * i;
        w[bit >> 5] |= c << (bit & 31);
        if ((bit & 31) + BITS > 32) w[(bit >> 5) + 1] |= c >> (32 - (bit & 31));
    }
    if (!store) return;
    uint8_t *dst = rec + 4 * BITS * j;
    if constexpr (BITS % 4 == 0) {
#pragma unroll
        for (int i = 0; i < BITS / 4; i++)
            reinterpret_cast<uint4 *>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else if constexpr (BITS % 2 == 0) {
#pragma unroll
        for (int i = 0; i < BITS / 2; i++) reinterpret_cast<uint2 *>(dst)[i] = make_uint2(w[2 * i], w[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < BITS; i++) reinterpret_cast<uint32_t *>(dst)[i] = w[i];
    }
}

// keys: m = max |y|, code = clamp(floor((y * fl(1/m) + 1) * 2^(b-1)))
template <int KB>
__device__ __forceinline__ void key_epilogue(unsigned taddr, uint8_t *rec, float *scale, bool store) {
    float v[32];
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        tmem_ld32(taddr + 32 * j, v);
#pragma unroll
        for (int i = 0; i < 32; i++) m = fmaxf(m, fabsf(v[i]));
    }
    const float r = m > 0.f ? __frcp_rn(m) : 0.f;
    constexpr float half_cells = static_cast<float>(1 << (KB - 1));
    auto code = [&](int i) {
        const float u = __fmul_rn(__fadd_rn(__fmul_rn(v[i], r), 1.0f), half_cells);
        const int k = static_cast<int>(floorf(u));
        return static_cast<uint32_t>(min(max(k, 0), (1 << KB) - 1));
    };
#pragma unroll 1
    for (int j = 0; j < 4; j++) {
        tmem_ld32(taddr + 32 * j, v);
        pack_store_chunk<KB>(rec, j, store, code);
    }
    if (store) *scale = m;
}

// values: sigma = sqrt(tree(y^2) / d), code = #{thresholds < y * fl(1/sigma)}
template <int VB>
__device__ __forceinline__ void value_epilogue(unsigned taddr, const float *thr, uint8_t *rec, float *scale,
                                               bool store) {
    float v[32];
    float part[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        tmem_ld32(taddr + 32 * j, v);
        part[j] = tree_sumsq<32, 0>(v);
    }
    const float ss = __fadd_rn(__fadd_rn(part[0], part[1]), __fadd_rn(part[2], part[3]));
    const float sigma = __fsqrt_rn(__fdiv_rn(ss, static_cast<float>(kD)));
    const float r = sigma > 0.f ? __frcp_rn(sigma) : 0.f;
    // up to 4 bits: count the thresholds below u from registers; wider codes:
    // binary search with volatile shared loads (one dependent load per step;
    // plain loads get if-converted into loads of every threshold)
    constexpr int kRegThr = VB <= 4 ? (1 << VB) - 1 : 1;
    float tr[kRegThr];
#pragma unroll
    for (int j = 0; j < kRegThr; j++) tr[j] = thr[j];
    const unsigned thr_s = su32(thr);
    auto code = [&](int i) {
        const float u = __fmul_rn(v[i], r);
        int k = 0;
        if constexpr (VB <= 4) {
#pragma unroll
            for (int j = 0; j < kRegThr; j++) k += tr[j] < u ? 1 : 0;
        } else {
#pragma unroll
            for (int step = 1 << (VB - 1); step >= 1; step >>= 1) {
                float t;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(t) : "r"(thr_s + 4u * (k + step - 1)));
                k += t < u ? step : 0;
            }
        }
        return static_cast<uint32_t>(k);
    };
#pragma unroll 1
    for (int j = 0; j < 4; j++) {
        tmem_ld32(taddr + 32 * j, v);
        pack_store_chunk<VB>(rec, j, store, code);
    }
    if (store) *scale = sigma;
}

struct TileId {
    int which, b, h, t0;
};
__device__ __forceinline__ TileId tile_of(long long id, int H, int n_t) {
    TileId r;
    r.t0 = static_cast<int>(id % n_t) * kTile;
    long long v = id / n_t;
    r.which = static_cast<int>(v & 1);
    v >>= 1;
    r.h = static_cast<int>(v % H);
    r.b = static_cast<int>(v / H);
    return r;
}

__global__ void __launch_bounds__(kThreadsDense, 1)
    compress_dense_kernel(const __grid_constant__ CompressParams p, const __grid_constant__ CUtensorMap map_k,
                          const __grid_constant__ CUtensorMap map_v, const long long n_tiles) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const unsigned sbase = su32(smem);
    const unsigned sB = sbase, sA = sbase + kOffA;
    float *thr = reinterpret_cast<float *>(smem + kOffThr);
    const unsigned bars = sbase + kOffBar;
    // barriers: full[stages], empty[stages], tfull[groups], tempty[groups]
    auto full = [&](int s) { return bars + 8u * s; };
    auto empty = [&](int s) { return bars + 8u * (kStagesA + s); };
    auto tfull = [&](int a) { return bars + 8u * (2 * kStagesA + a); };
    auto tempty = [&](int a) { return bars + 8u * (2 * kStagesA + kGroups + a); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + 16 * 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_t = (p.T + kTile - 1) / kTile;
    const long long n_local = n_tiles > blockIdx.x ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesA; s++) {
            bar_init(full(s), 1);
            bar_init(empty(s), 1);
        }
        for (int a = 0; a < kGroups; a++) {
            bar_init(tfull(a), 1);
            bar_init(tempty(a), 4 * 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // B operand: 16 Q split into fp16 hi + lo, K-major rows of the output
    // coordinate n, two 64-column halves, 128-byte swizzle (chunk ^= row & 7)
    for (int idx = threadIdx.x; idx < kD * kD; idx += kThreadsDense) {
        const int n = idx >> 7, k = idx & 127;
        const float v = 16.0f * p.Q[idx];
        const __half hi = __float2half_rn(v);
        const __half lo = __float2half_rn(v - __half2float(hi));
        const int kk = k & 63;
        const int off = (k >> 6) * kBoxBytes + n * 128 + ((((kk * 2) >> 4) ^ (n & 7)) << 4) + ((kk * 2) & 15);
        *reinterpret_cast<__half *>(smem + off) = hi;
        *reinterpret_cast<__half *>(smem + 2 * kBoxBytes + off) = lo;
    }
    for (int i = threadIdx.x; i < kCbTotal; i += kThreadsDense) thr[i] = p.thr[i];
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const unsigned tbase = *tmem_slot;

    if (warp == kWarpTma) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            long long i = 0;
            bool ok = true;
            for (; i < n_local && ok; i++) {
                const int s = static_cast<int>(i % kStagesA);
                if (!bar_wait(empty(s), static_cast<unsigned>(((i / kStagesA) & 1) ^ 1))) {
                    ok = false;
                    break;
                }
                const TileId t = tile_of(blockIdx.x + i * gridDim.x, p.H, n_t);
                const CUtensorMap *map = t.which ? &map_v : &map_k;
                bar_expect_tx(full(s), kTileBytes);
                tma_load_box(sA + s * kTileBytes, map, 0, t.t0, t.h, t.b, full(s));
                tma_load_box(sA + s * kTileBytes + kBoxBytes, map, 64, t.t0, t.h, t.b, full(s));
            }
            if (!ok) {
                atomicExch(&g_error, 1);
                // the copies already issued land before the CTA goes away
                for (long long j = i > kStagesA ? i - kStagesA : 0; j < i; j++)
                    bar_wait(full(static_cast<int>(j % kStagesA)), static_cast<unsigned>((j / kStagesA) & 1));
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            long long i = 0;
            bool ok = true;
            for (; i < n_local; i++) {
                const int s = static_cast<int>(i % kStagesA), acc = static_cast<int>(i % kGroups);
                if (!bar_wait(full(s), static_cast<unsigned>((i / kStagesA) & 1)) ||
                    !bar_wait(tempty(acc), static_cast<unsigned>(((i / kGroups) & 1) ^ 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const unsigned d = tbase + static_cast<unsigned>(acc * 128);
                const unsigned a0 = sA + s * kTileBytes;
#pragma unroll
                for (int part = 0; part < 2; part++) {  // hi, then lo
#pragma unroll
                    for (int kb = 0; kb < 2; kb++)
#pragma unroll
                        for (int k = 0; k < 4; k++)
                            mma_f16(d, smem_desc(a0 + kb * kBoxBytes + 32 * k),
                                    smem_desc(sB + part * 2 * kBoxBytes + kb * kBoxBytes + 32 * k),
                                    (part | kb | k) != 0);
                }
                mma_commit(empty(s));
                mma_commit(tfull(acc));
            }
            if (!ok) atomicExch(&g_error, 1);
            if (i > 0) {  // the last tile's MMAs have completed (a commit covers all earlier MMAs)
                const long long j = i - 1;
                bar_wait(tfull(static_cast<int>(j % kGroups)), static_cast<unsigned>((j / kGroups) & 1));
            }
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int e = warp >> 2, quarter = warp & 3;
        const int row = 32 * quarter + lane;
        for (long long i = e; i < n_local; i += kGroups) {
            // warp-uniform outcome: tcgen05.ld below needs the whole warp
            if (!__all_sync(0xffffffffu, bar_wait(tfull(e), static_cast<unsigned>((i / kGroups) & 1)))) {
                if (lane == 0) atomicExch(&g_error, 1);
                break;
            }
            tc_fence_after();
            const unsigned taddr = tbase + (static_cast<unsigned>(32 * quarter) << 16) + static_cast<unsigned>(e * 128);
            const TileId t = tile_of(blockIdx.x + i * gridDim.x, p.H, n_t);
            const int tok = t.t0 + row;
            const bool store = tok < p.T;  // rows past the end hold zeros; the warp still reads TMEM together
            const int pos = p.t_begin + min(tok, p.T - 1);
            const size_t sidx = (static_cast<size_t>(t.b) * p.H + t.h) * p.capacity + pos;
            if (t.which == 0) {
                const int kb = p.kbits[t.h];
                uint8_t *rec = p.kcodes + static_cast<size_t>(t.b) * p.kblock + p.koff[t.h] +
                               static_cast<size_t>(pos) * (16 * kb);
                float *sc = p.kscale + sidx;
                switch (kb) {
                    case 1: key_epilogue<1>(taddr, rec, sc, store); break;
                    case 2: key_epilogue<2>(taddr, rec, sc, store); break;
                    case 3: key_epilogue<3>(taddr, rec, sc, store); break;
                    case 4: key_epilogue<4>(taddr, rec, sc, store); break;
                    case 5: key_epilogue<5>(taddr, rec, sc, store); break;
                    case 6: key_epilogue<6>(taddr, rec, sc, store); break;
                    case 7: key_epilogue<7>(taddr, rec, sc, store); break;
                    default: key_epilogue<8>(taddr, rec, sc, store); break;
                }
            } else {
                const int vb = p.vbits[t.h];
                uint8_t *rec = p.vcodes + static_cast<size_t>(t.b) * p.vblock + p.voff[t.h] +
                               static_cast<size_t>(pos) * (16 * vb);
                float *sc = p.vscale + sidx;
                const float *th = thr + cb_off(vb);
                switch (vb) {
                    case 1: value_epilogue<1>(taddr, th, rec, sc, store); break;
                    case 2: value_epilogue<2>(taddr, th, rec, sc, store); break;
                    case 3: value_epilogue<3>(taddr, th, rec, sc, store); break;
                    case 4: value_epilogue<4>(taddr, th, rec, sc, store); break;
                    case 5: value_epilogue<5>(taddr, th, rec, sc, store); break;
                    case 6: value_epilogue<6>(taddr, th, rec, sc, store); break;
                    case 7: value_epilogue<7>(taddr, th, rec, sc, store); break;
                    default: value_epilogue<8>(taddr, th, rec, sc, store); break;
                }
            }
            // the accumulator is free once every thread of the warpgroup has read it
            tc_fence_before();
            bar_arrive(tempty(e));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols) : "memory");
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// [B][H][T][d] fp16 with element strides sb, sh, st: dims (d, T, H, B), boxes of
// 64 x 128 x 1 x 1 with the 128-byte swizzle; rows past T read as zeros
bool make_map(CUtensorMap *map, const uint16_t *base, const CompressParams &p) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(p.T),
                                static_cast<cuuint64_t>(p.H), static_cast<cuuint64_t>(p.B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.st) * 2, static_cast<cuuint64_t>(p.sh) * 2,
                                   static_cast<cuuint64_t>(p.sb) * 2};
    const cuuint32_t box[4] = {64, kTile, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<uint16_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace dense

cudaError_t launch_compress_dense(const CompressParams &p, cudaStream_t s) {
    using namespace dense;
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(compress_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    CUtensorMap mk, mv;
    if (!make_map(&mk, p.K, p) || !make_map(&mv, p.V, p)) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long n_tiles = 2LL * p.B * p.H * ((p.T + kTile - 1) / kTile);
    if (n_tiles == 0) return cudaSuccess;
    const int grid = static_cast<int>(std::min<long long>(n_tiles, sms));
    compress_dense_kernel<<<grid, kThreadsDense, kSmemBytes, s>>>(p, mk, mv, n_tiles);
    return cudaGetLastError();
}

cudaError_t read_compress_dense_error(int *flag) {
    return cudaMemcpyFromSymbol(flag, dense::g_error, sizeof(int));
}

cudaError_t clear_compress_dense_error() {
    const int zero = 0;
    return cudaMemcpyToSymbol(dense::g_error, &zero, sizeof(int));
}

}  // namespace tqk
