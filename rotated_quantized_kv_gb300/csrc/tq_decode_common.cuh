// tq_decode_common.cuh -- device helpers shared by the decode-attention
// kernels (split-K over packed and fp16 segments, prep, combine).
#pragma once

#include <utility>

#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tqk {
namespace dec {

constexpr int kThreads = 128;                 // 4 warps per CTA
constexpr int kPartStride = 4 + kD;           // m, l, pad, pad, acc[d]
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, int src_bytes) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ TMA bulk copies
// One thread issues 1-D bulk copies global -> shared that complete on an
// mbarrier (transaction bytes); consumers wait on the barrier's phase.
__device__ __forceinline__ unsigned smem_u32(const void *p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// Orders this thread's earlier generic-proxy shared accesses before its later
// async-proxy (bulk copy) writes.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// The same copy with an L2 eviction policy (policy_evict_first: read once,
// streamed), so that a stream much larger than L2 does not push out the small
// working set that is read again (partial records, queries).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, unsigned bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for a barrier phase: gives up after `polls` polls (default
// 2^20; each poll may suspend in hardware for a while), so a copy that never
// completes cannot hang the GPU.  Returns false on timeout.
constexpr int kWaitPolls = 1 << 20;
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity, int polls = kWaitPolls) {
    for (int i = 0; i < polls; i++)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// 2^x with the hardware approximation (relative error ~2^-22).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

__device__ __forceinline__ float warp_max_g(float v) {  // over the 8 lanes sharing lane & 3
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
    return v;
}
__device__ __forceinline__ float warp_sum_g(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    return v;
}

// Running state of one warp: per thread, query head c = lane & 3 of the GQA
// group; acc holds the P.V accumulator fragment (8 m-tiles x 4).
struct WarpState {
    float m, l;
    float wsum;      // sum of the weights p * value scale (linear value decodes only)
    float wsum_odd;  // the same over the odd tokens of token pairs (head_dim 64)
    float acc[8][4];
};

__device__ __forceinline__ void init_state(WarpState &st) {
    st.m = kNegInf;
    st.l = 0.f;
    st.wsum = 0.f;
    st.wsum_odd = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; mt++)
#pragma unroll
        for (int q = 0; q < 4; q++) st.acc[mt][q] = 0.f;
}

// Online-softmax update of one 16-token tile (scores s of tokens g and g+8 for
// head c, already in base-2 logits) and the B fragment of P (times the value
// scale vs) for the P.V MMA: column n = g holds head g/2, hi (g even) or lo
// (g odd) fp16 part, rows = tokens 2c, 2c+1 (b0) and 2c+8, 2c+9 (b1).
__device__ __forceinline__ void softmax_tile(WarpState &st, float s0, float s1, bool v0ok, bool v1ok,
                                             float vs0, float vs1, int g, int c, bool head_ok,
                                             uint32_t &b0, uint32_t &b1) {
    float t = fmaxf(v0ok ? s0 : kNegInf, v1ok ? s1 : kNegInf);
    t = warp_max_g(t);
    const float mnew = fmaxf(st.m, t);
    float p0 = 0.f, p1 = 0.f;
    if (mnew != kNegInf) {
        p0 = v0ok ? ex2(s0 - mnew) : 0.f;
        p1 = v1ok ? ex2(s1 - mnew) : 0.f;
    }
    // rescale only when some head's running max moved (rare after the first tiles)
    if (__any_sync(0xffffffffu, mnew > st.m)) {
        const float corr = (mnew == kNegInf) ? 1.f : ex2(st.m - mnew);
        st.l *= corr;
#pragma unroll
        for (int mt = 0; mt < 8; mt++)
#pragma unroll
            for (int q = 0; q < 4; q++) st.acc[mt][q] *= corr;
    }
    st.m = mnew;
    st.l += p0 + p1;
    // selects, not products: value scales of masked tokens may be stale bytes
    const float w0 = (head_ok && v0ok) ? p0 * vs0 : 0.f;
    const float w1 = (head_ok && v1ok) ? p1 * vs1 : 0.f;
    const int src0 = 8 * c + (g >> 1), src1 = src0 + 4;
    const float x0 = __shfl_sync(0xffffffffu, w0, src0);
    const float x1 = __shfl_sync(0xffffffffu, w0, src1);
    const float x2 = __shfl_sync(0xffffffffu, w1, src0);
    const float x3 = __shfl_sync(0xffffffffu, w1, src1);
    // hi part for even columns, lo = x - hi for odd ones (branch-free: the
    // columns alternate within a warp)
    const __half2 h01 = __floats2half2_rn(x0, x1);
    const __half2 h23 = __floats2half2_rn(x2, x3);
    const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
    const float m = (g & 1) ? 1.f : 0.f;  // subtract hi only for the lo columns
    const __half2 p01 = __floats2half2_rn(x0 - m * f01.x, x1 - m * f01.y);
    const __half2 p23 = __floats2half2_rn(x2 - m * f23.x, x3 - m * f23.y);
    b0 = *reinterpret_cast<const uint32_t *>(&p01);
    b1 = *reinterpret_cast<const uint32_t *>(&p23);
}

// Online softmax over two 16-token tiles with a lazy running max, for the
// packed kernel.  Thread (g, c) holds the scores (base-2 logits) of tokens g
// and g+8 of tile A (s[0], s[1]) and tile B (s[2], s[3]) for query head c.
// Probabilities are taken relative to the head's reference max m; the
// cross-lane max and the rescale run only when a score exceeds m by more than
// 8 (so every probability stays <= 2^8, exact enough in fp16).  The P.V B
// fragments are plain fp16 probabilities times the value scale: column n = g
// holds head g (columns of heads >= gqa carry values nobody reads), rows =
// tokens 2c, 2c+1 (b0) and 2c+8, 2c+9 (b1).  The P.V accumulator columns 2c,
// 2c+1 of lane (g, c) are heads 2c, 2c+1, so a rescale fetches those heads'
// factors from their owners.  FULL: all 32 tokens valid (no masking).  WSUM:
// also accumulate the weights (for value decodes that are affine in the code).
template <bool FULL, bool WSUM>
__device__ __forceinline__ void softmax_pair(WarpState &st, const float (&s)[4], const bool (&ok)[4],
                                             const float (&vs)[4], int g, int c, uint32_t (&b)[4]) {
    const int lane = threadIdx.x & 31;
    float smax, vmax;
    if constexpr (FULL) {
        smax = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
        vmax = fmaxf(fmaxf(vs[0], vs[1]), fmaxf(vs[2], vs[3]));
    } else {
        smax = kNegInf;
        vmax = 0.f;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            smax = fmaxf(smax, ok[i] ? s[i] : kNegInf);
            vmax = fmaxf(vmax, ok[i] ? vs[i] : 0.f);
        }
    }
    // The running max may lag the true one by up to 8 (log2 units), so that
    // most tiles skip the rescale; weights then reach 2^8 * scale, which stays
    // inside fp16 while scales are <= 255.  Larger scales rescale exactly
    // (weights <= scale <= 65504, the fp16 range of the cached values).
    if (__any_sync(0xffffffffu, smax > st.m + 8.0f || (smax > st.m && vmax > 255.0f))) {
        const float mnew = fmaxf(st.m, warp_max_g(smax));
        const float corr = (mnew == kNegInf) ? 1.f : ex2(st.m - mnew);
        st.l *= corr;
        if constexpr (WSUM) st.wsum *= corr;
        const float c0 = __shfl_sync(0xffffffffu, corr, (lane & ~3) | ((2 * c) & 3));
        const float c1 = __shfl_sync(0xffffffffu, corr, (lane & ~3) | ((2 * c + 1) & 3));
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            st.acc[mt][0] *= c0;
            st.acc[mt][1] *= c1;
            st.acc[mt][2] *= c0;
            st.acc[mt][3] *= c1;
        }
        st.m = mnew;
    }
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        if constexpr (FULL) {
            const float p = ex2(s[i] - st.m);
            st.l += p;
            w[i] = p * vs[i];
        } else {
            const float p = ok[i] ? ex2(s[i] - st.m) : 0.f;
            st.l += p;
            w[i] = ok[i] ? p * vs[i] : 0.f;  // a select: masked scales may be stale bytes
        }
    }
    if constexpr (WSUM) st.wsum += (w[0] + w[1]) + (w[2] + w[3]);
    // transpose: lane (g, c) needs head g's weights of tokens 2c, 2c+1, 2c+8, 2c+9
    const int src0 = 8 * c + (g & 3), src1 = src0 + 4;
#pragma unroll
    for (int t = 0; t < 2; t++) {
        const float x0 = __shfl_sync(0xffffffffu, w[2 * t], src0);
        const float x1 = __shfl_sync(0xffffffffu, w[2 * t], src1);
        const float x2 = __shfl_sync(0xffffffffu, w[2 * t + 1], src0);
        const float x3 = __shfl_sync(0xffffffffu, w[2 * t + 1], src1);
        const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
        b[2 * t] = *reinterpret_cast<const uint32_t *>(&h01);
        b[2 * t + 1] = *reinterpret_cast<const uint32_t *>(&h23);
    }
}

// Partial record of one warp of the packed kernel (accumulator columns 2c,
// 2c+1 of lane (g, c) are heads 2c, 2c+1; lanes c = h own head h's m and l).
// fin(mt, r, acc, W): the accumulator value of row r of m-tile mt as written
// (W: the head's summed weights, for value decodes that are affine in the code).
template <typename DimOf, typename Fin>
__device__ __forceinline__ void write_warp_partial_pair(WarpState &st, float *rec_base, int gqa, DimOf dim_of,
                                                        Fin fin) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const float l = warp_sum_g(st.l);
    const float W = warp_sum_g(st.wsum);
    const float W0 = __shfl_sync(0xffffffffu, W, (lane & ~3) | ((2 * c) & 3));
    const float W1 = __shfl_sync(0xffffffffu, W, (lane & ~3) | ((2 * c + 1) & 3));
    if (c < gqa && g == 0) {
        rec_base[c * kPartStride] = st.m;
        rec_base[c * kPartStride + 1] = l;
    }
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const int h = 2 * c + e;
        const float Wh = e ? W1 : W0;
        if (h < gqa) {
            float *rec = rec_base + h * kPartStride + 4;
#pragma unroll
            for (int mt = 0; mt < 8; mt++) {
                rec[dim_of(mt, 0)] = fin(mt, 0, st.acc[mt][e], Wh);
                rec[dim_of(mt, 1)] = fin(mt, 1, st.acc[mt][2 + e], Wh);
            }
        }
    }
}

// ------------------------------------------------------------ head_dim 64
// The packed kernel reads two consecutive tokens (2 v, 2 v + 1) as one 128-dim
// "virtual" record (their two 64-dim records are adjacent).  Scores come per
// (virtual row, parity); the P.V B fragment's eight columns are (head n & 3,
// parity n >> 2), so accumulator row (dim) of thread group g is meaningful for
// the columns whose parity is that of its half (g < 4: even tokens, dims
// 0..63; g >= 4: odd tokens, virtual dims 64..127); the merge adds the halves.

// softmax_pair for token pairs: s[4 t + 2 r + p] = tile t, virtual row g + 8 r,
// parity p; the B fragment column g (head g & 3, parity g >> 2) of virtual
// tokens 2c, 2c+1 (b[2t]) and 2c+8, 2c+9 (b[2t+1]).
template <bool FULL, bool WSUM>
__device__ __forceinline__ void softmax_pair2(WarpState &st, const float (&s)[8], const bool (&ok)[8],
                                              const float (&vs)[8], int g, int c, uint32_t (&b)[4]) {
    const int lane = threadIdx.x & 31;
    float smax = kNegInf, vmax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        smax = fmaxf(smax, (FULL || ok[i]) ? s[i] : kNegInf);
        vmax = fmaxf(vmax, (FULL || ok[i]) ? vs[i] : 0.f);
    }
    if (__any_sync(0xffffffffu, smax > st.m + 8.0f || (smax > st.m && vmax > 255.0f))) {
        const float mnew = fmaxf(st.m, warp_max_g(smax));
        const float corr = (mnew == kNegInf) ? 1.f : ex2(st.m - mnew);
        st.l *= corr;
        if constexpr (WSUM) {
            st.wsum *= corr;
            st.wsum_odd *= corr;
        }
        const float c0 = __shfl_sync(0xffffffffu, corr, (lane & ~3) | ((2 * c) & 3));
        const float c1 = __shfl_sync(0xffffffffu, corr, (lane & ~3) | ((2 * c + 1) & 3));
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            st.acc[mt][0] *= c0;
            st.acc[mt][1] *= c1;
            st.acc[mt][2] *= c0;
            st.acc[mt][3] *= c1;
        }
        st.m = mnew;
    }
    float w[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const float p = (FULL || ok[i]) ? ex2(s[i] - st.m) : 0.f;
        st.l += p;
        w[i] = (FULL || ok[i]) ? p * vs[i] : 0.f;  // a select: masked scales may be stale bytes
    }
    if constexpr (WSUM) {
        st.wsum += (w[0] + w[2]) + (w[4] + w[6]);
        st.wsum_odd += (w[1] + w[3]) + (w[5] + w[7]);
    }
    const int src0 = 8 * c + (g & 3), src1 = src0 + 4;
    const bool odd = (g >> 2) != 0;
#pragma unroll
    for (int t = 0; t < 2; t++) {
        float x[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {  // (row g_s, source): (0, src0), (0, src1), (1, src0), (1, src1)
            const int r = k >> 1;
            const int src = (k & 1) ? src1 : src0;
            const float xe = __shfl_sync(0xffffffffu, w[4 * t + 2 * r], src);
            const float xo = __shfl_sync(0xffffffffu, w[4 * t + 2 * r + 1], src);
            x[k] = odd ? xo : xe;
        }
        const __half2 h01 = __floats2half2_rn(x[0], x[1]), h23 = __floats2half2_rn(x[2], x[3]);
        b[2 * t] = *reinterpret_cast<const uint32_t *>(&h01);
        b[2 * t + 1] = *reinterpret_cast<const uint32_t *>(&h23);
    }
}

// write_warp_partial_pair for token pairs: lane (g, c) holds columns 2c, 2c+1 =
// (heads (2c) & 3, (2c+1) & 3; parity c >> 1) and writes the rows of its half
// (g < 4 with even columns, g >= 4 with odd ones) as virtual dims 0..127 of
// its heads' records.
template <typename DimOf, typename Fin>
__device__ __forceinline__ void write_warp_partial_pair2(WarpState &st, float *rec_base, int gqa, DimOf dim_of,
                                                         Fin fin) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const float l = warp_sum_g(st.l);
    const float We = warp_sum_g(st.wsum), Wo = warp_sum_g(st.wsum_odd);
    const bool odd = (c >> 1) != 0;
    const float W0e = __shfl_sync(0xffffffffu, We, (lane & ~3) | ((2 * c) & 3));
    const float W0o = __shfl_sync(0xffffffffu, Wo, (lane & ~3) | ((2 * c) & 3));
    const float W1e = __shfl_sync(0xffffffffu, We, (lane & ~3) | ((2 * c + 1) & 3));
    const float W1o = __shfl_sync(0xffffffffu, Wo, (lane & ~3) | ((2 * c + 1) & 3));
    if (c < gqa && g == 0) {
        rec_base[c * kPartStride] = st.m;
        rec_base[c * kPartStride + 1] = l;
    }
    if ((g >= 4) != odd) return;
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const int h = (2 * c + e) & 3;
        const float Wh = e ? (odd ? W1o : W1e) : (odd ? W0o : W0e);
        if (h < gqa) {
            float *rec = rec_base + h * kPartStride + 4;
#pragma unroll
            for (int mt = 0; mt < 8; mt++) {
                rec[dim_of(mt, 0)] = fin(mt, 0, st.acc[mt][e], Wh);
                rec[dim_of(mt, 1)] = fin(mt, 1, st.acc[mt][2 + e], Wh);
            }
        }
    }
}

// Spills.  A warp's running state (m, l, sums) is folded into its partial
// record every few dozen tiles and restarted from zero sums, so that no sum the
// tensor cores accumulate runs long: mma.sync adds its products to the fp32
// accumulator with truncation, which over ~1000 tiles of one warp drifts by
// ~1e-3 of the result, while the folds below round to nearest.  The first
// spill of a group writes the record (write_warp_partial_pair*), whose max
// m_ref then stays: later spills add the state times f = 2^(m - m_ref) >= 1
// (m never decreases within a group) with fire-and-forget vector atomic adds
// (fold_warp_partial).  Should m outgrow m_ref by more than 2^64 (a score
// range that could overflow the scaled sums), merge_warp_partial rescales the
// record to the state's max instead.  Both follow the column ownership of
// write_warp_partial_pair (NP = 1) and write_warp_partial_pair2 (NP = 2): the
// 16 accumulator rows of lane (g, c) are, for every value decoder VD, the dims
// [16 g, 16 g + 16) of its heads' records in the order VD::dim, so each head
// takes four 16-byte accesses.  fin is linear in (acc, W).
template <int NP>
struct PairColumns {
    int h[2];     // heads of the lane's accumulator columns 2c, 2c+1
    bool wr[2];   // whether the lane writes them
    bool odd;     // token pairs: the columns hold the odd half
    __device__ __forceinline__ PairColumns(int gqa) {
        const int g = (threadIdx.x & 31) >> 2, c = threadIdx.x & 3;
        odd = NP == 2 && (c >> 1) != 0;
#pragma unroll
        for (int e = 0; e < 2; e++) {
            h[e] = NP == 2 ? (2 * c + e) & 3 : 2 * c + e;
            wr[e] = h[e] < gqa && (NP == 1 || (g >= 4) == odd);
        }
    }
};

// 2 mt + r of the accumulator row that holds dim d of the lane's 16
template <typename VD>
__host__ __device__ constexpr int acc_row_of_dim(int d) {
    for (int mt = 0; mt < 8; mt++)
        for (int r = 0; r < 2; r++)
            if (VD::dim(mt, r) == d) return 2 * mt + r;
    return -1;
}
template <typename F, int... I>
__device__ __forceinline__ void static_for_impl(F &&f, std::integer_sequence<int, I...>) {
    (f(std::integral_constant<int, I>{}), ...);
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F &&f) {
    static_for_impl(f, std::make_integer_sequence<int, N>{});
}
// the lane's 16 finished sums of column e, in dim order
template <typename VD, typename Fin>
__device__ __forceinline__ void lane_rows(const WarpState &st, int e, float Wh, Fin fin, float (&v)[16]) {
    static_for<16>([&](auto D) {
        constexpr int s = acc_row_of_dim<VD>(decltype(D)::value);
        static_assert(s >= 0, "VD::dim: a permutation of 0..15");
        v[decltype(D)::value] = fin(s >> 1, s & 1, st.acc[s >> 1][2 * (s & 1) + e], Wh);
    });
}
__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// f: head c's factor on lane c
template <int NP, typename VD, typename Fin>
__device__ __forceinline__ void fold_warp_partial(WarpState &st, float *rec_base, int gqa, Fin fin, float f) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const PairColumns<NP> pc(gqa);
    const float l = warp_sum_g(st.l);
    const float We = warp_sum_g(st.wsum);
    const float Wo = NP == 2 ? warp_sum_g(st.wsum_odd) : 0.f;
    if (c < gqa && g == 0) atomicAdd(rec_base + c * kPartStride + 1, l * f);
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const int src = (lane & ~3) | ((2 * c + e) & 3);
        const float fh = __shfl_sync(0xffffffffu, f, src);
        const float Wse = __shfl_sync(0xffffffffu, We, src), Wso = __shfl_sync(0xffffffffu, Wo, src);
        const float Wh = pc.odd ? Wso : Wse;
        if (pc.wr[e]) {
            float v[16];
            lane_rows<VD>(st, e, Wh, fin, v);
            float *row = rec_base + pc.h[e] * kPartStride + 4 + 16 * g;
#pragma unroll
            for (int j = 0; j < 4; j++)
                red_add_v4(row + 4 * j, v[4 * j] * fh, v[4 * j + 1] * fh, v[4 * j + 2] * fh, v[4 * j + 3] * fh);
        }
    }
}

// With M = max(m of the record, m of the state): record = record 2^(m_rec -
// M) + state 2^(m - M), for m, l and every summed dimension.  The record is
// read as it stands in L2 (earlier folds were atomic adds there).
template <int NP, typename VD, typename Fin>
__device__ __forceinline__ void merge_warp_partial(WarpState &st, float *rec_base, int gqa, Fin fin) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const PairColumns<NP> pc(gqa);
    float mp = kNegInf, lp = 0.f;
    if (c < gqa) {
        mp = __ldcg(rec_base + c * kPartStride);
        lp = __ldcg(rec_base + c * kPartStride + 1);
    }
    const float l = warp_sum_g(st.l);
    const float We = warp_sum_g(st.wsum);
    const float Wo = NP == 2 ? warp_sum_g(st.wsum_odd) : 0.f;
    const float M = fmaxf(mp, st.m);
    const float fp = M == kNegInf ? 0.f : ex2(mp - M), fn = M == kNegInf ? 0.f : ex2(st.m - M);
    __syncwarp();  // every lane has read the record's m and l before they are rewritten
    if (c < gqa && g == 0) {
        rec_base[c * kPartStride] = M;
        rec_base[c * kPartStride + 1] = lp * fp + l * fn;
    }
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const int src = (lane & ~3) | ((2 * c + e) & 3);
        const float fph = __shfl_sync(0xffffffffu, fp, src), fnh = __shfl_sync(0xffffffffu, fn, src);
        const float Wse = __shfl_sync(0xffffffffu, We, src), Wso = __shfl_sync(0xffffffffu, Wo, src);
        const float Wh = pc.odd ? Wso : Wse;
        if (pc.wr[e]) {
            float4 *row = reinterpret_cast<float4 *>(rec_base + pc.h[e] * kPartStride + 4 + 16 * g);
            float4 o[4];
#pragma unroll
            for (int j = 0; j < 4; j++) o[j] = __ldcg(row + j);
            float v[16];
            lane_rows<VD>(st, e, Wh, fin, v);
#pragma unroll
            for (int j = 0; j < 4; j++)
                row[j] = make_float4(o[j].x * fph + v[4 * j] * fnh, o[j].y * fph + v[4 * j + 1] * fnh,
                                     o[j].z * fph + v[4 * j + 2] * fnh, o[j].w * fph + v[4 * j + 3] * fnh);
        }
    }
}

// After a spill the state restarts from zero sums, keeping its reference max.
__device__ __forceinline__ void restart_sums(WarpState &st) {
    st.l = 0.f;
    st.wsum = 0.f;
    st.wsum_odd = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; mt++)
#pragma unroll
        for (int q = 0; q < 4; q++) st.acc[mt][q] = 0.f;
}

// Merge the four warps' states through shared memory and write the CTA's
// partial record.  dim_of(mt, r) gives the head dimension of accumulator row r
// (0: row g, 1: row g+8) of m-tile mt for this thread.
template <typename DimOf>
__device__ __forceinline__ void write_partial(WarpState &st, float *scratch, float *part, int gqa,
                                              DimOf dim_of) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, c = lane & 3;
    float *wm = scratch;          // [4 warps][4 heads]
    float *wl = scratch + 16;     // [4][4]
    float *wacc = scratch + 32;   // [4 warps][4 heads][128]
    const float l = warp_sum_g(st.l);
    if ((lane >> 2) == 0) {
        wm[warp * 4 + c] = st.m;
        wl[warp * 4 + c] = l;
    }
#pragma unroll
    for (int mt = 0; mt < 8; mt++) {
        float *dst = wacc + (warp * 4 + c) * kD;
        dst[dim_of(mt, 0)] = st.acc[mt][0] + st.acc[mt][1];
        dst[dim_of(mt, 1)] = st.acc[mt][2] + st.acc[mt][3];
    }
    __syncthreads();
    const int head = threadIdx.x >> 5;
    if (head < gqa) {
        float M = kNegInf;
    #pragma unroll
        for (int w = 0; w < kThreads / 32; w++) M = fmaxf(M, wm[w * 4 + head]);
        float f[kThreads / 32];
        float L = 0.f;
    #pragma unroll
        for (int w = 0; w < kThreads / 32; w++) {
            f[w] = (M == kNegInf) ? 0.f : ex2(wm[w * 4 + head] - M);
            L += f[w] * wl[w * 4 + head];
        }
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    #pragma unroll
        for (int w = 0; w < kThreads / 32; w++) {
            const float4 v = *reinterpret_cast<const float4 *>(wacc + (w * 4 + head) * kD + 4 * lane);
            a.x += f[w] * v.x;
            a.y += f[w] * v.y;
            a.z += f[w] * v.z;
            a.w += f[w] * v.w;
        }
        float *rec = part + head * kPartStride;
        if (lane == 0) {
            rec[0] = M;
            rec[1] = L;
        }
        *reinterpret_cast<float4 *>(rec + 4 + 4 * lane) = a;
    }
}

// ------------------------------------------------------------ rotations
// Walsh-Hadamard transform of a 128-vector held by one warp (lane owns dims
// 4 lane .. 4 lane + 3): stages 1, 2 in registers, 4..64 by shuffles.
__device__ __forceinline__ void warp_wht(float (&x)[4], int lane) {
    const float t0 = x[0] + x[1], t1 = x[0] - x[1], t2 = x[2] + x[3], t3 = x[2] - x[3];
    x[0] = t0 + t2;
    x[2] = t0 - t2;
    x[1] = t1 + t3;
    x[3] = t1 - t3;
#pragma unroll
    for (int hl = 1; hl < 32; hl <<= 1) {
        const bool upper = lane & hl;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float o = __shfl_xor_sync(0xffffffffu, x[e], hl);
            x[e] = upper ? (o - x[e]) : (x[e] + o);
        }
    }
}

__device__ __forceinline__ void apply_signs(float (&x)[4], const uint32_t *sign_bits, int lane) {
    const uint32_t w = sign_bits[lane >> 3] >> ((4 * lane) & 31);
#pragma unroll
    for (int e = 0; e < 4; e++)
        if ((w >> e) & 1u) x[e] = -x[e];
}

// y = R x for a warp-held vector: R = binary32(1/sqrt(d)) D H D.
__device__ __forceinline__ void warp_rotate(float (&x)[4], const uint32_t *sign_bits, float inv_sqrt_d, int lane) {
    apply_signs(x, sign_bits, lane);
    warp_wht(x, lane);
    apply_signs(x, sign_bits, lane);
#pragma unroll
    for (int e = 0; e < 4; e++) x[e] *= inv_sqrt_d;
}

// Dense rotation of a warp-held vector (lane holds coordinates 4 lane + e):
// y = Q x (transpose = false) or y = Q^T x, Q row-major d x d.  Each step
// reads one row of Q with one coalesced 16-byte load per lane.
// y_e = M[4 lane + e] . x for a 128 x 128 binary32 row-major M (16-byte
// aligned), x and y held as coordinates 4 lane .. 4 lane + 3 of each lane.
// Each row is read whole by the warp (a float4 per lane against the lane's
// four coordinates), so every load is one coalesced 512-byte row; the 32 rows
// {4 r + e} of block e are then summed across the lanes by recursive halving
// (step h: a lane keeps the half of its rows selected by its bit h and adds
// its partner's partials of them), which leaves row 4 L + e on lane L: 31
// shuffles per 32 rows instead of 5 per row.
__device__ __forceinline__ void warp_matvec(const float *M, const float (&x)[4], float (&y)[4], int lane) {
#pragma unroll
    for (int e = 0; e < 4; e++) {
        float pr[32];
#pragma unroll
        for (int r = 0; r < 32; r++) {
            const float4 m = __ldg(reinterpret_cast<const float4 *>(M + static_cast<size_t>(4 * r + e) * kD) + lane);
            pr[r] = fmaf(m.w, x[3], fmaf(m.z, x[2], fmaf(m.y, x[1], m.x * x[0])));
        }
#pragma unroll
        for (int h = 16; h >= 1; h >>= 1) {
            const bool up = (lane & h) != 0;
#pragma unroll
            for (int r = 0; r < h; r++) {
                const float send = up ? pr[r] : pr[r + h];
                const float keep = up ? pr[r + h] : pr[r];
                pr[r] = keep + __shfl_xor_sync(0xffffffffu, send, h);
            }
        }
        y[e] = pr[0];
    }
}

__device__ __forceinline__ void warp_rotate_dense(float (&x)[4], const float *Q, bool transpose, int lane) {
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    if (transpose) {  // y_j = sum_i Q[i][j] x_i
#pragma unroll 4
        for (int i = 0; i < kD; i++) {
            const float xi = __shfl_sync(0xffffffffu, x[i & 3], i >> 2);
            const float4 r = __ldg(reinterpret_cast<const float4 *>(Q + static_cast<size_t>(i) * kD) + lane);
            y[0] = fmaf(r.x, xi, y[0]);
            y[1] = fmaf(r.y, xi, y[1]);
            y[2] = fmaf(r.z, xi, y[2]);
            y[3] = fmaf(r.w, xi, y[3]);
        }
    } else {  // y_j = sum_i Q[j][i] x_i
        warp_matvec(Q, x, y, lane);
    }
#pragma unroll
    for (int e = 0; e < 4; e++) x[e] = y[e];
}

__device__ __forceinline__ void load_q4(const uint16_t *q, int lane, float (&x)[4]) {
    const uint2 v = reinterpret_cast<const uint2 *>(q)[lane];
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
    x[0] = f0.x;
    x[1] = f0.y;
    x[2] = f1.x;
    x[3] = f1.y;
}

// Power of two f such that f * max|x| over the warp lies in [0.5, 1) (1 for
// an all-zero or non-finite vector): scaling by f is exact.
__device__ __forceinline__ float warp_pow2_norm(const float (&x)[4]) {
    float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (!(m > 0.f) || !(m < __builtin_huge_valf())) return 1.f;
    int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 126;  // m in [2^(e-1), 2^e)
    e = max(-100, min(100, e));
    return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// fp16 hi and lo = x - hi of a warp-held vector as half2 words (dims 2i, 2i+1
// in word i): dst[0..63] hi, dst[64..127] lo; returns sum(hi + lo) over the warp.
__device__ __forceinline__ float store_hilo(uint32_t *dst, const float (&x)[4], int lane) {
    __half hi[4], lo[4];
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; e++) {
        hi[e] = __float2half_rn(x[e]);
        lo[e] = __float2half_rn(x[e] - __half2float(hi[e]));
        s += __half2float(hi[e]) + __half2float(lo[e]);
    }
    dst[2 * lane] = pack_half2(hi[0], hi[1]);
    dst[2 * lane + 1] = pack_half2(hi[2], hi[3]);
    dst[64 + 2 * lane] = pack_half2(lo[0], lo[1]);
    dst[64 + 2 * lane + 1] = pack_half2(lo[2], lo[3]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// ------------------------------------------------------------ head_dim 128 nh
// A warp-held vector of nh 128-dim blocks: x[j][e] is dimension 128 j + 4 lane + e.

// y = R x with R = binary32(1/sqrt(d)) D H D, d = 128 nh: the Walsh-Hadamard
// transform of each block, then the butterflies between blocks (widths 128,
// 256, ...) in registers; block j's signs are words 4 j .. 4 j + 3.
template <int NH>
__device__ __forceinline__ void warp_rotate_wide(float (&x)[NH][4], const uint32_t *sign_bits, float inv_sqrt_d,
                                                 int lane) {
#pragma unroll
    for (int j = 0; j < NH; j++) {
        apply_signs(x[j], sign_bits + 4 * j, lane);
        warp_wht(x[j], lane);
    }
#pragma unroll
    for (int w = 1; w < NH; w <<= 1) {
#pragma unroll
        for (int j = 0; j < NH; j++) {
            if (j & w) continue;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float a = x[j][e], b = x[j + w][e];
                x[j][e] = a + b;
                x[j + w][e] = a - b;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NH; j++) {
        apply_signs(x[j], sign_bits + 4 * j, lane);
#pragma unroll
        for (int e = 0; e < 4; e++) x[j][e] *= inv_sqrt_d;
    }
}

// y = R x for a 64-vector on lanes 0..15 (lane l: dims 4 l .. 4 l + 3); lanes
// 16..31 run the same steps on their own copy (shuffles stay within each half).
__device__ __forceinline__ void warp_rotate_64(float (&x)[4], const uint32_t *sign_bits, float inv_sqrt_d,
                                               int lane) {
    const int l = lane & 15;
    apply_signs(x, sign_bits, l);
    const float t0 = x[0] + x[1], t1 = x[0] - x[1], t2 = x[2] + x[3], t3 = x[2] - x[3];
    x[0] = t0 + t2;
    x[2] = t0 - t2;
    x[1] = t1 + t3;
    x[3] = t1 - t3;
#pragma unroll
    for (int hl = 1; hl < 16; hl <<= 1) {
        const bool upper = lane & hl;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float o = __shfl_xor_sync(0xffffffffu, x[e], hl);
            x[e] = upper ? (o - x[e]) : (x[e] + o);
        }
    }
    apply_signs(x, sign_bits, l);
#pragma unroll
    for (int e = 0; e < 4; e++) x[e] *= inv_sqrt_d;
}

// warp_pow2_norm over all blocks.
template <int NH>
__device__ __forceinline__ float warp_pow2_norm_wide(const float (&x)[NH][4]) {
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < NH; j++)
        m = fmaxf(m, fmaxf(fmaxf(fabsf(x[j][0]), fabsf(x[j][1])), fmaxf(fabsf(x[j][2]), fabsf(x[j][3]))));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (!(m > 0.f) || !(m < __builtin_huge_valf())) return 1.f;
    int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 126;
    e = max(-100, min(100, e));
    return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// fp16 hi and lo = x - hi of block j as half2 words: hi at hi[64 j + 2 lane, +1],
// lo at lo[64 j + 2 lane, +1]; returns this lane's sum of hi + lo.
__device__ __forceinline__ float store_hilo_block(uint32_t *hi_w, uint32_t *lo_w, const float (&x)[4], int j,
                                                  int lane) {
    __half hi[4], lo[4];
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; e++) {
        hi[e] = __float2half_rn(x[e]);
        lo[e] = __float2half_rn(x[e] - __half2float(hi[e]));
        s += __half2float(hi[e]) + __half2float(lo[e]);
    }
    hi_w[64 * j + 2 * lane] = pack_half2(hi[0], hi[1]);
    hi_w[64 * j + 2 * lane + 1] = pack_half2(hi[2], hi[3]);
    lo_w[64 * j + 2 * lane] = pack_half2(lo[0], lo[1]);
    lo_w[64 * j + 2 * lane + 1] = pack_half2(lo[2], lo[3]);
    return s;
}

// Named barrier over `threads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------ dependent launches
// Let the next kernel of the call start launching CTAs into free SM slots.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Wait until the previous kernel of the call has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------ fused combine
// After a CTA wrote its partial record(s) of (layer, batch b, KV head h): count
// the CTA; the CTA that brings the count to the group's total merges every
// partial record of the group (no CTA ever waits for another).  Warp w merges query head h*gqa + w:
// max-rescale merge of the packed-space and fp16-space sums, one inverse
// rotation of the packed sum (R is its own inverse), normalisation, store.
// Called by all threads; returns with all threads synchronised.  `flag` is one
// int of shared memory.
//
// With NH > 1 (head_dim 128 NH) record r of a group holds 128-dim block r mod
// NH of its query head's sum; the NH records of one warp group (or fp16
// chunk) carry the same m and l, counted once.
template <int NH>
__device__ __forceinline__ void combine_wide(const DecodeDims &dims, const DecodeWorkspace &ws, int layer, int b,
                                             int h, int warp, int lane);
// NP = 2 (head_dim 64): records hold 128 virtual dims, the sum over even
// tokens in dims 0..63 and over odd tokens in 64..127; the merge adds them.
__device__ __forceinline__ void combine_np2(const DecodeDims &dims, const DecodeWorkspace &ws, int layer, int b,
                                            int h, int warp, int lane);

template <int NH = 1, int NP = 1>
__device__ __forceinline__ void finish_and_combine(const DecodeDims &dims, const DecodeWorkspace &ws, int layer,
                                                   int b, int h, int *flag) {
    __threadfence();
    __syncthreads();
    const size_t lbh = (static_cast<size_t>(layer) * dims.B + b) * dims.H + h;
    if (threadIdx.x == 0) {
        const int done = atomicAdd(ws.counter + lbh, 1);
        *flag = (done == ws.lbh_total[lbh] - 1);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if constexpr (NH > 1) {
        if (*flag && warp < dims.gqa) {
            __threadfence();
            combine_wide<NH>(dims, ws, layer, b, h, warp, lane);
        }
    } else if constexpr (NP == 2) {
        if (*flag && warp < dims.gqa) {
            __threadfence();
            combine_np2(dims, ws, layer, b, h, warp, lane);
        }
    } else if (*flag && warp < dims.gqa) {
        __threadfence();
        const LayerPlan &lp = ws.layer[layer];
        const int n_items = lp.n_items[h];
        const size_t rec_stride = kMaxGqa * kPartStride;
        // one pass over the records with an online max: eight records'
        // loads in flight at a time (records of warps without tokens have
        // m = -inf and contribute nothing)
        float M = kNegInf, L = 0.f;
        float ar[4] = {0.f, 0.f, 0.f, 0.f}, ao[4] = {0.f, 0.f, 0.f, 0.f};
        for (int ii = 0; ii < n_items; ii++) {
            const int item = lp.item[h][ii];
            const size_t gr = static_cast<size_t>(item) * dims.B + b;
            const int p0 = ws.grp_part[gr], np = ws.grp_nparts[gr];
            const bool rot = ws.items[item].kind == TQ_SEG_PACKED;  // rotated-space sums
            const float *base = ws.part + static_cast<size_t>(p0) * rec_stride + warp * kPartStride;
            for (int c0 = 0; c0 < np; c0 += 8) {
                float m[8], l[8];
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    const int c = min(c0 + u, np - 1);
                    const float *rec = base + static_cast<size_t>(c) * rec_stride;
                    m[u] = c0 + u < np ? __ldcg(rec) : kNegInf;
                    l[u] = __ldcg(rec + 1);
                    v[u] = __ldcg(reinterpret_cast<const float4 *>(rec + 4) + lane);
                }
                float mc = m[0];
#pragma unroll
                for (int u = 1; u < 8; u++) mc = fmaxf(mc, m[u]);
                if (mc > M) {  // a new running max: rescale what is summed so far
                    const float sc = ex2(M - mc);
                    L *= sc;
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        ar[e] *= sc;
                        ao[e] *= sc;
                    }
                    M = mc;
                }
                float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    if (m[u] == kNegInf) continue;
                    const float f = ex2(m[u] - M);
                    L += f * l[u];
                    a[0] += f * v[u].x;
                    a[1] += f * v[u].y;
                    a[2] += f * v[u].z;
                    a[3] += f * v[u].w;
                }
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    ar[e] += rot ? a[e] : 0.f;
                    ao[e] += rot ? 0.f : a[e];
                }
            }
        }
        if (lp.dense) warp_rotate_dense(ar, lp.dense, true, lane);
        else warp_rotate(ar, lp.sign_bits, dims.inv_sqrt_d, lane);
        const float inv = L > 0.f ? 1.0f / L : 0.f;
        float4 o;
        o.x = (ar[0] + ao[0]) * inv;
        o.y = (ar[1] + ao[1]) * inv;
        o.z = (ar[2] + ao[2]) * inv;
        o.w = (ar[3] + ao[3]) * inv;
        const size_t qrow = (static_cast<size_t>(layer) * dims.B + b) * dims.Hq + h * dims.gqa + warp;
        reinterpret_cast<float4 *>(ws.out + qrow * kD)[lane] = o;
        if (ws.ml && lane == 0) {  // for the attention-mass kernel
            ws.ml[qrow * 2] = M;
            ws.ml[qrow * 2 + 1] = L;
        }
    }
    __syncthreads();
}

template <int NH>
__device__ __forceinline__ void combine_wide(const DecodeDims &dims, const DecodeWorkspace &ws, int layer, int b,
                                             int h, int warp, int lane) {
    static_assert(NH == 2 || NH == 4, "records are read eight at a time, NH | 8");
    const LayerPlan &lp = ws.layer[layer];
    const int n_items = lp.n_items[h];
    const size_t rec_stride = kMaxGqa * kPartStride;
    float M = kNegInf, L = 0.f;
    float ar[NH][4], ao[NH][4];
#pragma unroll
    for (int j = 0; j < NH; j++)
#pragma unroll
        for (int e = 0; e < 4; e++) ar[j][e] = ao[j][e] = 0.f;
    for (int ii = 0; ii < n_items; ii++) {
        const int item = lp.item[h][ii];
        const size_t gr = static_cast<size_t>(item) * dims.B + b;
        const int p0 = ws.grp_part[gr], np = ws.grp_nparts[gr];
        const bool rot = ws.items[item].kind == TQ_SEG_PACKED;
        const float *base = ws.part + static_cast<size_t>(p0) * rec_stride + warp * kPartStride;
        for (int c0 = 0; c0 < np; c0 += 8) {  // record c0 + u holds block u mod NH
            float m[8], l[8];
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int c = min(c0 + u, np - 1);
                const float *rec = base + static_cast<size_t>(c) * rec_stride;
                m[u] = c0 + u < np ? __ldcg(rec) : kNegInf;
                l[u] = __ldcg(rec + 1);
                v[u] = __ldcg(reinterpret_cast<const float4 *>(rec + 4) + lane);
            }
            float mc = m[0];
#pragma unroll
            for (int u = 1; u < 8; u++) mc = fmaxf(mc, m[u]);
            if (mc > M) {
                const float sc = ex2(M - mc);
                L *= sc;
#pragma unroll
                for (int j = 0; j < NH; j++)
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        ar[j][e] *= sc;
                        ao[j][e] *= sc;
                    }
                M = mc;
            }
            float a[NH][4];
#pragma unroll
            for (int j = 0; j < NH; j++)
#pragma unroll
                for (int e = 0; e < 4; e++) a[j][e] = 0.f;
#pragma unroll
            for (int u = 0; u < 8; u++) {
                if (m[u] == kNegInf) continue;
                const float f = ex2(m[u] - M);
                if (u % NH == 0) L += f * l[u];
                a[u % NH][0] += f * v[u].x;
                a[u % NH][1] += f * v[u].y;
                a[u % NH][2] += f * v[u].z;
                a[u % NH][3] += f * v[u].w;
            }
#pragma unroll
            for (int j = 0; j < NH; j++)
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    ar[j][e] += rot ? a[j][e] : 0.f;
                    ao[j][e] += rot ? 0.f : a[j][e];
                }
        }
    }
    warp_rotate_wide<NH>(ar, lp.sign_bits, dims.inv_sqrt_d, lane);
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    const size_t qrow = (static_cast<size_t>(layer) * dims.B + b) * dims.Hq + h * dims.gqa + warp;
    float4 *dst = reinterpret_cast<float4 *>(ws.out + qrow * (NH * kD));
#pragma unroll
    for (int j = 0; j < NH; j++)
        dst[32 * j + lane] = make_float4((ar[j][0] + ao[j][0]) * inv, (ar[j][1] + ao[j][1]) * inv,
                                         (ar[j][2] + ao[j][2]) * inv, (ar[j][3] + ao[j][3]) * inv);
}

__device__ __forceinline__ void combine_np2(const DecodeDims &dims, const DecodeWorkspace &ws, int layer, int b,
                                            int h, int warp, int lane) {
    const LayerPlan &lp = ws.layer[layer];
    const int n_items = lp.n_items[h];
    const size_t rec_stride = kMaxGqa * kPartStride;
    float M = kNegInf, L = 0.f;
    float ar[4] = {0.f, 0.f, 0.f, 0.f}, ao[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ii = 0; ii < n_items; ii++) {
        const int item = lp.item[h][ii];
        const size_t gr = static_cast<size_t>(item) * dims.B + b;
        const int p0 = ws.grp_part[gr], np = ws.grp_nparts[gr];
        const bool rot = ws.items[item].kind == TQ_SEG_PACKED;
        const float *base = ws.part + static_cast<size_t>(p0) * rec_stride + warp * kPartStride;
        for (int c0 = 0; c0 < np; c0 += 8) {
            float m[8], l[8];
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int c = min(c0 + u, np - 1);
                const float *rec = base + static_cast<size_t>(c) * rec_stride;
                m[u] = c0 + u < np ? __ldcg(rec) : kNegInf;
                l[u] = __ldcg(rec + 1);
                v[u] = __ldcg(reinterpret_cast<const float4 *>(rec + 4) + lane);
            }
            float mc = m[0];
#pragma unroll
            for (int u = 1; u < 8; u++) mc = fmaxf(mc, m[u]);
            if (mc > M) {
                const float sc = ex2(M - mc);
                L *= sc;
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    ar[e] *= sc;
                    ao[e] *= sc;
                }
                M = mc;
            }
            float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int u = 0; u < 8; u++) {
                if (m[u] == kNegInf) continue;
                const float f = ex2(m[u] - M);
                L += f * l[u];
                a[0] += f * v[u].x;
                a[1] += f * v[u].y;
                a[2] += f * v[u].z;
                a[3] += f * v[u].w;
            }
#pragma unroll
            for (int e = 0; e < 4; e++) {
                ar[e] += rot ? a[e] : 0.f;
                ao[e] += rot ? 0.f : a[e];
            }
        }
    }
    // virtual dims 4 lane + e: lanes 16..31 hold the odd tokens' dims 4 (lane - 16) + e
#pragma unroll
    for (int e = 0; e < 4; e++) {
        ar[e] += __shfl_xor_sync(0xffffffffu, ar[e], 16);
        ao[e] += __shfl_xor_sync(0xffffffffu, ao[e], 16);
    }
    warp_rotate_64(ar, lp.sign_bits, dims.inv_sqrt_d, lane);
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    const size_t qrow = (static_cast<size_t>(layer) * dims.B + b) * dims.Hq + h * dims.gqa + warp;
    if (lane < 16)
        reinterpret_cast<float4 *>(ws.out + qrow * (kD / 2))[lane] =
            make_float4((ar[0] + ao[0]) * inv, (ar[1] + ao[1]) * inv, (ar[2] + ao[2]) * inv, (ar[3] + ao[3]) * inv);
}

// Write one warp's state as a partial record (no cross-warp merge): for each
// query head c < gqa, m (base-2 units) and l, and the 128 accumulator dims;
// dim_of(mt, r) is the head dimension of accumulator row r of m-tile mt.
template <typename DimOf>
__device__ __forceinline__ void write_warp_partial(WarpState &st, float *rec_base, int gqa, DimOf dim_of) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const float l = warp_sum_g(st.l);
    if (c < gqa) {
        float *rec = rec_base + c * kPartStride;
        if (g == 0) {
            rec[0] = st.m;
            rec[1] = l;
        }
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            rec[4 + dim_of(mt, 0)] = st.acc[mt][0] + st.acc[mt][1];
            rec[4 + dim_of(mt, 1)] = st.acc[mt][2] + st.acc[mt][3];
        }
    }
}

// Equal contiguous ranges of S stages over G persistent CTAs: CTA i takes
// [i S / G, (i+1) S / G); the CTA holding stage s is the last i with
// i S / G <= s.
__host__ __device__ __forceinline__ long long range_begin(long long i, long long S, long long G) { return i * S / G; }
__host__ __device__ __forceinline__ long long cta_of_stage(long long s, long long S, long long G) {
    return ((s + 1) * G + S - 1) / S - 1;
}

}  // namespace dec
}  // namespace tqk
