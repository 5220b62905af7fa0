// tq_decode.cu -- decode attention directly on the compressed KV cache.
//
// Method: "turboquant-mlx" skill note, "Optimisations Metal" (fused attention on
// the compressed cache, the inverse transform pulled out of the V sum);
// "turboquant-mlx" (TurboQuant-MLX v2.0 README), "Implementation Status"
// (compressed-domain attention) and "RaBitQ vs QJL correction"; "TurboMOQ",
// "QJL residual correction (sub-2-bit)".
//
// Because R is orthogonal and symmetric, q . (R yhat) = (R q) . yhat: the query
// is rotated once (prep kernel), scores and the value sum run on the packed
// codes in the rotated space, and one inverse rotation is applied to the merged
// value sum (combine kernel).  Keys dequantize affinely, yhat = alpha*code + beta
// (alpha = m 2^(1-b), beta = m (2^-b - 1)), so q'.yhat = alpha (q'.code) +
// beta sum(q'): the tensor cores multiply the raw integer codes.
//
// Split-K flash decoding (GB300): one CTA of 4 warps per (segment, batch, KV
// head, token chunk).  Packed records stream through a 4-stage cp.async
// pipeline in 64-token stages; each warp owns a 16-token tile per stage and runs
//   Q.K : mma.m16n8k16 with A = 16 tokens x 16 dims of raw codes (as fp16
//         subnormals, exact) and B = the 4 query heads of the GQA group, each
//         split into fp16 hi + lo columns (8 columns, no padding);
//   softmax: online, in base 2, per query head;
//   P.V : mma.m16n8k16 with A = 16 dims x 16 tokens of fp16 codebook values and
//         B = probabilities times the value scale, again hi + lo columns.
// Each CTA writes one partial (m, l, acc) per query head; the combine kernel
// merges partials across chunks and segments, rotates the packed-space sum
// back and adds the fp16-segment sum.  No CTA waits on another.
#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tqk {
namespace {

constexpr int kThreads = 128;
constexpr int kPartStride = 4 + kD;  // m, l, pad, pad, acc[d]
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

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return static_cast<uint32_t>(__half_as_ushort(lo)) |
           (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

__device__ __forceinline__ float warp_max_g(float v) {  // over the 8 lanes sharing lane&3
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

// Bits [B*j, B*j + B) of a little-endian word window (j compile-time).
template <int B, int NW>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[NW], int j) {
    const int bit = B * j, wi = bit >> 5, sh = bit & 31;
    uint32_t v;
    if (sh + B <= 32) {
        v = w[wi] >> sh;
    } else {
        v = __funnelshift_r(w[wi], w[wi + 1], sh);
    }
    return v & ((1u << B) - 1u);
}

// Codes j and j+1 as a pair of fp16 subnormals (code * 2^-24, exact).
template <int B, int NW>
__device__ __forceinline__ uint32_t code_pair(const uint32_t (&w)[NW], int j) {
    return code_at<B>(w, j) | (code_at<B>(w, j + 1) << 16);
}

template <int NW>
__device__ __forceinline__ void lds_words(uint32_t (&w)[NW], const uint8_t *p) {
    if constexpr (NW % 4 == 0) {
#pragma unroll
        for (int i = 0; i < NW / 4; i++) {
            const uint4 v = reinterpret_cast<const uint4 *>(p)[i];
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
    } else if constexpr (NW % 2 == 0) {
#pragma unroll
        for (int i = 0; i < NW / 2; i++) {
            const uint2 v = reinterpret_cast<const uint2 *>(p)[i];
            w[2 * i] = v.x; w[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < NW; i++) w[i] = reinterpret_cast<const uint32_t *>(p)[i];
    }
}

// Raw Q.K of a 16-token tile: thread (g, c) owns dims [32c, 32c+32) of the
// record.  MMA k-column 2c+e of k-step kk is dim 32c + 4kk + e and column
// 2c+8+e is dim 32c + 4kk + 2 + e, so each A register holds two adjacent codes.
// Returns the hi+lo-combined dot products for tokens g and g+8 (head c).
template <int B>
__device__ __forceinline__ void qk_tile(const uint8_t *rec0, const uint8_t *rec1,
                                        const uint32_t (&bq)[8][2], float &raw0, float &raw1) {
    uint32_t w0[B], w1[B];
    lds_words(w0, rec0);
    lds_words(w1, rec1);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
        mma16816(acc, code_pair<B>(w0, 4 * kk), code_pair<B>(w1, 4 * kk), code_pair<B>(w0, 4 * kk + 2),
                 code_pair<B>(w1, 4 * kk + 2), bq[kk][0], bq[kk][1]);
    }
    raw0 = acc[0] + acc[1];
    raw1 = acc[2] + acc[3];
}

// Scores (already scaled to base-2 logits) of tokens g and g+8 for head c.
template <int KB, bool QJL>
__device__ __forceinline__ void kphase(const uint8_t *kst, const uint8_t *qst, const float *kscale,
                                       const float *qnorm, int tile0, int g, int c,
                                       const uint32_t (&bq)[8][2], const uint32_t (&bt)[8][2],
                                       float qsum, float tsum, float qk_scale, float (&s)[2]) {
    constexpr int RK = 16 * KB;
    float raw0, raw1;
    qk_tile<KB>(kst + (tile0 + g) * RK + 4 * KB * c, kst + (tile0 + g + 8) * RK + 4 * KB * c, bq,
                raw0, raw1);
    // alpha includes the 2^24 of the subnormal encoding
    constexpr float alpha_u = 16777216.0f * 2.0f / static_cast<float>(1 << KB);
    constexpr float beta_u = 1.0f / static_cast<float>(1 << KB) - 1.0f;
    const float m0 = kscale[tile0 + g], m1 = kscale[tile0 + g + 8];
    s[0] = m0 * (alpha_u * raw0 + beta_u * qsum);
    s[1] = m1 * (alpha_u * raw1 + beta_u * qsum);
    if constexpr (QJL) {
        float r0, r1;
        qk_tile<1>(qst + (tile0 + g) * 16 + 4 * c, qst + (tile0 + g + 8) * 16 + 4 * c, bt, r0, r1);
        // <S q', s> with s = 2 bit - 1: 2 (sum over set bits) - sum(t)
        constexpr float gam = 1.2533141373155003f / kJl;  // sqrt(pi/2) / jl
        s[0] += gam * qnorm[tile0 + g] * (33554432.0f * r0 - tsum);
        s[1] += gam * qnorm[tile0 + g + 8] * (33554432.0f * r1 - tsum);
    }
    s[0] *= qk_scale;
    s[1] *= qk_scale;
}

// P.V of a tile: thread (g, c) handles dims [16g, 16g+16) of the record (MMA row
// (mt, g) = dim 16g + 2mt, row (mt, g+8) = dim 16g + 2mt + 1) for tokens 2c,
// 2c+1, 2c+8, 2c+9.  Codebook values come from a shared fp16 table.
template <int VB>
__device__ __forceinline__ void vphase(const uint8_t *vst, int tile0, int g, int c,
                                       const unsigned short *ctab, uint32_t b0, uint32_t b1,
                                       float (&acc)[8][4]) {
    constexpr int RV = 16 * VB;
    constexpr int NW = (2 * VB + 3) / 4 + 1;  // words covering the 2*VB-byte window + shift
    const int off = 2 * VB * g;
    const int sh = (off & 3) * 8;
    uint32_t x[4][NW];
#pragma unroll
    for (int tt = 0; tt < 4; tt++) {
        const int tok = tile0 + 2 * c + (tt & 1) + (tt >> 1) * 8;
        const uint32_t *p = reinterpret_cast<const uint32_t *>(vst + tok * RV + (off & ~3));
        uint32_t raw[NW];
#pragma unroll
        for (int i = 0; i < NW - 1; i++) raw[i] = p[i];
        raw[NW - 1] = 0;
#pragma unroll
        for (int i = 0; i < NW - 1; i++) x[tt][i] = __funnelshift_r(raw[i], raw[i + 1], sh);
        x[tt][NW - 1] = 0;
    }
#pragma unroll
    for (int mt = 0; mt < 8; mt++) {
        uint32_t a[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int j = 2 * mt + (q & 1);     // a0: row g (even dim), a1: row g+8 (odd)
            const int ta = (q >> 1) * 2;        // a0/a1: tokens 2c, 2c+1; a2/a3: 2c+8, 2c+9
            const unsigned short lo = ctab[code_at<VB>(x[ta], j)];
            const unsigned short hi = ctab[code_at<VB>(x[ta + 1], j)];
            a[q] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        mma16816(acc[mt], a[0], a[1], a[2], a[3], b0, b1);
    }
}

struct WarpState {
    float m, l;
    float acc[8][4];
};

// Online softmax update for one tile and the B fragment of the probabilities.
__device__ __forceinline__ void softmax_tile(WarpState &st, float (&s)[2], const bool (&valid)[2],
                                             const float (&vs)[2], int g, int c, bool head_ok,
                                             uint32_t &b0, uint32_t &b1) {
    float t = fmaxf(valid[0] ? s[0] : kNegInf, valid[1] ? s[1] : kNegInf);
    t = warp_max_g(t);
    const float mnew = fmaxf(st.m, t);
    float corr, p0, p1;
    if (mnew == kNegInf) {
        corr = 1.f;
        p0 = p1 = 0.f;
    } else {
        corr = exp2f(st.m - mnew);
        p0 = valid[0] ? exp2f(s[0] - mnew) : 0.f;
        p1 = valid[1] ? exp2f(s[1] - mnew) : 0.f;
    }
    st.l = st.l * corr + p0 + p1;
    st.m = mnew;
#pragma unroll
    for (int mt = 0; mt < 8; mt++)
#pragma unroll
        for (int q = 0; q < 4; q++) st.acc[mt][q] *= corr;
    float w0 = head_ok ? p0 * vs[0] : 0.f;
    float w1 = head_ok ? p1 * vs[1] : 0.f;
    // transpose: column n = g (head g/2, part g&1) needs tokens 2c, 2c+1, 2c+8, 2c+9
    const int src0 = 8 * c + (g >> 1), src1 = src0 + 4;
    const float v0 = __shfl_sync(0xffffffffu, w0, src0);
    const float v1 = __shfl_sync(0xffffffffu, w0, src1);
    const float v2 = __shfl_sync(0xffffffffu, w1, src0);
    const float v3 = __shfl_sync(0xffffffffu, w1, src1);
    const bool lo = g & 1;
    auto part = [lo](float v) {
        const __half h = __float2half_rn(v);
        return lo ? __float2half_rn(v - __half2float(h)) : h;
    };
    b0 = pack_half2(part(v0), part(v1));
    b1 = pack_half2(part(v2), part(v3));
}

// Merge the four warps' states through shared memory and write the CTA's
// partial record.  space: 0 = packed (rotated, dims owned per thread as
// 16g + 2mt + {0,1}), 1 = fp16 (original, dims 16mt + g + {0, 8}).
__device__ void write_partial(WarpState &st, float *scratch, float *part, int gqa, int space) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    float *wm = scratch;                    // [4 warps][4 heads]
    float *wl = scratch + 16;               // [4][4]
    float *wacc = scratch + 32;             // [4 warps][4 heads][128]
    const float l = warp_sum_g(st.l);
    if (g == 0) {
        wm[warp * 4 + c] = st.m;
        wl[warp * 4 + c] = l;
    }
#pragma unroll
    for (int mt = 0; mt < 8; mt++) {
        int d0, d1;
        if (space == 0) { d0 = 16 * g + 2 * mt; d1 = d0 + 1; }
        else { d0 = 16 * mt + g; d1 = d0 + 8; }
        float *dst = wacc + (warp * 4 + c) * kD;
        dst[d0] = st.acc[mt][0] + st.acc[mt][1];
        dst[d1] = st.acc[mt][2] + st.acc[mt][3];
    }
    __syncthreads();
    const int head = threadIdx.x >> 5;   // 4 heads x 32 threads, 4 dims each
    if (head >= gqa) return;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; w++) M = fmaxf(M, wm[w * 4 + head]);
    float f[kDecodeWarps];
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; w++) {
        f[w] = (M == kNegInf) ? 0.f : exp2f(wm[w * 4 + head] - M);
        L += f[w] * wl[w * 4 + head];
    }
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kDecodeWarps; w++) {
        const float4 v = *reinterpret_cast<const float4 *>(wacc + (w * 4 + head) * kD + 4 * lane);
        a.x += f[w] * v.x; a.y += f[w] * v.y; a.z += f[w] * v.z; a.w += f[w] * v.w;
    }
    float *rec = part + head * kPartStride;
    if (lane == 0) {
        rec[0] = M;
        rec[1] = L;
    }
    *reinterpret_cast<float4 *>(rec + 4 + 4 * lane) = a;
}

__device__ __forceinline__ int find_segment(const SegPlan *seg, int lo, int hi, int cta) {
    // largest i in [lo, hi) with seg[i].cta_begin <= cta
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (seg[mid].cta_begin <= cta) lo = mid; else hi = mid;
    }
    return lo;
}

struct Tables {
    unsigned short centroid[kCbTotal];  // fp16 bit patterns, flat by bit width
};

// -------------------------------------------------------------- packed kernel
__global__ void __launch_bounds__(kThreads, 3)
    decode_packed_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int n_packed_seg,
                         const int stage_bytes, const __grid_constant__ Tables tab) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int cta = blockIdx.x;
    const int si = find_segment(ws.seg, 0, n_packed_seg, cta);
    const SegPlan &sp = ws.seg[si];
    const int local = cta - sp.cta_begin;
    const int chunk = local % sp.n_chunks;
    const int bh = local / sp.n_chunks;
    const int h = bh % dims.H, b = bh / dims.H;
    const int tok0 = chunk * sp.chunk;
    const int ntok = min(sp.chunk, sp.n_tokens - tok0);
    const int kb = sp.kbits[h], vb = sp.vbits[h];
    const bool qjl = sp.qrank[h] >= 0;
    const int rk = 16 * kb, rv = 16 * vb;
    const int cap = sp.capacity;

    const uint8_t *kc = sp.kcodes + static_cast<size_t>(b) * sp.kblock + sp.koff[h] + static_cast<size_t>(tok0) * rk;
    const uint8_t *vc = sp.vcodes + static_cast<size_t>(b) * sp.vblock + sp.voff[h] + static_cast<size_t>(tok0) * rv;
    const size_t sidx = (static_cast<size_t>(b) * dims.H + h) * cap + tok0;
    const float *ks = sp.kscale + sidx;
    const float *vs = sp.vscale + sidx;
    const uint8_t *qs = nullptr;
    const float *qn = nullptr;
    if (qjl) {
        const size_t qi = (static_cast<size_t>(b) * sp.nq + sp.qrank[h]) * cap + tok0;
        qs = sp.qjl_signs + qi * (kJl / 8);
        qn = sp.qjl_norm + qi;
    }
    // stage layout: [K 64*rk][V 64*rv][kscale 256][vscale 256][signs 1024][norms 256]
    const int offV = kStageTokens * rk, offKS = offV + kStageTokens * rv, offVS = offKS + 256;
    const int offQS = offVS + 256, offQN = offQS + kStageTokens * 16;
    const int n_st = (ntok + kStageTokens - 1) / kStageTokens;

    unsigned short *ctab = reinterpret_cast<unsigned short *>(smem + kStages * stage_bytes);
    for (int i = threadIdx.x; i < (1 << vb); i += kThreads) ctab[i] = tab.centroid[cb_off(vb) + i];

    auto load_stage = [&](int s) {
        uint8_t *dst = smem + (s % kStages) * stage_bytes;
        const int t0 = s * kStageTokens;
        const int n = min(kStageTokens, ntok - t0);
        // chunk lists: K codes, V codes, k scales, v scales, [signs, norms]
        const int nK = kStageTokens * rk / 16, nV = kStageTokens * rv / 16;
        const int nS = kStageTokens * 4 / 16;
        const int nQ = qjl ? kStageTokens * 16 / 16 : 0, nN = qjl ? nS : 0;
        const int total = nK + nV + 2 * nS + nQ + nN;
        for (int i = threadIdx.x; i < total; i += kThreads) {
            const uint8_t *src;
            int valid_bytes, dofs, idx;
            if (i < nK) { idx = i; src = kc + static_cast<size_t>(t0) * rk; valid_bytes = n * rk; dofs = 0; }
            else if (i < nK + nV) { idx = i - nK; src = vc + static_cast<size_t>(t0) * rv; valid_bytes = n * rv; dofs = offV; }
            else if (i < nK + nV + nS) { idx = i - nK - nV; src = reinterpret_cast<const uint8_t *>(ks + t0); valid_bytes = n * 4; dofs = offKS; }
            else if (i < nK + nV + 2 * nS) { idx = i - nK - nV - nS; src = reinterpret_cast<const uint8_t *>(vs + t0); valid_bytes = n * 4; dofs = offVS; }
            else if (i < nK + nV + 2 * nS + nQ) { idx = i - nK - nV - 2 * nS; src = qs + static_cast<size_t>(t0) * 16; valid_bytes = n * 16; dofs = offQS; }
            else { idx = i - nK - nV - 2 * nS - nQ; src = reinterpret_cast<const uint8_t *>(qn + t0); valid_bytes = n * 4; dofs = offQN; }
            const int rem = valid_bytes - idx * 16;
            const int nb = rem >= 16 ? 16 : (rem > 0 ? rem : 0);
            cp_async16_zfill(dst + dofs + idx * 16, nb > 0 ? src + idx * 16 : src, nb);
        }
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int gqa = dims.gqa;
    const int j0 = h * gqa;
    // B fragments of the rotated query (and of S q' for QJL heads)
    uint32_t bq[8][2], bt[8][2];
    float qsum = 0.f, tsum = 0.f;
    {
        const int head = g >> 1, pt = g & 1;
        const size_t qidx = (static_cast<size_t>(sp.layer) * dims.B + b) * dims.Hq + j0 + head;
        const bool ok = head < gqa;
        const uint32_t *qw = ws.qrot + (qidx * 2 + pt) * (kD / 2) + 16 * c;
        const uint32_t *tw = ws.qjlt + (qidx * 2 + pt) * (kD / 2) + 16 * c;
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
            bq[kk][0] = ok ? qw[2 * kk] : 0u;
            bq[kk][1] = ok ? qw[2 * kk + 1] : 0u;
            bt[kk][0] = (ok && qjl) ? tw[2 * kk] : 0u;
            bt[kk][1] = (ok && qjl) ? tw[2 * kk + 1] : 0u;
        }
        if (c < gqa) {
            const size_t sidx2 = ((static_cast<size_t>(sp.layer) * dims.B + b) * dims.Hq + j0 + c) * 4;
            qsum = ws.qsum[sidx2];
            tsum = ws.qsum[sidx2 + 1];
        }
    }

    WarpState st;
    st.m = kNegInf;
    st.l = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; mt++)
#pragma unroll
        for (int q = 0; q < 4; q++) st.acc[mt][q] = 0.f;

#pragma unroll
    for (int s = 0; s < kStages - 1; s++) {
        if (s < n_st) load_stage(s);
        cp_async_commit();
    }
    for (int s = 0; s < n_st; s++) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        if (s + kStages - 1 < n_st) load_stage(s + kStages - 1);
        cp_async_commit();

        const uint8_t *buf = smem + (s % kStages) * stage_bytes;
        const int n = min(kStageTokens, ntok - s * kStageTokens);
        const int tile0 = warp * 16;
        if (tile0 < n) {
            const float *kss = reinterpret_cast<const float *>(buf + offKS);
            const float *vss = reinterpret_cast<const float *>(buf + offVS);
            const float *qns = reinterpret_cast<const float *>(buf + offQN);
            float sc[2];
            switch (kb * 2 + (qjl ? 1 : 0)) {
#define TQ_K(KB)                                                                                         \
    case 2 * KB: kphase<KB, false>(buf, buf + offQS, kss, qns, tile0, g, c, bq, bt, qsum, tsum, dims.qk_scale, sc); break; \
    case 2 * KB + 1: kphase<KB, true>(buf, buf + offQS, kss, qns, tile0, g, c, bq, bt, qsum, tsum, dims.qk_scale, sc); break;
                TQ_K(1) TQ_K(2) TQ_K(3) TQ_K(4) TQ_K(5) TQ_K(6) TQ_K(7) TQ_K(8)
#undef TQ_K
                default: sc[0] = sc[1] = 0.f; break;
            }
            const bool valid[2] = {tile0 + g < n, tile0 + g + 8 < n};
            const float vsc[2] = {vss[tile0 + g], vss[tile0 + g + 8]};
            uint32_t b0, b1;
            softmax_tile(st, sc, valid, vsc, g, c, c < gqa, b0, b1);
            switch (vb) {
#define TQ_V(VB) case VB: vphase<VB>(buf + offV, tile0, g, c, ctab, b0, b1, st.acc); break;
                TQ_V(1) TQ_V(2) TQ_V(3) TQ_V(4) TQ_V(5) TQ_V(6) TQ_V(7) TQ_V(8)
#undef TQ_V
                default: break;
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    float *part = ws.part + static_cast<size_t>(sp.part_begin + local) * (kMaxGqa * kPartStride);
    write_partial(st, reinterpret_cast<float *>(smem), part, gqa, 0);
}

// -------------------------------------------------------------- fp16 kernel
constexpr int kRow16 = 272;  // padded row of 128 fp16 (conflict-free ldmatrix)

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void *p) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(s));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void *p) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(s));
}

constexpr int kStages16 = 3;
constexpr int kStage16Bytes = 2 * kStageTokens * kRow16;

__global__ void __launch_bounds__(kThreads, 2)
    decode_fp16_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int seg_lo,
                       const int seg_hi) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int cta = blockIdx.x;
    const int si = find_segment(ws.seg, seg_lo, seg_hi, cta);
    const SegPlan &sp = ws.seg[si];
    const int local = cta - sp.cta_begin;
    const int chunk = local % sp.n_chunks;
    const int bh = local / sp.n_chunks;
    const int h = bh % dims.H, b = bh / dims.H;
    const int tok0 = chunk * sp.chunk;
    const int ntok = min(sp.chunk, sp.n_tokens - tok0);
    const size_t base = ((static_cast<size_t>(b) * dims.H + h) * sp.capacity + tok0) * kD * 2;
    const uint8_t *K = sp.kcodes + base, *V = sp.vcodes + base;
    const int n_st = (ntok + kStageTokens - 1) / kStageTokens;

    auto load_stage = [&](int s) {
        uint8_t *dst = smem + (s % kStages16) * kStage16Bytes;
        const int t0 = s * kStageTokens;
        const int n = min(kStageTokens, ntok - t0);
        for (int i = threadIdx.x; i < 2 * kStageTokens * 16; i += kThreads) {
            const int which = i / (kStageTokens * 16), r = (i >> 4) % kStageTokens, ch = i & 15;
            const uint8_t *src = (which ? V : K) + static_cast<size_t>(t0 + r) * (kD * 2) + ch * 16;
            const bool ok = r < n;
            cp_async16_zfill(dst + (which * kStageTokens + r) * kRow16 + ch * 16, ok ? src : K, ok ? 16 : 0);
        }
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int gqa = dims.gqa;
    const int j0 = h * gqa;
    uint32_t bq[8][2];
    {
        const int head = g >> 1, pt = g & 1;
        const size_t qidx = (static_cast<size_t>(sp.layer) * dims.B + b) * dims.Hq + j0 + head;
        const bool ok = head < gqa;
        const uint32_t *qw = ws.qorig + (qidx * 2 + pt) * (kD / 2);
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
            bq[kk][0] = ok ? qw[8 * kk + c] : 0u;
            bq[kk][1] = ok ? qw[8 * kk + c + 4] : 0u;
        }
    }
    WarpState st;
    st.m = kNegInf;
    st.l = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; mt++)
#pragma unroll
        for (int q = 0; q < 4; q++) st.acc[mt][q] = 0.f;

#pragma unroll
    for (int s = 0; s < kStages16 - 1; s++) {
        if (s < n_st) load_stage(s);
        cp_async_commit();
    }
    for (int s = 0; s < n_st; s++) {
        cp_async_wait<kStages16 - 2>();
        __syncthreads();
        if (s + kStages16 - 1 < n_st) load_stage(s + kStages16 - 1);
        cp_async_commit();
        const uint8_t *buf = smem + (s % kStages16) * kStage16Bytes;
        const int n = min(kStageTokens, ntok - s * kStageTokens);
        const int tile0 = warp * 16;
        if (tile0 < n) {
            const uint8_t *Ks = buf, *Vs = buf + kStageTokens * kRow16;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
                uint32_t a[4];
                const int row = tile0 + (lane & 7) + ((lane >> 3) & 1) * 8;
                ldmatrix_x4(a, Ks + row * kRow16 + kk * 32 + (lane >> 4) * 16);
                mma16816(acc, a[0], a[1], a[2], a[3], bq[kk][0], bq[kk][1]);
            }
            float sc[2] = {(acc[0] + acc[1]) * dims.qk_scale, (acc[2] + acc[3]) * dims.qk_scale};
            const bool valid[2] = {tile0 + g < n, tile0 + g + 8 < n};
            const float one[2] = {1.f, 1.f};
            uint32_t b0, b1;
            softmax_tile(st, sc, valid, one, g, c, c < gqa, b0, b1);
#pragma unroll
            for (int mt = 0; mt < 8; mt++) {
                uint32_t a[4];
                const int mat = lane >> 3;
                const int row = tile0 + (lane & 7) + (mat >> 1) * 8;
                ldmatrix_x4_trans(a, Vs + row * kRow16 + (16 * mt + (mat & 1) * 8) * 2);
                mma16816(st.acc[mt], a[0], a[1], a[2], a[3], b0, b1);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    float *part = ws.part + static_cast<size_t>(sp.part_begin + local) * (kMaxGqa * kPartStride);
    write_partial(st, reinterpret_cast<float *>(smem), part, gqa, 1);
}

// -------------------------------------------------------------- prep kernel
// One warp per (layer, batch, query head): q' = R q in binary32 (lane owns dims
// 4 lane .. 4 lane + 3), fp16 hi/lo splits of q and q', their sums, and for
// layers with QJL heads t = S q' (hi/lo and sum).
__device__ __forceinline__ void warp_wht(float (&x)[4], int lane) {
    float a = x[0], b = x[1], cc = x[2], d = x[3];
    // h = 1
    float t0 = a + b, t1 = a - b, t2 = cc + d, t3 = cc - d;
    // h = 2
    x[0] = t0 + t2; x[2] = t0 - t2; x[1] = t1 + t3; x[3] = t1 - t3;
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

__device__ __forceinline__ void store_hilo(uint32_t *dst, const float (&x)[4], int lane) {
    // dst: [2][64] words (hi then lo); lane writes words 2 lane, 2 lane + 1
    __half hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        hi[e] = __float2half_rn(x[e]);
        lo[e] = __float2half_rn(x[e] - __half2float(hi[e]));
    }
    dst[2 * lane] = pack_half2(hi[0], hi[1]);
    dst[2 * lane + 1] = pack_half2(hi[2], hi[3]);
    dst[64 + 2 * lane] = pack_half2(lo[0], lo[1]);
    dst[64 + 2 * lane + 1] = pack_half2(lo[2], lo[3]);
}

__device__ __forceinline__ float hilo_sum(const float (&x)[4]) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; e++) {
        const __half hi = __float2half_rn(x[e]);
        const __half lo = __float2half_rn(x[e] - __half2float(hi));
        s += __half2float(hi) + __half2float(lo);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

__global__ void __launch_bounds__(kThreads) decode_prep_kernel(const DecodeDims dims, const DecodeWorkspace ws,
                                                               const uint16_t *q, const float *S) {
    __shared__ float qsh[kThreads / 32][kD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wid = blockIdx.x * (kThreads / 32) + warp;
    const int total = dims.L * dims.B * dims.Hq;
    if (wid >= total) return;
    const int l = wid / (dims.B * dims.Hq);
    const LayerPlan &lp = ws.layer[l];
    float x[4];
    {
        const uint2 v = reinterpret_cast<const uint2 *>(q + static_cast<size_t>(wid) * kD)[lane];
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
        x[0] = f0.x; x[1] = f0.y; x[2] = f1.x; x[3] = f1.y;
    }
    store_hilo(ws.qorig + static_cast<size_t>(wid) * kD, x, lane);
    apply_signs(x, lp.sign_bits, lane);
    warp_wht(x, lane);
    apply_signs(x, lp.sign_bits, lane);
#pragma unroll
    for (int e = 0; e < 4; e++) x[e] *= dims.inv_sqrt_d;
    store_hilo(ws.qrot + static_cast<size_t>(wid) * kD, x, lane);
    const float qs = hilo_sum(x);
    float ts = 0.f;
    if (lp.has_qjl) {
#pragma unroll
        for (int e = 0; e < 4; e++) qsh[warp][4 * lane + e] = x[e];
        __syncwarp();
        float t[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float *row = S + static_cast<size_t>(4 * lane + e) * kD;
            float acc = 0.f;
            for (int i = 0; i < kD; i++) acc = fmaf(row[i], qsh[warp][i], acc);
            t[e] = acc;
        }
        store_hilo(ws.qjlt + static_cast<size_t>(wid) * kD, t, lane);
        ts = hilo_sum(t);
    }
    if (lane == 0) {
        ws.qsum[static_cast<size_t>(wid) * 4] = qs;
        ws.qsum[static_cast<size_t>(wid) * 4 + 1] = ts;
    }
}

// -------------------------------------------------------------- combine kernel
__global__ void __launch_bounds__(kThreads) decode_combine_kernel(const DecodeDims dims, const DecodeWorkspace ws,
                                                                  float *out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wid = blockIdx.x * (kThreads / 32) + warp;
    const int total = dims.L * dims.B * dims.Hq;
    if (wid >= total) return;
    const int j = wid % dims.Hq;
    const int b = (wid / dims.Hq) % dims.B;
    const int l = wid / (dims.Hq * dims.B);
    const int h = j / dims.gqa, jj = j % dims.gqa;
    const LayerPlan &lp = ws.layer[l];
    const size_t rec_stride = kMaxGqa * kPartStride;
    // pass 1: global max
    float M = kNegInf;
    const int n1 = lp.seg_end - lp.seg_begin, n2 = lp.f16_end - lp.f16_begin;
    for (int ii = 0; ii < n1 + n2; ii++) {
        const SegPlan &sp = ws.seg[ii < n1 ? lp.seg_begin + ii : lp.f16_begin + ii - n1];
        const size_t p0 = static_cast<size_t>(sp.part_begin) + static_cast<size_t>(b * dims.H + h) * sp.n_chunks;
        for (int ch = lane; ch < sp.n_chunks; ch += 32)
            M = fmaxf(M, ws.part[(p0 + ch) * rec_stride + jj * kPartStride]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    float ar[4] = {0.f, 0.f, 0.f, 0.f}, ao[4] = {0.f, 0.f, 0.f, 0.f};
    if (M != kNegInf) {
        for (int ii = 0; ii < n1 + n2; ii++) {
            const SegPlan &sp = ws.seg[ii < n1 ? lp.seg_begin + ii : lp.f16_begin + ii - n1];
            const size_t p0 = static_cast<size_t>(sp.part_begin) + static_cast<size_t>(b * dims.H + h) * sp.n_chunks;
            const bool rot = sp.kind == TQ_SEG_PACKED;
            for (int ch = 0; ch < sp.n_chunks; ch++) {
                const float *rec = ws.part + (p0 + ch) * rec_stride + jj * kPartStride;
                const float m = rec[0];
                if (m == kNegInf) continue;
                const float f = exp2f(m - M);
                L += f * rec[1];
                const float4 v = *reinterpret_cast<const float4 *>(rec + 4 + 4 * lane);
                float *a = rot ? ar : ao;
                a[0] += f * v.x; a[1] += f * v.y; a[2] += f * v.z; a[3] += f * v.w;
            }
        }
    }
    // inverse rotation of the packed-space sum (R is its own inverse)
    apply_signs(ar, lp.sign_bits, lane);
    warp_wht(ar, lane);
    apply_signs(ar, lp.sign_bits, lane);
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    float4 o;
    o.x = (ar[0] * dims.inv_sqrt_d + ao[0]) * inv;
    o.y = (ar[1] * dims.inv_sqrt_d + ao[1]) * inv;
    o.z = (ar[2] * dims.inv_sqrt_d + ao[2]) * inv;
    o.w = (ar[3] * dims.inv_sqrt_d + ao[3]) * inv;
    reinterpret_cast<float4 *>(out + static_cast<size_t>(wid) * kD)[lane] = o;
}

}  // namespace

size_t packed_stage_bytes(int kb_max, int vb_max, bool qjl) {
    return static_cast<size_t>(kStageTokens) * 16 * (kb_max + vb_max) + 512 +
           (qjl ? kStageTokens * 16 + 256 : 0);
}

cudaError_t launch_decode_kernels(const DecodeDims &dims, const DecodeWorkspace &ws, int n_packed_seg,
                                  int kb_max, int vb_max, bool any_qjl, const uint16_t *q,
                                  const float *S, const unsigned short *centroid_half, float *out,
                                  cudaStream_t s, cudaEvent_t ev_start, cudaEvent_t ev_stop) {
    static bool configured = false;
    const int stage_bytes = static_cast<int>(packed_stage_bytes(kb_max, vb_max, any_qjl));
    const size_t smem_packed = static_cast<size_t>(kStages) * stage_bytes + 512;  // + centroid table
    const size_t smem16 = static_cast<size_t>(kStages16) * kStage16Bytes;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_packed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(packed_stage_bytes(8, 8, true) * kStages + 512));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(decode_fp16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem16));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int n_warps = dims.L * dims.B * dims.Hq;
    const int prep_blocks = (n_warps + 3) / 4;
    decode_prep_kernel<<<prep_blocks, kThreads, 0, s>>>(dims, ws, q, S);
    if (dims.n_packed_ctas > 0) {
        Tables tab;
        for (int i = 0; i < kCbTotal; i++) tab.centroid[i] = centroid_half[i];
        if (ev_start) cudaEventRecord(ev_start, s);
        decode_packed_kernel<<<dims.n_packed_ctas, kThreads, smem_packed, s>>>(dims, ws, n_packed_seg,
                                                                            stage_bytes, tab);
        if (ev_stop) cudaEventRecord(ev_stop, s);
    }
    if (dims.n_fp16_ctas > 0) {
        decode_fp16_kernel<<<dims.n_fp16_ctas, kThreads, smem16, s>>>(dims, ws, n_packed_seg, dims.n_seg);
    }
    decode_combine_kernel<<<prep_blocks, kThreads, 0, s>>>(dims, ws, out);
    return cudaGetLastError();
}

}  // namespace tqk
