// tq_mass.cu -- passes after a decode call that rescore the packed tokens:
// the per-token attention mass and the QJL correction of sketched values.
//
// Attention mass: the signal of attention-weighted tier demotion ("TurboMOQ",
// "Attention-weighted tier demotion": tiers follow the attention weights of
// each decode step).
//
// mass[b][h][t] = (1/g) sum over the g query heads j of KV head h of
// 2^(s_j(t) - M_j) / L_j, with s_j(t) the base-2 score of token t and (M_j, L_j)
// the merged running max and sum the decode kernels left in the workspace.
//
// Packed tokens: the scores are recomputed on the tensor cores exactly as the
// split-K kernel computes them (key codes left at their bit offsets as fp16
// subnormals times the prep kernel's fp16 hi/lo rotated query, mma.m16n8k16,
// the affine key levels and the QJL term applied to the raw products), so
// only the key records, scales and sketches are read.  One CTA of 4 warps
// takes kMassTokens tokens of one (item, batch element); a warp takes its
// quarter in 16-token tiles, four per step; lane (g, c) scores tokens g and
// g + 8 for query head c and the four heads are summed across the lane quad.
// fp16 tokens (sinks, newest tier, chunk buffer) are scored one token per
// thread on the CUDA cores against the unrotated query.
#include "tq_decode_packed.cuh"
#include "tq_mass.h"

namespace tqk {
namespace dec {
namespace {

static_assert(kMassTokens % (16 * (kThreads / 32)) == 0, "whole 16-token tiles per warp");
constexpr int kWarpTokens = kMassTokens / (kThreads / 32);  // packed tokens per warp

// largest i in [0, n) with items[i].mass_cta_begin <= cta
__device__ __forceinline__ int find_mass_item(const WorkItem *items, int n, int cta) {
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (items[mid].mass_cta_begin <= cta) lo = mid;
        else hi = mid;
    }
    return lo;
}

struct MassShared {
    float qf[kMaxGqa][kD];       // unrotated queries (fp16 items)
    float mx[kMaxGqa], inv_l[kMaxGqa];
};

// A warp's packed tokens [t0, t0 + kWarpTokens) of batch element b in
// 16-token tiles, four per unrolled step (their loads are independent and
// issue together, which keeps enough bytes in flight per SM).
template <int KB, bool QJL>
__device__ __forceinline__ void mass_packed_warp(const DecodeDims &dims, const DecodeWorkspace &ws,
                                                 const WorkItem &it, int b, int t0, size_t qbase,
                                                 const MassShared &sh) {
    using KU = KUnpack<KB>;
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int gqa = dims.gqa, head = g >> 1, part = g & 1;
    // raw = (q / 2^e) . code * 2^(kA - 24); q . yhat = m (alpha q.code + beta sum q)
    constexpr float alphaA = static_cast<float>(1 << (24 - KU::kA)) * 2.0f / static_cast<float>(1 << KB);
    constexpr float beta = 1.0f / static_cast<float>(1 << KB) - 1.0f;
    // the prep kernel rotated every query of a call with packed segments
    uint32_t q[16], bq[16];
    const uint32_t *qw = ws.qrot + ((qbase + head) * 2 + part) * (kD / 2) + 16 * c;
#pragma unroll
    for (int i = 0; i < 16; i++) q[i] = head < gqa ? qw[i] : 0u;
    gather_b<KU>(q, bq);
    const float qsum = c < gqa ? ws.qsum[(qbase + c) * 4] : 0.f;
    const float aq = c < gqa ? alphaA * ws.qsum[(qbase + c) * 4 + 2] : 0.f;
    uint32_t bt[16];
    float tsum = 0.f;
    if constexpr (QJL) {
        const uint32_t *tw = ws.qjlt + ((qbase + head) * 2 + part) * (kD / 2) + 16 * c;
#pragma unroll
        for (int i = 0; i < 16; i++) q[i] = head < gqa ? tw[i] : 0u;
        gather_b<SignUnpack>(q, bt);
        tsum = c < gqa ? ws.qsum[(qbase + c) * 4 + 1] : 0.f;
    }
    const float m_c = c < gqa ? sh.mx[c] : 0.f, il_c = c < gqa ? sh.inv_l[c] : 0.f;
    const float inv_g = 1.0f / static_cast<float>(gqa);
    const int n = it.n_tokens;
    const uint8_t *kc = it.kc + b * it.kstride;
    const float *ks = it.ks + static_cast<size_t>(b) * it.sstride;
    float *mass = it.mass + static_cast<size_t>(b) * it.sstride;
    const int t_end = min(t0 + kWarpTokens, n);
    const int last = ((n + 15) & ~15) - 1;  // records exist up to the next multiple of 16
    // four tiles per step with every row clamped into the segment, so that all
    // their loads are unconditional and issue together (masked by t < n after)
    for (int t4 = t0; t4 < t_end; t4 += 64) {
#pragma unroll
    for (int tt = 0; tt < 4; tt++) {
        const int tile = t4 + 16 * tt;
        const int ta = tile + g, tb = ta + 8;
        const int ra = min(ta, last), rb = min(tb, last);
        float raw0, raw1;
        qk_raw<KU, KB>(kc + static_cast<size_t>(ra) * (16 * KB) + 4 * KB * c,
                       kc + static_cast<size_t>(rb) * (16 * KB) + 4 * KB * c, bq, raw0, raw1);
        float s0 = (ta < n ? ks[ra] : 0.f) * (aq * raw0 + beta * qsum);
        float s1 = (tb < n ? ks[rb] : 0.f) * (aq * raw1 + beta * qsum);
        if constexpr (QJL) {
            const size_t r0 = static_cast<size_t>(b) * it.qstride;
            float q0, q1;
            qk_raw<SignUnpack, 1>(it.qs + (r0 + ra) * (kJl / 8) + 4 * c, it.qs + (r0 + rb) * (kJl / 8) + 4 * c, bt,
                                  q0, q1);
            constexpr float gam = 1.2533141373155003f / kJl;  // sqrt(pi/2) / jl
            s0 += gam * (ta < n ? it.qn[r0 + ra] : 0.f) * (33554432.0f * q0 - tsum);
            s1 += gam * (tb < n ? it.qn[r0 + rb] : 0.f) * (33554432.0f * q1 - tsum);
        }
        float p0 = c < gqa ? ex2(fmaf(s0, dims.qk_scale, -m_c)) * il_c : 0.f;
        float p1 = c < gqa ? ex2(fmaf(s1, dims.qk_scale, -m_c)) * il_c : 0.f;
        p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
        p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
        p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
        p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
        if (c == 0) {
            if (ta < n) mass[ta] = p0 * inv_g;
            if (tb < n) mass[tb] = p1 * inv_g;
        }
    }
    }
}

__global__ void __launch_bounds__(kThreads, 4)
    attention_mass_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int n_items) {
    __shared__ __align__(16) MassShared sh;
    const int idx = find_mass_item(ws.items, n_items, blockIdx.x);
    const WorkItem &it = ws.items[idx];
    const int nch = (it.n_tokens + kMassTokens - 1) / kMassTokens;  // CTAs per batch element
    const int local = blockIdx.x - it.mass_cta_begin;
    const int b = local / nch;
    const int tok0 = (local - b * nch) * kMassTokens;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gqa = dims.gqa;
    const bool packed = it.kind == TQ_SEG_PACKED;
    const size_t qbase = (static_cast<size_t>(it.layer) * dims.B + b) * dims.Hq + static_cast<size_t>(it.head) * gqa;
    if (warp < kMaxGqa) {
        const bool on = warp < gqa;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (!packed) {  // fp16 tokens: the unrotated query
            if (on) load_q4(ws.q + (qbase + warp) * kD, lane, x);
#pragma unroll
            for (int e = 0; e < 4; e++) sh.qf[warp][4 * lane + e] = x[e];
        }
        if (lane == 0) {
            sh.mx[warp] = on ? ws.ml[(qbase + warp) * 2] : 0.f;
            const float l = on ? ws.ml[(qbase + warp) * 2 + 1] : 0.f;
            sh.inv_l[warp] = l > 0.f ? 1.0f / l : 0.f;
        }
    }
    __syncthreads();
    if (packed) {
        const int t0 = tok0 + kWarpTokens * warp;
        if (t0 >= it.n_tokens) return;
        const bool qj = it.qjl != 0;
#define TQ_MASS_CASE(K)                                                                \
    case K:                                                                            \
        if (qj) mass_packed_warp<K, true>(dims, ws, it, b, t0, qbase, sh);             \
        else mass_packed_warp<K, false>(dims, ws, it, b, t0, qbase, sh);               \
        break;
        switch (it.kb) {
            TQ_MASS_CASE(1)
            TQ_MASS_CASE(2)
            TQ_MASS_CASE(3)
            TQ_MASS_CASE(4)
            TQ_MASS_CASE(5)
            TQ_MASS_CASE(6)
            TQ_MASS_CASE(7)
            default:
                if (qj) mass_packed_warp<8, true>(dims, ws, it, b, t0, qbase, sh);
                else mass_packed_warp<8, false>(dims, ws, it, b, t0, qbase, sh);
                break;
        }
#undef TQ_MASS_CASE
        return;
    }
    // fp16 tokens: one thread per token against the unrotated query
    const int t_stop = min(tok0 + kMassTokens, it.n_tokens);
    for (int t = tok0 + threadIdx.x; t < t_stop; t += kThreads) {
    const uint4 *k = reinterpret_cast<const uint4 *>(it.kc + b * it.kstride + static_cast<size_t>(t) * (kD * 2));
    float dot[kMaxGqa] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int i8 = 0; i8 < kD / 8; i8++) {
        const uint4 v = k[i8];
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[e]));
#pragma unroll
            for (int j = 0; j < kMaxGqa; j++)
                dot[j] = fmaf(sh.qf[j][8 * i8 + 2 * e], f.x, fmaf(sh.qf[j][8 * i8 + 2 * e + 1], f.y, dot[j]));
        }
    }
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxGqa; j++)
        if (j < gqa) m += ex2(fmaf(dot[j], dims.qk_scale, -sh.mx[j])) * sh.inv_l[j];
    it.mass[static_cast<size_t>(b) * it.sstride + t] = m / static_cast<float>(gqa);
    }
}

// ------------------------------------------------------------ QJL on values
// z[l][b][j][i] = sum_t p_j(t) rho(t) s_i(t) over the packed tokens whose values
// carry a residual sketch (s = 2 bit - 1 the signs of S r, rho = ||r||), with
// p the final attention weights (rescored as above and normalised by the merged
// max and sum).  A warp's tiles: the scores give lane (g, c) the weights of
// tokens g, g + 8 for head c; shuffles turn w = p rho into the B fragment of an
// mma.m16n8k16 whose A fragment holds the sign bits as fp16 subnormals (the
// 1-bit value decoder), so the accumulator holds sum_t w bit 2^(s - 24) and
// sum_t w s = 2 sum_t w bit - sum_t w.  The CTA's warps add into shared memory,
// the CTA into z with one atomic per (head, coordinate).
__device__ __forceinline__ int find_vqjl_item(const WorkItem *items, int n, int cta) {
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (items[mid].vqjl_cta_begin <= cta) lo = mid;
        else hi = mid;
    }
    return lo;
}

template <int KB, bool QJL>
__device__ __forceinline__ void vqjl_warp(const DecodeDims &dims, const DecodeWorkspace &ws, const WorkItem &it,
                                          int b, int t0, size_t qbase, const MassShared &sh, float (*zsh)[kD]) {
    using KU = KUnpack<KB>;
    using VS = VDec<1, 7>;  // sign records decode as 1-bit codes
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int gqa = dims.gqa, head = g >> 1, part = g & 1;
    constexpr float alphaA = static_cast<float>(1 << (24 - KU::kA)) * 2.0f / static_cast<float>(1 << KB);
    constexpr float beta = 1.0f / static_cast<float>(1 << KB) - 1.0f;
    uint32_t q[16], bq[16];
    const uint32_t *qw = ws.qrot + ((qbase + head) * 2 + part) * (kD / 2) + 16 * c;
#pragma unroll
    for (int i = 0; i < 16; i++) q[i] = head < gqa ? qw[i] : 0u;
    gather_b<KU>(q, bq);
    const float qsum = c < gqa ? ws.qsum[(qbase + c) * 4] : 0.f;
    const float aq = c < gqa ? alphaA * ws.qsum[(qbase + c) * 4 + 2] : 0.f;
    uint32_t bt[16];
    float tsum = 0.f;
    if constexpr (QJL) {
        const uint32_t *tw = ws.qjlt + ((qbase + head) * 2 + part) * (kD / 2) + 16 * c;
#pragma unroll
        for (int i = 0; i < 16; i++) q[i] = head < gqa ? tw[i] : 0u;
        gather_b<SignUnpack>(q, bt);
        tsum = c < gqa ? ws.qsum[(qbase + c) * 4 + 1] : 0.f;
    }
    const float m_c = c < gqa ? sh.mx[c] : 0.f, il_c = c < gqa ? sh.inv_l[c] : 0.f;
    const int n = it.n_tokens;
    const uint8_t *kc = it.kc + b * it.kstride;
    const float *ks = it.ks + static_cast<size_t>(b) * it.sstride;
    const uint8_t *vs = it.vqs + static_cast<size_t>(b) * it.vqstride * (kJl / 8);
    const float *vn = it.vqn + static_cast<size_t>(b) * it.vqstride;
    VCtx vx;
    vx.off = 2 * c * 16 + 4 * (g >> 1);
    vx.sh = (g & 1) ? 0x7632 : 0x5410;
    float z[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; mt++) z[mt][0] = z[mt][1] = z[mt][2] = z[mt][3] = 0.f;
    float wsum = 0.f;  // this lane's B-fragment weights: head g
    const int t_end = min(t0 + kWarpTokens, n);
    const int last = ((n + 15) & ~15) - 1;  // records exist up to the next multiple of 16
    for (int t2 = t0; t2 < t_end; t2 += 32) {  // two tiles per step, rows clamped (as the mass pass)
#pragma unroll
    for (int tt = 0; tt < 2; tt++) {
        const int tile = t2 + 16 * tt;
        const int ta = tile + g, tb = ta + 8;
        const int ra = min(ta, last), rb = min(tb, last);
        float raw0, raw1;
        qk_raw<KU, KB>(kc + static_cast<size_t>(ra) * (16 * KB) + 4 * KB * c,
                       kc + static_cast<size_t>(rb) * (16 * KB) + 4 * KB * c, bq, raw0, raw1);
        float s0 = (ta < n ? ks[ra] : 0.f) * (aq * raw0 + beta * qsum);
        float s1 = (tb < n ? ks[rb] : 0.f) * (aq * raw1 + beta * qsum);
        if constexpr (QJL) {
            const size_t r0 = static_cast<size_t>(b) * it.qstride;
            float q0, q1;
            qk_raw<SignUnpack, 1>(it.qs + (r0 + ra) * (kJl / 8) + 4 * c, it.qs + (r0 + rb) * (kJl / 8) + 4 * c, bt,
                                  q0, q1);
            constexpr float gam = 1.2533141373155003f / kJl;
            s0 += gam * (ta < n ? it.qn[r0 + ra] : 0.f) * (33554432.0f * q0 - tsum);
            s1 += gam * (tb < n ? it.qn[r0 + rb] : 0.f) * (33554432.0f * q1 - tsum);
        }
        // weights of (token g, head c) and (token g + 8, head c), times the sketch norm
        const float w0 = c < gqa && ta < n ? ex2(fmaf(s0, dims.qk_scale, -m_c)) * il_c * vn[ra] : 0.f;
        const float w1 = c < gqa && tb < n ? ex2(fmaf(s1, dims.qk_scale, -m_c)) * il_c * vn[rb] : 0.f;
        // B fragment of head g: tokens 2c, 2c + 1 (rows 0-7) and 2c + 8, 2c + 9
        const int src = 8 * c + (g & 3);
        float v0 = __shfl_sync(0xffffffffu, w0, src), v1 = __shfl_sync(0xffffffffu, w0, src + 4);
        float v2 = __shfl_sync(0xffffffffu, w1, src), v3 = __shfl_sync(0xffffffffu, w1, src + 4);
        if (g >= gqa) v0 = v1 = v2 = v3 = 0.f;
        wsum += (v0 + v1) + (v2 + v3);
        const __half2 h01 = __floats2half2_rn(v0, v1), h23 = __floats2half2_rn(v2, v3);
        const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&h01), b1 = *reinterpret_cast<const uint32_t *>(&h23);
        uint32_t fa[8], fb[8], fc[8], fd[8];
        // a tile past the end reads the last whole tile (its weights are 0)
        const uint8_t *vrow = vs + static_cast<size_t>(min(tile, last - 15)) * (kJl / 8);
        VS::pair(vrow, kJl / 8, vx, fa, fb);                  // tokens 2c, 2c + 1
        VS::pair(vrow + 8 * (kJl / 8), kJl / 8, vx, fc, fd);  // tokens 2c + 8, 2c + 9
#pragma unroll
        for (int mt = 0; mt < 8; mt++) mma16816(z[mt], fa[mt], fb[mt], fc[mt], fd[mt], b0, b1);
    }
    }
    wsum += __shfl_xor_sync(0xffffffffu, wsum, 1);
    wsum += __shfl_xor_sync(0xffffffffu, wsum, 2);  // W of head g
    const float W0 = __shfl_sync(0xffffffffu, wsum, 8 * c), W1 = __shfl_sync(0xffffffffu, wsum, 8 * c + 4);
#pragma unroll
    for (int mt = 0; mt < 8; mt++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int r = e >> 1, hq = 2 * c + (e & 1);
            if (hq < gqa) {
                const float v = 2.0f * z[mt][e] * VS::unscale(mt, r) - ((e & 1) ? W1 : W0);
                atomicAdd(&zsh[hq][16 * g + VS::dim(mt, r)], v);
            }
        }
}

__global__ void __launch_bounds__(kThreads)
    value_qjl_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int n_items) {
    __shared__ __align__(16) MassShared sh;
    __shared__ float zsh[kMaxGqa][kD];
    const int idx = find_vqjl_item(ws.items, n_items, blockIdx.x);
    const WorkItem &it = ws.items[idx];
    const int nch = (it.n_tokens + kMassTokens - 1) / kMassTokens;
    const int local = blockIdx.x - it.vqjl_cta_begin;
    const int b = local / nch;
    const int tok0 = (local - b * nch) * kMassTokens;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gqa = dims.gqa;
    const size_t qbase = (static_cast<size_t>(it.layer) * dims.B + b) * dims.Hq + static_cast<size_t>(it.head) * gqa;
    for (int i = threadIdx.x; i < kMaxGqa * kD; i += kThreads) zsh[i / kD][i % kD] = 0.f;
    if (warp < kMaxGqa) {
        const bool on = warp < gqa;
        if (lane == 0) {
            sh.mx[warp] = on ? ws.ml[(qbase + warp) * 2] : 0.f;
            const float l = on ? ws.ml[(qbase + warp) * 2 + 1] : 0.f;
            sh.inv_l[warp] = l > 0.f ? 1.0f / l : 0.f;
        }
    }
    __syncthreads();
    const int t0 = tok0 + kWarpTokens * warp;
    if (t0 < it.n_tokens) {
        const bool qj = it.qjl != 0;
#define TQ_VQJL_CASE(K)                                                            \
    case K:                                                                        \
        if (qj) vqjl_warp<K, true>(dims, ws, it, b, t0, qbase, sh, zsh);           \
        else vqjl_warp<K, false>(dims, ws, it, b, t0, qbase, sh, zsh);             \
        break;
        switch (it.kb) {
            TQ_VQJL_CASE(1)
            TQ_VQJL_CASE(2)
            TQ_VQJL_CASE(3)
            TQ_VQJL_CASE(4)
            TQ_VQJL_CASE(5)
            TQ_VQJL_CASE(6)
            TQ_VQJL_CASE(7)
            default:
                if (qj) vqjl_warp<8, true>(dims, ws, it, b, t0, qbase, sh, zsh);
                else vqjl_warp<8, false>(dims, ws, it, b, t0, qbase, sh, zsh);
                break;
        }
#undef TQ_VQJL_CASE
    }
    __syncthreads();
    for (int i = threadIdx.x; i < gqa * kD; i += kThreads)
        atomicAdd(ws.z + (qbase + i / kD) * kD + (i % kD), zsh[i / kD][i % kD]);
}

// out[l][b][j] += R (sqrt(pi/2)/jl S^T z[l][b][j]) (R^T = R for the SRHT; Q^T
// for a dense rotation), one warp per query head of a layer with value sketches.
__global__ void __launch_bounds__(kThreads)
    value_qjl_apply_kernel(const DecodeDims dims, const DecodeWorkspace ws, const float *S) {
    const int wid = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (wid >= dims.L * dims.B * dims.Hq) return;
    const int l = wid / (dims.B * dims.Hq);
    const LayerPlan &lp = ws.layer[l];
    if (!lp.has_vqjl) return;
    float x[4];
    const float4 zv = reinterpret_cast<const float4 *>(ws.z + static_cast<size_t>(wid) * kD)[lane];
    x[0] = zv.x;
    x[1] = zv.y;
    x[2] = zv.z;
    x[3] = zv.w;
    warp_rotate_dense(x, S, true, lane);  // S^T z
    constexpr float coef = 1.2533141373155003f / kJl;
#pragma unroll
    for (int e = 0; e < 4; e++) x[e] *= coef;
    if (lp.dense) warp_rotate_dense(x, lp.dense, true, lane);
    else warp_rotate(x, lp.sign_bits, dims.inv_sqrt_d, lane);
    float4 *o = reinterpret_cast<float4 *>(ws.out + static_cast<size_t>(wid) * kD) + lane;
    float4 ov = *o;
    ov.x += x[0];
    ov.y += x[1];
    ov.z += x[2];
    ov.w += x[3];
    *o = ov;
}

}  // namespace
}  // namespace dec

cudaError_t launch_value_qjl(const DecodeDims &dims, const DecodeWorkspace &ws, int n_items, int n_ctas,
                             const float *S, cudaStream_t s) {
    dec::value_qjl_kernel<<<n_ctas, dec::kThreads, 0, s>>>(dims, ws, n_items);
    const int n_warps = dims.L * dims.B * dims.Hq;
    dec::value_qjl_apply_kernel<<<(n_warps + 3) / 4, dec::kThreads, 0, s>>>(dims, ws, S);
    return cudaGetLastError();
}

cudaError_t launch_attention_mass(const DecodeDims &dims, const DecodeWorkspace &ws, int n_items, int n_ctas,
                                  cudaStream_t s) {
    dec::attention_mass_kernel<<<n_ctas, dec::kThreads, 0, s>>>(dims, ws, n_items);
    return cudaGetLastError();
}

}  // namespace tqk
