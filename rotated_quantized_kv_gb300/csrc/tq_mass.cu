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
// quarter in 64-token steps staged through two shared buffers by cp.async
// (the next step in flight while one is scored), 16-token tiles within a
// step; lane (g, c) scores tokens g and g + 8 for query head c and the four
// heads are summed across the lane quad.
// fp16 tokens (sinks, newest tier, chunk buffer) are scored one token per
// thread on the CUDA cores against the unrotated query.
#include "tq_decode_packed.cuh"
#include "tq_mass.h"

namespace tqk {
namespace dec {
namespace {

static_assert(kMassTokens % (16 * (kThreads / 32)) == 0, "whole 16-token tiles per warp");
constexpr int kWarpTokens = kMassTokens / (kThreads / 32);  // packed tokens per warp


struct MassShared {
    float qf[kMaxGqa][kD];       // unrotated queries (fp16 items)
    float mx[kMaxGqa], inv_l[kMaxGqa];
};

// One 64-token step of a warp's records into a shared buffer, by cp.async
// (16-byte chunks spread over the lanes; rows past the segment's records read
// as zeros): key records (16 KB bytes a row), scales, and for QJL / value-
// sketch items their sign records (16 bytes) and norms.  Layout of a buffer:
// [keys][scales][key signs][key norms][value signs][value norms].
struct StepSrc {
    const uint8_t *kc;   // key records of row 0 (the batch element's)
    const float *ks;     // scales of row 0
    const uint8_t *qs;   // key sign records of row 0 (or null)
    const float *qn;
    const uint8_t *vs;   // value sign records of row 0 (or null)
    const float *vn;
};

template <int KB>
__device__ __forceinline__ void stage_step(uint8_t *buf, const StepSrc &src, int t, int last, int lane) {
    constexpr int RK = 16 * KB;
    const int rows_ok = min(kMassStep, last + 1 - t);  // whole rows of this step that exist
    // keys: kMassStep * RK / 16 chunks
    for (int i = lane; i < kMassStep * RK / 16; i += 32) {
        const int row = (i * 16) / RK;
        const bool ok = row < rows_ok;
        cp_async16_zfill(buf + i * 16, ok ? src.kc + static_cast<size_t>(t) * RK + i * 16 : src.kc, ok ? 16 : 0);
    }
    uint8_t *p = buf + kMassStep * RK;
    if (lane < kMassStep / 4) {  // scales: 4 per chunk
        const bool ok = 4 * lane < rows_ok;
        cp_async16_zfill(p + lane * 16, ok ? src.ks + t + 4 * lane : src.ks, ok ? 16 : 0);
    }
    p += kMassStep * 4;
    if (src.qs) {
        for (int i = lane; i < kMassStep; i += 32) {
            const bool ok = i < rows_ok;
            cp_async16_zfill(p + i * 16, ok ? src.qs + static_cast<size_t>(t + i) * 16 : src.qs, ok ? 16 : 0);
        }
        p += kMassStep * 16;
        if (lane < kMassStep / 4) {
            const bool ok = 4 * lane < rows_ok;
            cp_async16_zfill(p + lane * 16, ok ? src.qn + t + 4 * lane : src.qn, ok ? 16 : 0);
        }
        p += kMassStep * 4;
    }
    if (src.vs) {
        for (int i = lane; i < kMassStep; i += 32) {
            const bool ok = i < rows_ok;
            cp_async16_zfill(p + i * 16, ok ? src.vs + static_cast<size_t>(t + i) * 16 : src.vs, ok ? 16 : 0);
        }
        p += kMassStep * 16;
        if (lane < kMassStep / 4) {
            const bool ok = 4 * lane < rows_ok;
            cp_async16_zfill(p + lane * 16, ok ? src.vn + t + 4 * lane : src.vn, ok ? 16 : 0);
        }
    }
}

// A warp's packed tokens [t0, t0 + kWarpTokens) of batch element b in
// 64-token steps staged through two shared buffers (the next step's copies in
// flight while this one is scored), 16-token tiles within a step.
template <int KB, bool QJL>
__device__ __forceinline__ void mass_packed_warp(const DecodeDims &dims, const DecodeWorkspace &ws,
                                                 const WorkItem &it, int b, int t0, size_t qbase,
                                                 const MassShared &sh, uint8_t *buf0, int stage_bytes) {
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
    float *mass = it.mass + static_cast<size_t>(b) * it.sstride;
    const int t_end = min(t0 + kWarpTokens, n);
    const int last = ((n + 15) & ~15) - 1;  // records exist up to the next multiple of 16
    StepSrc src;
    src.kc = it.kc + b * it.kstride;
    src.ks = it.ks + static_cast<size_t>(b) * it.sstride;
    src.qs = QJL ? it.qs + static_cast<size_t>(b) * it.qstride * (kJl / 8) : nullptr;
    src.qn = QJL ? it.qn + static_cast<size_t>(b) * it.qstride : nullptr;
    src.vs = nullptr;
    src.vn = nullptr;
    constexpr int RK = 16 * KB;
    const int steps = (t_end - t0 + kMassStep - 1) / kMassStep;
    stage_step<KB>(buf0, src, t0, last, lane);
    cp_async_commit();
    for (int st = 0; st < steps; st++) {
        if (st + 1 < steps) stage_step<KB>(buf0 + ((st + 1) & 1) * stage_bytes, src, t0 + (st + 1) * kMassStep, last, lane);
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();
        const uint8_t *buf = buf0 + (st & 1) * stage_bytes;
        const float *kss = reinterpret_cast<const float *>(buf + kMassStep * RK);
        const uint8_t *qsb = buf + kMassStep * (RK + 4);
        const float *qnb = reinterpret_cast<const float *>(qsb + kMassStep * 16);
        const int ts = t0 + st * kMassStep;
#pragma unroll
        for (int tt = 0; tt < kMassStep / 16; tt++) {
            const int la = 16 * tt + g, lb = la + 8;  // rows within the step
            const int ta = ts + la, tb = ts + lb;
            float raw0, raw1;
            qk_raw<KU, KB>(buf + la * RK + 4 * KB * c, buf + lb * RK + 4 * KB * c, bq, raw0, raw1);
            float s0 = (ta < n ? kss[la] : 0.f) * (aq * raw0 + beta * qsum);
            float s1 = (tb < n ? kss[lb] : 0.f) * (aq * raw1 + beta * qsum);
            if constexpr (QJL) {
                float q0, q1;
                qk_raw<SignUnpack, 1>(qsb + la * 16 + 4 * c, qsb + lb * 16 + 4 * c, bt, q0, q1);
                constexpr float gam = 1.2533141373155003f / kJl;  // sqrt(pi/2) / jl
                s0 += gam * (ta < n ? qnb[la] : 0.f) * (33554432.0f * q0 - tsum);
                s1 += gam * (tb < n ? qnb[lb] : 0.f) * (33554432.0f * q1 - tsum);
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
        __syncwarp();  // the buffer is refilled two steps on
    }
    cp_async_wait<0>();
}

__global__ void __launch_bounds__(kThreads, 4)
    attention_mass_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int stage_bytes) {
    __shared__ __align__(16) MassShared sh;
    extern __shared__ __align__(16) uint8_t dyn[];
    const int idx = ws.mass_cta_item[blockIdx.x];
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
        uint8_t *buf0 = dyn + 2 * warp * stage_bytes;  // the warp's two step buffers
#define TQ_MASS_CASE(K)                                                                \
    case K:                                                                            \
        if (qj) mass_packed_warp<K, true>(dims, ws, it, b, t0, qbase, sh, buf0, stage_bytes);       \
        else mass_packed_warp<K, false>(dims, ws, it, b, t0, qbase, sh, buf0, stage_bytes);         \
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
                if (qj) mass_packed_warp<8, true>(dims, ws, it, b, t0, qbase, sh, buf0, stage_bytes);
                else mass_packed_warp<8, false>(dims, ws, it, b, t0, qbase, sh, buf0, stage_bytes);
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

template <int KB, bool QJL>
__device__ __forceinline__ void vqjl_warp(const DecodeDims &dims, const DecodeWorkspace &ws, const WorkItem &it,
                                          int b, int t0, size_t qbase, const MassShared &sh, float (*zsh)[kD],
                                          uint8_t *buf0, int stage_bytes) {
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
    StepSrc src;
    src.kc = it.kc + b * it.kstride;
    src.ks = it.ks + static_cast<size_t>(b) * it.sstride;
    src.qs = QJL ? it.qs + static_cast<size_t>(b) * it.qstride * (kJl / 8) : nullptr;
    src.qn = QJL ? it.qn + static_cast<size_t>(b) * it.qstride : nullptr;
    src.vs = it.vqs + static_cast<size_t>(b) * it.vqstride * (kJl / 8);
    src.vn = it.vqn + static_cast<size_t>(b) * it.vqstride;
    VCtx vx;
    vx.off = 2 * c * 16 + 4 * (g >> 1);
    vx.sh = (g & 1) ? 0x7632 : 0x5410;
    float z[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; mt++) z[mt][0] = z[mt][1] = z[mt][2] = z[mt][3] = 0.f;
    float wsum = 0.f;  // this lane's B-fragment weights: head g
    const int t_end = min(t0 + kWarpTokens, n);
    const int last = ((n + 15) & ~15) - 1;  // records exist up to the next multiple of 16
    constexpr int RK = 16 * KB;
    constexpr int kSignOff = kMassStep * (RK + 4 + (QJL ? 20 : 0));  // value signs within a buffer
    const int steps = (t_end - t0 + kMassStep - 1) / kMassStep;
    stage_step<KB>(buf0, src, t0, last, lane);
    cp_async_commit();
    for (int st = 0; st < steps; st++) {
        if (st + 1 < steps) stage_step<KB>(buf0 + ((st + 1) & 1) * stage_bytes, src, t0 + (st + 1) * kMassStep, last, lane);
        cp_async_commit();
        cp_async_wait<1>();
        __syncwarp();
        const uint8_t *buf = buf0 + (st & 1) * stage_bytes;
        const float *kss = reinterpret_cast<const float *>(buf + kMassStep * RK);
        const uint8_t *qsb = buf + kMassStep * (RK + 4);
        const float *qnb = reinterpret_cast<const float *>(qsb + kMassStep * 16);
        const uint8_t *vsb = buf + kSignOff;
        const float *vnb = reinterpret_cast<const float *>(vsb + kMassStep * 16);
        const int ts = t0 + st * kMassStep;
#pragma unroll 2
        for (int tt = 0; tt < kMassStep / 16; tt++) {
            const int la = 16 * tt + g, lb = la + 8;  // rows within the step
            const int ta = ts + la, tb = ts + lb;
            float raw0, raw1;
            qk_raw<KU, KB>(buf + la * RK + 4 * KB * c, buf + lb * RK + 4 * KB * c, bq, raw0, raw1);
            float s0 = (ta < n ? kss[la] : 0.f) * (aq * raw0 + beta * qsum);
            float s1 = (tb < n ? kss[lb] : 0.f) * (aq * raw1 + beta * qsum);
            if constexpr (QJL) {
                float q0, q1;
                qk_raw<SignUnpack, 1>(qsb + la * 16 + 4 * c, qsb + lb * 16 + 4 * c, bt, q0, q1);
                constexpr float gam = 1.2533141373155003f / kJl;
                s0 += gam * (ta < n ? qnb[la] : 0.f) * (33554432.0f * q0 - tsum);
                s1 += gam * (tb < n ? qnb[lb] : 0.f) * (33554432.0f * q1 - tsum);
            }
            // weights of (token g, head c) and (token g + 8, head c), times the sketch norm
            const float w0 = c < gqa && ta < n ? ex2(fmaf(s0, dims.qk_scale, -m_c)) * il_c * vnb[la] : 0.f;
            const float w1 = c < gqa && tb < n ? ex2(fmaf(s1, dims.qk_scale, -m_c)) * il_c * vnb[lb] : 0.f;
            // B fragment of head g: tokens 2c, 2c + 1 (rows 0-7) and 2c + 8, 2c + 9
            const int sl = 8 * c + (g & 3);
            float v0 = __shfl_sync(0xffffffffu, w0, sl), v1 = __shfl_sync(0xffffffffu, w0, sl + 4);
            float v2 = __shfl_sync(0xffffffffu, w1, sl), v3 = __shfl_sync(0xffffffffu, w1, sl + 4);
            if (g >= gqa) v0 = v1 = v2 = v3 = 0.f;
            wsum += (v0 + v1) + (v2 + v3);
            const __half2 h01 = __floats2half2_rn(v0, v1), h23 = __floats2half2_rn(v2, v3);
            const uint32_t b0 = *reinterpret_cast<const uint32_t *>(&h01), b1 = *reinterpret_cast<const uint32_t *>(&h23);
            uint32_t fa[8], fb[8], fc[8], fd[8];
            // rows past the records are zeros in the buffer (and their weights 0)
            const uint8_t *vrow = vsb + 16 * tt * (kJl / 8);
            VS::pair(vrow, kJl / 8, vx, fa, fb);                  // tokens 2c, 2c + 1
            VS::pair(vrow + 8 * (kJl / 8), kJl / 8, vx, fc, fd);  // tokens 2c + 8, 2c + 9
#pragma unroll
            for (int mt = 0; mt < 8; mt++) mma16816(z[mt], fa[mt], fb[mt], fc[mt], fd[mt], b0, b1);
        }
        __syncwarp();  // the buffer is refilled two steps on
    }
    cp_async_wait<0>();
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
    value_qjl_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int stage_bytes) {
    __shared__ __align__(16) MassShared sh;
    __shared__ float zsh[kMaxGqa][kD];
    extern __shared__ __align__(16) uint8_t dyn[];
    const int idx = ws.vqjl_cta_item[blockIdx.x];
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
        uint8_t *buf0 = dyn + 2 * warp * stage_bytes;  // the warp's two step buffers
#define TQ_VQJL_CASE(K)                                                            \
    case K:                                                                        \
        if (qj) vqjl_warp<K, true>(dims, ws, it, b, t0, qbase, sh, zsh, buf0, stage_bytes);     \
        else vqjl_warp<K, false>(dims, ws, it, b, t0, qbase, sh, zsh, buf0, stage_bytes);       \
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
                if (qj) vqjl_warp<8, true>(dims, ws, it, b, t0, qbase, sh, zsh, buf0, stage_bytes);
                else vqjl_warp<8, false>(dims, ws, it, b, t0, qbase, sh, zsh, buf0, stage_bytes);
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

cudaError_t launch_value_qjl(const DecodeDims &dims, const DecodeWorkspace &ws, int n_ctas,
                             int stage_bytes, const float *S, cudaStream_t s) {
    const int dyn = 2 * (dec::kThreads / 32) * stage_bytes;
    cudaError_t e = cudaFuncSetAttribute(dec::value_qjl_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e != cudaSuccess) return e;
    dec::value_qjl_kernel<<<n_ctas, dec::kThreads, dyn, s>>>(dims, ws, stage_bytes);
    const int n_warps = dims.L * dims.B * dims.Hq;
    dec::value_qjl_apply_kernel<<<(n_warps + 3) / 4, dec::kThreads, 0, s>>>(dims, ws, S);
    return cudaGetLastError();
}

cudaError_t launch_attention_mass(const DecodeDims &dims, const DecodeWorkspace &ws, int n_ctas,
                                  int stage_bytes, cudaStream_t s) {
    const int dyn = 2 * (dec::kThreads / 32) * stage_bytes;
    cudaError_t e =
        cudaFuncSetAttribute(dec::attention_mass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e != cudaSuccess) return e;
    dec::attention_mass_kernel<<<n_ctas, dec::kThreads, dyn, s>>>(dims, ws, stage_bytes);
    return cudaGetLastError();
}

}  // namespace tqk
