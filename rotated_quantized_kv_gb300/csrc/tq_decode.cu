// tq_decode.cu -- decode attention directly on the compressed KV cache: the
// split-K kernel over fp16 segments, the QJL query-preparation kernel and the
// launch sequence.  The split-K kernels over packed segments live in
// tq_decode_packed.cuh (one instantiation per class, tq_decode_kb*.cu).
//
// Method: "turboquant-mlx" skill note, "Optimisations Metal" (fused attention on
// the compressed cache, the inverse transform pulled out of the V sum);
// "turboquant-mlx" (TurboQuant-MLX v2.0 README), "Implementation Status"
// (compressed-domain attention) and "RaBitQ vs QJL correction"; "TurboMOQ",
// "QJL residual correction (sub-2-bit)".
//
// R is orthogonal and symmetric, so q . (R yhat) = (R q) . yhat: each CTA over
// packed tokens rotates its queries once, scores and sums values in the
// rotated space, and the CTA that finishes a (layer, batch, KV head) last
// merges all partials, rotates the packed-space sum back once and adds the
// fp16-segment sum (original space).  No CTA waits on another.
#include "tq_decode_common.cuh"

namespace tqk {
namespace dec {
namespace {

// -------------------------------------------------------------- fp16 kernel
constexpr int kRow16 = 272;  // padded row of 128 fp16 (conflict-free ldmatrix)
constexpr int kStage16Bytes = 2 * kStageTokens * kRow16;  // one 64-token chunk of K and V

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void *p) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void *p) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s));
}

// Tokens kept in fp16 (sinks, newest tier, chunk buffer), attended in the
// original space with the unrotated query: ldmatrix gives K rows as the A
// fragment of Q.K and V rows transposed as the A fragment of P.V.  One CTA per
// (item, batch element, 64-token chunk): a single staged chunk, so that many
// small CTAs (six per SM) cover the memory latency together.
__global__ void __launch_bounds__(kThreads, 6)
    decode_fp16_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int item_lo, const int item_hi) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int idx = find_item(ws.items, item_lo, item_hi, blockIdx.x);
    const WorkItem &it = ws.items[idx];
    const int local = blockIdx.x - it.cta_begin;
    const int b = local / it.n_chunks, chunk = local - b * it.n_chunks;
    const int tok0 = chunk * it.chunk;
    const int ntok = min(it.chunk, it.n_tokens - tok0);  // <= kStageTokens
    const uint8_t *K = it.kc + b * it.kstride + static_cast<size_t>(tok0) * (kD * 2);
    const uint8_t *V = it.vc + b * it.vstride + static_cast<size_t>(tok0) * (kD * 2);
    for (int i = threadIdx.x; i < 2 * kStageTokens * 16; i += kThreads) {
        const int which = i / (kStageTokens * 16), r = (i >> 4) % kStageTokens, ch = i & 15;
        const uint8_t *src = (which ? V : K) + static_cast<size_t>(r) * (kD * 2) + ch * 16;
        const bool ok = r < ntok;
        cp_async16_zfill(smem + (which * kStageTokens + r) * kRow16 + ch * 16, ok ? src : K, ok ? 16 : 0);
    }
    cp_async_commit();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int gqa = dims.gqa;
    const int j0 = it.head * gqa;
    pdl_launch_dependents();
    // B fragments of the (fp16, hence exact) queries: column g holds head g/2;
    // the lo columns (g odd) are zero.
    uint32_t bq[8][2];
    {
        const int head = g >> 1;
        const size_t qidx = (static_cast<size_t>(it.layer) * dims.B + b) * dims.Hq + j0 + head;
        const bool ok = head < gqa && (g & 1) == 0;
        const uint32_t *qw = reinterpret_cast<const uint32_t *>(ws.q + qidx * kD);
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
            bq[kk][0] = ok ? qw[8 * kk + c] : 0u;
            bq[kk][1] = ok ? qw[8 * kk + c + 4] : 0u;
        }
    }
    WarpState st;
    init_state(st);
    cp_async_wait<0>();
    __syncthreads();
    const int tile0 = warp * 16;
    if (tile0 < ntok) {
        const uint8_t *Ks = smem, *Vs = smem + kStageTokens * kRow16;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
            uint32_t a[4];
            const int row = tile0 + (lane & 7) + ((lane >> 3) & 1) * 8;
            ldmatrix_x4(a, Ks + row * kRow16 + kk * 32 + (lane >> 4) * 16);
            mma16816(acc, a[0], a[1], a[2], a[3], bq[kk][0], bq[kk][1]);
        }
        uint32_t b0, b1;
        softmax_tile(st, (acc[0] + acc[1]) * dims.qk_scale, (acc[2] + acc[3]) * dims.qk_scale, tile0 + g < ntok,
                     tile0 + g + 8 < ntok, 1.f, 1.f, g, c, c < gqa, b0, b1);
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            uint32_t a[4];
            const int mat = lane >> 3;
            const int row = tile0 + (lane & 7) + (mat >> 1) * 8;
            ldmatrix_x4_trans(a, Vs + row * kRow16 + (16 * mt + (mat & 1) * 8) * 2);
            mma16816(st.acc[mt], a[0], a[1], a[2], a[3], b0, b1);
        }
    }
    __syncthreads();  // the staged chunk is dead: its space becomes the merge scratch
    const int slot = ws.grp_part[static_cast<size_t>(idx) * dims.B + b] + chunk;
    float *part = ws.part + static_cast<size_t>(slot) * (kMaxGqa * kPartStride);
    write_partial(st, reinterpret_cast<float *>(smem), part, gqa,
                  [g](int mt, int r) { return 16 * mt + g + 8 * r; });
    pdl_wait();  // this grid's completion implies the completion of the earlier ones
    finish_and_combine(dims, ws, it.layer, b, it.head, reinterpret_cast<int *>(smem + kStage16Bytes));
}

// -------------------------------------------------------------- prep kernel
// Calls with QJL heads or dense-rotation layers: one warp per (layer, batch,
// query head) computes q' = R q (normalised by a power of two; R the layer's
// SRHT or dense Q) and, for QJL layers, t = S q' (fp16 hi/lo words), with
// sum q', sum t and the power of two, for the split-K kernels, which read them
// after griddepcontrol.wait.
__global__ void __launch_bounds__(kThreads)
    decode_prep_kernel(const DecodeDims dims, const DecodeWorkspace ws, const float *S) {
    __shared__ float qsh[kThreads / 32][kD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wid = blockIdx.x * (kThreads / 32) + warp;
    pdl_launch_dependents();
    if (wid >= dims.L * dims.B * dims.Hq) return;
    const int l = wid / (dims.B * dims.Hq);
    const LayerPlan &lp = ws.layer[l];
    float x[4];
    load_q4(ws.q + static_cast<size_t>(wid) * kD, lane, x);
    if (lp.dense) warp_rotate_dense(x, lp.dense, false, lane);
    else warp_rotate(x, lp.sign_bits, dims.inv_sqrt_d, lane);
    // q' / 2^e with its largest coordinate in [0.5, 1) (the packed kernels
    // scale the B fragment up by powers of two); t = S q' from q' itself
    const float f = warp_pow2_norm(x);
    float xn[4];
#pragma unroll
    for (int e = 0; e < 4; e++) xn[e] = x[e] * f;
    const float qs = store_hilo(ws.qrot + static_cast<size_t>(wid) * kD, xn, lane) / f;
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
        if (lp.qjl_mode == TQ_QJL_SIGN_PAIR) {
            // sign-pair estimator: t_j = sqrt(pi/2) ||q'|| sign((S q')_j), so that
            // the kernels' sqrt(pi/2)/jl * rho * <t, s> is (pi/2)/jl ||q'|| rho <sign(S q'), s>
            float n2 = 0.f;
#pragma unroll
            for (int e = 0; e < 4; e++) n2 = fmaf(x[e], x[e], n2);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
            const float c = 1.2533141373155003f * sqrtf(n2);
#pragma unroll
            for (int e = 0; e < 4; e++) t[e] = t[e] >= 0.f ? c : -c;
        }
        ts = store_hilo(ws.qjlt + static_cast<size_t>(wid) * kD, t, lane);
    }
    if (lane == 0) {
        ws.qsum[static_cast<size_t>(wid) * 4] = qs;
        ws.qsum[static_cast<size_t>(wid) * 4 + 1] = ts;
        ws.qsum[static_cast<size_t>(wid) * 4 + 2] = 1.0f / f;
    }
}

// ------------------------------------------------------ attention mass kernel
// One thread per token of an item with a mass buffer: the scores of the
// group's query heads are recomputed from the token's key record in binary32
// (packed: the rotated query against the affine key levels, plus the QJL term
// from the prep kernel's t = S q' words; fp16: the query against the key) and
// normalised by the merged max and sum the decode kernels left in ws.ml.
static_assert(kMassTokens == kThreads, "one thread per token");

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

// sum_i q[j][i] * code_i for the 4 query slots, codes of a KB-bit record
template <int KB>
__device__ __forceinline__ void mass_code_dots(const uint8_t *rec, const float (*qf)[kD], float (&dot)[kMaxGqa]) {
    uint32_t w[4 * KB + 1];
#pragma unroll
    for (int i = 0; i < KB; i++) {
        const uint4 v = reinterpret_cast<const uint4 *>(rec)[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    w[4 * KB] = 0u;
#pragma unroll
    for (int i4 = 0; i4 < kD / 4; i4++) {
        float c[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int bit = KB * (4 * i4 + e);
            const uint64_t win = (static_cast<uint64_t>(w[(bit >> 5) + 1]) << 32) | w[bit >> 5];
            c[e] = static_cast<float>(static_cast<uint32_t>(win >> (bit & 31)) & ((1u << KB) - 1u));
        }
#pragma unroll
        for (int j = 0; j < kMaxGqa; j++) {
            const float4 q = reinterpret_cast<const float4 *>(qf[j])[i4];
            dot[j] = fmaf(q.x, c[0], fmaf(q.y, c[1], fmaf(q.z, c[2], fmaf(q.w, c[3], dot[j]))));
        }
    }
}

template <int KB>
__device__ __forceinline__ void mass_packed_scores(const WorkItem &it, int b, int t, const float (*qf)[kD],
                                                   const float *qs, float (&sc)[kMaxGqa]) {
    float dot[kMaxGqa] = {0.f, 0.f, 0.f, 0.f};
    mass_code_dots<KB>(it.kc + b * it.kstride + static_cast<size_t>(t) * (16 * KB), qf, dot);
    // level(c) = c * 2^(1-KB) + 2^(-KB) - 1
    const float m = it.ks[static_cast<size_t>(b) * it.sstride + t];
    constexpr float alpha = 2.0f / static_cast<float>(1 << KB);
    constexpr float beta = 1.0f / static_cast<float>(1 << KB) - 1.0f;
#pragma unroll
    for (int j = 0; j < kMaxGqa; j++) sc[j] = m * fmaf(alpha, dot[j], beta * qs[j]);
}

__global__ void __launch_bounds__(kThreads)
    attention_mass_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int n_items) {
    __shared__ __align__(16) float qf[kMaxGqa][kD];
    __shared__ __align__(16) float tf[kMaxGqa][kD];
    __shared__ float qs[kMaxGqa], ts[kMaxGqa], mx[kMaxGqa], inv_l[kMaxGqa];
    const int idx = find_mass_item(ws.items, n_items, blockIdx.x);
    const WorkItem &it = ws.items[idx];
    const int nch = (it.n_tokens + kMassTokens - 1) / kMassTokens;
    const int local = blockIdx.x - it.mass_cta_begin;
    const int b = local / nch;
    const int t = (local - b * nch) * kMassTokens + threadIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gqa = dims.gqa;
    const bool packed = it.kind == TQ_SEG_PACKED;
    const size_t qrow = (static_cast<size_t>(it.layer) * dims.B + b) * dims.Hq + it.head * gqa + warp;
    if (warp < kMaxGqa) {
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        float tv[4] = {0.f, 0.f, 0.f, 0.f};
        if (warp < gqa) {
            load_q4(ws.q + qrow * kD, lane, x);
            if (packed) {
                const LayerPlan &lp = ws.layer[it.layer];
                if (lp.dense) {  // the prep kernel's q' / 2^e (hi + lo) times 2^e
                    const __half *qh = reinterpret_cast<const __half *>(ws.qrot + qrow * kD);
                    const float f = ws.qsum[qrow * 4 + 2];
#pragma unroll
                    for (int e = 0; e < 4; e++)
                        x[e] = (__half2float(qh[4 * lane + e]) + __half2float(qh[kD + 4 * lane + e])) * f;
                } else {
                    warp_rotate(x, lp.sign_bits, dims.inv_sqrt_d, lane);
                }
            }
            if (packed && it.qjl) {
                const __half *th = reinterpret_cast<const __half *>(ws.qjlt + qrow * kD);
#pragma unroll
                for (int e = 0; e < 4; e++)
                    tv[e] = __half2float(th[4 * lane + e]) + __half2float(th[kD + 4 * lane + e]);
            }
        }
        float sum = x[0] + x[1] + x[2] + x[3];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
#pragma unroll
        for (int e = 0; e < 4; e++) {
            qf[warp][4 * lane + e] = x[e];
            tf[warp][4 * lane + e] = tv[e];
        }
        if (lane == 0) {
            qs[warp] = sum;
            const bool on = warp < gqa;
            ts[warp] = on && packed && it.qjl ? ws.qsum[qrow * 4 + 1] : 0.f;
            mx[warp] = on ? ws.ml[qrow * 2] : 0.f;
            const float l = on ? ws.ml[qrow * 2 + 1] : 0.f;
            inv_l[warp] = l > 0.f ? 1.0f / l : 0.f;
        }
    }
    __syncthreads();
    if (t >= it.n_tokens) return;
    float sc[kMaxGqa] = {0.f, 0.f, 0.f, 0.f};
    if (packed) {
        switch (it.kb) {
            case 1: mass_packed_scores<1>(it, b, t, qf, qs, sc); break;
            case 2: mass_packed_scores<2>(it, b, t, qf, qs, sc); break;
            case 3: mass_packed_scores<3>(it, b, t, qf, qs, sc); break;
            case 4: mass_packed_scores<4>(it, b, t, qf, qs, sc); break;
            case 5: mass_packed_scores<5>(it, b, t, qf, qs, sc); break;
            case 6: mass_packed_scores<6>(it, b, t, qf, qs, sc); break;
            case 7: mass_packed_scores<7>(it, b, t, qf, qs, sc); break;
            default: mass_packed_scores<8>(it, b, t, qf, qs, sc); break;
        }
        if (it.qjl) {  // + sqrt(pi/2)/jl * rho * (2 sum_{bit set} t_i - sum t)
            const size_t rq = static_cast<size_t>(b) * it.qstride + t;
            float dot[kMaxGqa] = {0.f, 0.f, 0.f, 0.f};
            mass_code_dots<1>(it.qs + rq * (kJl / 8), tf, dot);
            const float g = 1.2533141373155003f / kJl * it.qn[rq];
#pragma unroll
            for (int j = 0; j < kMaxGqa; j++) sc[j] = fmaf(g, 2.0f * dot[j] - ts[j], sc[j]);
        }
    } else {
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
                    dot[j] = fmaf(qf[j][8 * i8 + 2 * e], f.x, fmaf(qf[j][8 * i8 + 2 * e + 1], f.y, dot[j]));
            }
        }
#pragma unroll
        for (int j = 0; j < kMaxGqa; j++) sc[j] = dot[j];
    }
    float mass = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxGqa; j++)
        if (j < gqa) mass += ex2(fmaf(sc[j], dims.qk_scale, -mx[j])) * inv_l[j];
    it.mass[static_cast<size_t>(b) * it.sstride + t] = mass / static_cast<float>(gqa);
}

PackedLauncher packed_launcher(int kb, int vb, bool qjl) {
    switch (kb) {
        case 1: return packed_launcher_kb1(vb, qjl);
        case 2: return packed_launcher_kb2(vb, qjl);
        case 3: return packed_launcher_kb3(vb, qjl);
        case 4: return packed_launcher_kb4(vb, qjl);
        case 5: return packed_launcher_kb5(vb, qjl);
        case 6: return packed_launcher_kb6(vb, qjl);
        case 7: return packed_launcher_kb7(vb, qjl);
        case 8: return packed_launcher_kb8(vb, qjl);
        default: return nullptr;
    }
}

}  // namespace
}  // namespace dec

cudaError_t launch_decode_kernels(const DecodeDims &dims, const DecodeWorkspace &ws, const ClassLaunch *classes,
                                  int n_classes, const float *S, const unsigned short *const *value_half,
                                  const float *value_c1,
                                  cudaStream_t s, cudaEvent_t ev_start, cudaEvent_t ev_stop) {
    static bool configured = false;
    const size_t smem16 = static_cast<size_t>(dec::kStage16Bytes) + 16;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(dec::decode_fp16_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem16));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // Order: [prep] -> packed classes -> fp16 segments.  Every kernel after the
    // first may start early (programmatic dependent launch); each grid waits
    // for its predecessor before its final merges, the QJL classes also wait
    // for prep before reading its outputs.  The persistent packed grids come
    // first so that all their CTAs start together (their stage ranges are fixed:
    // a CTA that starts late finishes late); the many small fp16 CTAs come last
    // and fill the SMs the packed grid frees at its end.
    bool first = true;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (dims.any_prep) {
        const int n_warps = dims.L * dims.B * dims.Hq;
        dec::decode_prep_kernel<<<(n_warps + 3) / 4, dec::kThreads, 0, s>>>(dims, ws, S);
        first = false;
    }
    bool any_packed = false;
    for (int i = 0; i < n_classes; i++) any_packed |= classes[i].kb != 16 && classes[i].n_ctas > 0;
    if (ev_start && any_packed) {
        cudaEventRecord(ev_start, s);
        first = true;  // an event in between serialises anyway
    }
    for (int i = 0; i < n_classes; i++) {
        const ClassLaunch &c = classes[i];
        if (c.n_ctas <= 0 || c.kb == 16) continue;
        const PackedLauncher fn = dec::packed_launcher(c.kb, c.vb, c.qjl != 0);
        if (!fn) return cudaErrorInvalidValue;
        const cudaError_t e =
            fn(dims, ws, c.item_lo, c.item_hi, c.n_ctas, c.n_stages, value_half[i], value_c1[i], s, !first);
        if (e != cudaSuccess) return e;
        first = false;
    }
    if (ev_stop && any_packed) {
        cudaEventRecord(ev_stop, s);
        first = true;
    }
    for (int i = 0; i < n_classes; i++) {
        const ClassLaunch &c = classes[i];
        if (c.n_ctas <= 0 || c.kb != 16) continue;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c.n_ctas);
        cfg.blockDim = dim3(dec::kThreads);
        cfg.dynamicSmemBytes = smem16;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = first ? 0 : 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, dec::decode_fp16_kernel, dims, ws, c.item_lo, c.item_hi);
        if (e != cudaSuccess) return e;
        first = false;
    }
    return cudaGetLastError();
}

cudaError_t launch_attention_mass(const DecodeDims &dims, const DecodeWorkspace &ws, int n_items, int n_ctas,
                                  cudaStream_t s) {
    dec::attention_mass_kernel<<<n_ctas, dec::kThreads, 0, s>>>(dims, ws, n_items);
    return cudaGetLastError();
}

}  // namespace tqk
