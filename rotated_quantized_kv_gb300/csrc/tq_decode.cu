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
// head_dim 128 nh: padded rows of 128 nh fp16, a 64-token chunk of K and V, then
// the cross-warp merge scratch (write_partial) and the flag
// (head_dim 64: np = 2, rows of 64 fp16)
__host__ __device__ constexpr int row16(int nh, int np = 1) { return 256 * nh / np + 16; }
__host__ __device__ constexpr int stage16_bytes(int nh, int np = 1) { return 2 * kStageTokens * row16(nh, np); }
constexpr int kMergeScratchBytes = (32 + kDecodeWarps * kMaxGqa * kD) * 4;
__host__ __device__ constexpr int fp16_smem_bytes(int nh, int np = 1) {
    return nh == 1 && np == 1 ? kStage16Bytes + 16 : stage16_bytes(nh, np) + kMergeScratchBytes + 16;
}

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
//
// NH > 1 (head_dim 128 NH): the scores run over all NH 128-dim blocks, then
// each block's P.V is merged across the warps and written as record
// chunk NH + j of the group (block j), all with the chunk's m and l.
// NP = 2 (head_dim 64): rows of 64 dims; the record's virtual dims 64..127
// stay zero (the merge adds the two halves).
template <int NH, int NP = 1>
__global__ void __launch_bounds__(kThreads, NH == 1 && NP == 1 ? 6 : 1)
    decode_fp16_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int *__restrict__ cta_item) {
    constexpr int kDh = NH * kD / NP, kRow = row16(NH, NP);
    extern __shared__ __align__(16) uint8_t smem[];
    const int idx = cta_item[blockIdx.x];
    const WorkItem &it = ws.items[idx];
    const int local = blockIdx.x - it.cta_begin;
    const int b = local / it.n_chunks, chunk = local - b * it.n_chunks;
    const int tok0 = chunk * it.chunk;
    const int ntok = min(it.chunk, it.n_tokens - tok0);  // <= kStageTokens
    const uint8_t *K = it.kc + b * it.kstride + static_cast<size_t>(tok0) * (kDh * 2);
    const uint8_t *V = it.vc + b * it.vstride + static_cast<size_t>(tok0) * (kDh * 2);
    constexpr int kCh = 16 * NH / NP;  // 16-byte pieces of a row
    for (int i = threadIdx.x; i < 2 * kStageTokens * kCh; i += kThreads) {
        const int which = i / (kStageTokens * kCh), r = (i / kCh) % kStageTokens, ch = i % kCh;
        const uint8_t *src = (which ? V : K) + static_cast<size_t>(r) * (kDh * 2) + ch * 16;
        const bool ok = r < ntok;
        cp_async16_zfill(smem + (which * kStageTokens + r) * kRow + ch * 16, ok ? src : K, ok ? 16 : 0);
    }
    cp_async_commit();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int gqa = dims.gqa;
    const int j0 = it.head * gqa;
    pdl_launch_dependents();
    // B fragments of the (fp16, hence exact) queries: column g holds head g/2;
    // the lo columns (g odd) are zero.
    uint32_t bq[8 * NH / NP][2];
    {
        const int head = g >> 1;
        const size_t qidx = (static_cast<size_t>(it.layer) * dims.B + b) * dims.Hq + j0 + head;
        const bool ok = head < gqa && (g & 1) == 0;
        const uint32_t *qw = reinterpret_cast<const uint32_t *>(ws.q + qidx * kDh);
#pragma unroll
        for (int kk = 0; kk < 8 * NH / NP; kk++) {
            bq[kk][0] = ok ? qw[8 * kk + c] : 0u;
            bq[kk][1] = ok ? qw[8 * kk + c + 4] : 0u;
        }
    }
    WarpState st;
    init_state(st);
    cp_async_wait<0>();
    __syncthreads();
    const int tile0 = warp * 16;
    if constexpr (NH == 1 && NP == 1) {
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
    } else {
    const uint8_t *Ks = smem, *Vs = smem + kStageTokens * kRow;
    uint32_t b0 = 0u, b1 = 0u;
    if (tile0 < ntok) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8 * NH / NP; kk++) {
            uint32_t a[4];
            const int row = tile0 + (lane & 7) + ((lane >> 3) & 1) * 8;
            ldmatrix_x4(a, Ks + row * kRow + kk * 32 + (lane >> 4) * 16);
            mma16816(acc, a[0], a[1], a[2], a[3], bq[kk][0], bq[kk][1]);
        }
        softmax_tile(st, (acc[0] + acc[1]) * dims.qk_scale, (acc[2] + acc[3]) * dims.qk_scale, tile0 + g < ntok,
                     tile0 + g + 8 < ntok, 1.f, 1.f, g, c, c < gqa, b0, b1);
    }
    float *scratch = reinterpret_cast<float *>(smem + stage16_bytes(NH, NP));
    const int slot0 = ws.grp_part[static_cast<size_t>(idx) * dims.B + b] + chunk * NH;
#pragma unroll 1
    for (int j = 0; j < NH; j++) {
#pragma unroll
        for (int mt = 0; mt < 8; mt++)
#pragma unroll
            for (int q = 0; q < 4; q++) st.acc[mt][q] = 0.f;
        if (tile0 < ntok) {
#pragma unroll
            for (int mt = 0; mt < 8 / NP; mt++) {
                uint32_t a[4];
                const int mat = lane >> 3;
                const int row = tile0 + (lane & 7) + (mat >> 1) * 8;
                ldmatrix_x4_trans(a, Vs + row * kRow + (kD * j + 16 * mt + (mat & 1) * 8) * 2);
                mma16816(st.acc[mt], a[0], a[1], a[2], a[3], b0, b1);
            }
        }
        if (j > 0) __syncthreads();  // the previous block's merge is done with the scratch
        float *part = ws.part + static_cast<size_t>(slot0 + j) * (kMaxGqa * kPartStride);
        write_partial(st, scratch, part, gqa, [g](int mt, int r) { return 16 * mt + g + 8 * r; });
    }
    pdl_wait();
    finish_and_combine<NH, NP>(dims, ws, it.layer, b, it.head,
                               reinterpret_cast<int *>(smem + stage16_bytes(NH, NP) + kMergeScratchBytes));
    }
}

// -------------------------------------------------------------- prep kernel
// Calls with QJL heads or dense-rotation layers: one warp per (layer, batch,
// query head) computes q' = R q (normalised by a power of two; R the layer's
// SRHT or dense Q) and, for QJL layers, t = S q' (fp16 hi/lo words), with
// sum q', sum t and the power of two, for the split-K kernels, which read them
// after griddepcontrol.wait.
//
// NH > 1 (head_dim 128 NH, SRHT layers only): the same for a vector of NH
// 128-dim blocks; hi words at [64 j, 64 j + 64) for block j, lo words after
// all NH blocks' hi words.
//
// NP = 2 (head_dim 64): lanes 0..15 hold dims 4 l .. 4 l + 3; hi words
// [0, 32), lo words [32, 64).
template <int NH, int NP = 1>
__global__ void __launch_bounds__(kThreads)
    decode_prep_kernel(const DecodeDims dims, const DecodeWorkspace ws, const float *S) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wid = blockIdx.x * (kThreads / 32) + warp;
    pdl_launch_dependents();
    if (wid >= dims.L * dims.B * dims.Hq) return;
    const int l = wid / (dims.B * dims.Hq);
    const LayerPlan &lp = ws.layer[l];
    if constexpr (NP == 2) {
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (lane < 16) load_q4(ws.q + static_cast<size_t>(wid) * (kD / 2), lane, x);
        warp_rotate_64(x, lp.sign_bits, dims.inv_sqrt_d, lane);
        if (lane >= 16) x[0] = x[1] = x[2] = x[3] = 0.f;
        const float f = warp_pow2_norm(x);
        float xn[4];
#pragma unroll
        for (int e = 0; e < 4; e++) xn[e] = x[e] * f;
        uint32_t *hi = ws.qrot + static_cast<size_t>(wid) * (kD / 2);
        float qs = 0.f;
        if (lane < 16) qs = store_hilo_block(hi, hi + kD / 4, xn, 0, lane);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) qs += __shfl_xor_sync(0xffffffffu, qs, o);
        if (lane == 0) {
            ws.qsum[static_cast<size_t>(wid) * 4] = qs / f;
            ws.qsum[static_cast<size_t>(wid) * 4 + 1] = 0.f;
            ws.qsum[static_cast<size_t>(wid) * 4 + 2] = 1.0f / f;
        }
        return;
    }
    if constexpr (NH > 1) {
        float y[NH][4];
#pragma unroll
        for (int j = 0; j < NH; j++) load_q4(ws.q + static_cast<size_t>(wid) * (NH * kD) + kD * j, lane, y[j]);
        warp_rotate_wide<NH>(y, lp.sign_bits, dims.inv_sqrt_d, lane);
        const float f = warp_pow2_norm_wide<NH>(y);
        uint32_t *hi = ws.qrot + static_cast<size_t>(wid) * (NH * kD);
        float qs = 0.f;
#pragma unroll
        for (int j = 0; j < NH; j++) {
            float yn[4];
#pragma unroll
            for (int e = 0; e < 4; e++) yn[e] = y[j][e] * f;
            qs += store_hilo_block(hi, hi + NH * kD / 2, yn, j, lane);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) qs += __shfl_xor_sync(0xffffffffu, qs, o);
        if (lane == 0) {
            ws.qsum[static_cast<size_t>(wid) * 4] = qs / f;
            ws.qsum[static_cast<size_t>(wid) * 4 + 1] = 0.f;
            ws.qsum[static_cast<size_t>(wid) * 4 + 2] = 1.0f / f;
        }
        return;
    }
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
        // t_j = (S q')_j for j = 4 lane + e (coalesced rows of S)
        float t[4];
        warp_matvec(S, x, t, lane);
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

PackedLauncher packed_launcher_narrow(int kb, int vb) {
    switch (kb) {
        case 1: return packed_launcher_narrow_kb1(vb);
        case 2: return packed_launcher_narrow_kb2(vb);
        case 3: return packed_launcher_narrow_kb3(vb);
        case 4: return packed_launcher_narrow_kb4(vb);
        case 5: return packed_launcher_narrow_kb5(vb);
        case 6: return packed_launcher_narrow_kb6(vb);
        case 7: return packed_launcher_narrow_kb7(vb);
        case 8: return packed_launcher_narrow_kb8(vb);
        default: return nullptr;
    }
}

PackedLauncher packed_launcher_wide(int kb, int vb, int nh) {
    switch (kb) {
        case 1: return packed_launcher_wide_kb1(vb, nh);
        case 2: return packed_launcher_wide_kb2(vb, nh);
        case 3: return packed_launcher_wide_kb3(vb, nh);
        case 4: return packed_launcher_wide_kb4(vb, nh);
        case 5: return packed_launcher_wide_kb5(vb, nh);
        case 6: return packed_launcher_wide_kb6(vb, nh);
        case 7: return packed_launcher_wide_kb7(vb, nh);
        case 8: return packed_launcher_wide_kb8(vb, nh);
        default: return nullptr;
    }
}

template <int NH, int NP = 1>
cudaError_t configure_fp16() {
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(decode_fp16_kernel<NH, NP>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, fp16_smem_bytes(NH, NP));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return cudaSuccess;
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
                                  cudaStream_t s, cudaEvent_t ev_start, cudaEvent_t ev_stop, int *n_launched) {
    *n_launched = 0;
    const int nh = dims.nh, np = dims.np;
    if ((nh != 1 && nh != 2 && nh != 4) || (np != 1 && np != 2) || (np == 2 && nh != 1)) return cudaErrorInvalidValue;
    {
        const cudaError_t e = np == 2    ? dec::configure_fp16<1, 2>()
                              : nh == 1 ? dec::configure_fp16<1>()
                              : nh == 2 ? dec::configure_fp16<2>()
                                        : dec::configure_fp16<4>();
        if (e != cudaSuccess) return e;
    }
    const size_t smem16 = static_cast<size_t>(dec::fp16_smem_bytes(nh, np));
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
        const unsigned grid = static_cast<unsigned>((n_warps + 3) / 4);
        if (np == 2) dec::decode_prep_kernel<1, 2><<<grid, dec::kThreads, 0, s>>>(dims, ws, S);
        else if (nh == 1) dec::decode_prep_kernel<1><<<grid, dec::kThreads, 0, s>>>(dims, ws, S);
        else if (nh == 2) dec::decode_prep_kernel<2><<<grid, dec::kThreads, 0, s>>>(dims, ws, S);
        else dec::decode_prep_kernel<4><<<grid, dec::kThreads, 0, s>>>(dims, ws, S);
        first = false;
        ++*n_launched;
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
        const PackedLauncher fn = c.qjl && (nh != 1 || np != 1) ? nullptr
                                  : np == 2                   ? dec::packed_launcher_narrow(c.kb, c.vb)
                                  : nh == 1                   ? dec::packed_launcher(c.kb, c.vb, c.qjl != 0)
                                                              : dec::packed_launcher_wide(c.kb, c.vb, nh);
        if (!fn) return cudaErrorInvalidValue;
        const cudaError_t e =
            fn(dims, ws, ws.cta_item + c.cta_off, c.n_ctas, c.n_stages, value_half[i], value_c1[i], s, !first);
        if (e != cudaSuccess) return e;
        first = false;
        ++*n_launched;
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
        const cudaError_t e =
            np == 2   ? cudaLaunchKernelEx(&cfg, dec::decode_fp16_kernel<1, 2>, dims, ws, ws.cta_item + c.cta_off)
            : nh == 1 ? cudaLaunchKernelEx(&cfg, dec::decode_fp16_kernel<1>, dims, ws, ws.cta_item + c.cta_off)
            : nh == 2 ? cudaLaunchKernelEx(&cfg, dec::decode_fp16_kernel<2>, dims, ws, ws.cta_item + c.cta_off)
                      : cudaLaunchKernelEx(&cfg, dec::decode_fp16_kernel<4>, dims, ws, ws.cta_item + c.cta_off);
        if (e != cudaSuccess) return e;
        ++*n_launched;
        first = false;
    }
    return cudaGetLastError();
}

}  // namespace tqk
