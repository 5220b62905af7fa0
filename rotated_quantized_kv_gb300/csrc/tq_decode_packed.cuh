// tq_decode_packed.cuh -- split-K decode attention over packed segments,
// specialised per (key bits, value bits, QJL) class.
//
// Method: attention on the compressed cache ("turboquant-mlx" skill note,
// "Optimisations Metal"; "turboquant-mlx", "Implementation Status"), keys
// scored in the rotated space q' . yhat with yhat = alpha*code + beta, values
// summed in the rotated space and rotated back once by the combine kernel.
//
// Persistent CTAs of 4 warps share the class's 128-token stages (over all
// (layer x segment x KV head, batch) groups) in equal contiguous ranges.  One
// thread streams each CTA's stages into 2-4 shared buffers with TMA bulk copies
// (cp.async.bulk, completion on an mbarrier per buffer); warp w owns tokens
// [32w, 32w + 32) of each stage, two 16-token tiles:
//   Q.K  mma.m16n8k16: A = 16 tokens x 16 dims of raw key codes written as
//        fp16 subnormals (code * 2^-24, exact), B = the GQA group's 4 query
//        heads as fp16 hi/lo column pairs.  Thread (g, c) owns dims
//        [32c, 32c + 32) of a record; which two codes share an A register is
//        chosen per bit width so that one or two integer instructions extract
//        them (KUnpack), and the B fragment is gathered with the same map.
//   P.V  mma.m16n8k16: A = 16 dims x 16 tokens of fp16 codebook values, B =
//        probabilities (<= 2^8 with a lazy running max) times the value scale
//        in fp16, one column per query head.  Thread (g, c)
//        owns dims [16g, 16g + 16); codebook lookups are byte permutes (PRMT)
//        on register-resident tables for 1-4 bits, shared-memory loads above.
#pragma once

#include "tq_decode_common.cuh"

namespace tqk {
namespace dec {

// ------------------------------------------------------------------- keys
// run(): 16 A registers from the thread's KB-word window (codes 0..31 of its
// 32-dim slice); register r feeds k-step r/2 (r even: a0/a1 rows, r odd: a2/a3).
// dim(r, half): the code index (0..31) in the low (0) / high (1) fp16 half.
template <int KB>
struct KUnpack {  // 3, 5, 6, 7 bits: pairs (j, j+16) from 16-bit slices
    static constexpr __host__ __device__ int dim(int r, int half) { return r + 16 * half; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[KB], uint32_t (&a)[16]) {
        constexpr uint32_t M = (1u << KB) - 1u;
        constexpr uint32_t MM = M | (M << 16);
        uint32_t X[KB];  // low half: slice s of codes 0-15, high half: slice s of codes 16-31
#pragma unroll
        for (int s = 0; s < KB; s++) {
            const int ua = s, ub = KB + s;  // 16-bit units of the window
            const uint32_t sel = ((ua & 1) ? 0x32u : 0x10u) | (((ub & 1) ? 0x76u : 0x54u) << 8);
            X[s] = prmt(w[ua >> 1], w[ub >> 1], sel);
        }
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const int bit = KB * j, s = bit >> 4, loc = bit & 15;
            if (loc + KB <= 16) {
                a[j] = (loc ? (X[s] >> loc) : X[s]) & MM;
            } else {
                const int ba = bit, bb = 16 * KB + bit;
                const uint32_t va = ((ba & 31) + KB <= 32) ? (w[ba >> 5] >> (ba & 31))
                                                           : __funnelshift_r(w[ba >> 5], w[(ba >> 5) + 1], ba & 31);
                const uint32_t vb = ((bb & 31) + KB <= 32) ? (w[bb >> 5] >> (bb & 31))
                                                           : __funnelshift_r(w[bb >> 5], w[(bb >> 5) + 1], bb & 31);
                a[j] = prmt(va, vb, 0x5410u) & MM;
            }
        }
    }
};

template <>
struct KUnpack<1> {  // pairs (r, r+16) of one word
    static constexpr __host__ __device__ int dim(int r, int half) { return r + 16 * half; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[1], uint32_t (&a)[16]) {
#pragma unroll
        for (int r = 0; r < 16; r++) a[r] = (w[0] >> r) & 0x00010001u;
    }
};

template <>
struct KUnpack<2> {  // word i, shift 2e: codes (16i + e, 16i + e + 8)
    static constexpr __host__ __device__ int dim(int r, int half) { return 16 * (r >> 3) + (r & 7) + 8 * half; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[2], uint32_t (&a)[16]) {
#pragma unroll
        for (int r = 0; r < 16; r++) a[r] = (w[r >> 3] >> (2 * (r & 7))) & 0x00030003u;
    }
};

template <>
struct KUnpack<4> {  // word i, shift 4e: codes (8i + e, 8i + e + 4)
    static constexpr __host__ __device__ int dim(int r, int half) { return 8 * (r >> 2) + (r & 3) + 4 * half; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[4], uint32_t (&a)[16]) {
#pragma unroll
        for (int r = 0; r < 16; r++) a[r] = (w[r >> 2] >> (4 * (r & 3))) & 0x000F000Fu;
    }
};

template <>
struct KUnpack<8> {  // bytes (2e, 2e+1) of word i zero-extended: codes (4i + 2e, 4i + 2e + 1)
    static constexpr __host__ __device__ int dim(int r, int half) { return 4 * (r >> 1) + 2 * (r & 1) + half; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[8], uint32_t (&a)[16]) {
#pragma unroll
        for (int r = 0; r < 16; r++) a[r] = prmt(w[r >> 1], 0u, (r & 1) ? 0x4342u : 0x4140u);
    }
};

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

// Raw Q.K (in units of 2^-24 code units) of tokens g and g+8 for head c.
template <int KB>
__device__ __forceinline__ void qk_raw(const uint8_t *rec0, const uint8_t *rec1, const uint32_t (&bq)[16],
                                       float &raw0, float &raw1) {
    uint32_t w0[KB], w1[KB], a0[16], a1[16];
    lds_words(w0, rec0);
    lds_words(w1, rec1);
    KUnpack<KB>::run(w0, a0);
    KUnpack<KB>::run(w1, a1);
    float e[4] = {0.f, 0.f, 0.f, 0.f}, o[4] = {0.f, 0.f, 0.f, 0.f};  // two chains for ILP
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) {
        mma16816(e, a0[2 * kk], a1[2 * kk], a0[2 * kk + 1], a1[2 * kk + 1], bq[2 * kk], bq[2 * kk + 1]);
        mma16816(o, a0[2 * kk + 2], a1[2 * kk + 2], a0[2 * kk + 3], a1[2 * kk + 3], bq[2 * kk + 2],
                 bq[2 * kk + 3]);
    }
    raw0 = (e[0] + e[1]) + (o[0] + o[1]);
    raw1 = (e[2] + e[3]) + (o[2] + o[3]);
}

// B fragment (16 registers) of a natural-order fp16 vector slice: words q[0..15]
// hold dims 2i, 2i+1 of the thread's 32-dim slice; register r pairs dims
// KU::dim(r, 0) and KU::dim(r, 1).
template <typename KU>
__device__ __forceinline__ void gather_b(const uint32_t (&q)[16], uint32_t (&b)[16]) {
#pragma unroll
    for (int r = 0; r < 16; r++) {
        const int d0 = KU::dim(r, 0), d1 = KU::dim(r, 1);
        const uint32_t sel = ((d0 & 1) ? 0x32u : 0x10u) | (((d1 & 1) ? 0x76u : 0x54u) << 8);
        b[r] = prmt(q[d0 >> 1], q[d1 >> 1], sel);
    }
}

// ------------------------------------------------------------------- values
// Window of the thread's 16 value codes (bits [16g VB, 16g VB + 16 VB) of the
// record) as little-endian words.
template <int VB>
struct VWin {
    static constexpr int NW = (2 * VB + 3) / 4;
    // p: the record plus the thread's window offset rounded down to 4 bytes;
    // sh: 8 * (window offset mod 4), 0 or 16
    static __device__ __forceinline__ void load(const uint8_t *p8, int sh, uint32_t (&x)[NW]) {
        const uint32_t *p = reinterpret_cast<const uint32_t *>(p8);
        if constexpr (VB % 2 == 0) {
#pragma unroll
            for (int i = 0; i < NW; i++) x[i] = p[i];
        } else {
            uint32_t raw[NW];
#pragma unroll
            for (int i = 0; i < NW; i++) raw[i] = p[i];
#pragma unroll
            for (int i = 0; i < NW; i++) x[i] = __funnelshift_r(raw[i], i + 1 < NW ? raw[i + 1] : 0u, sh);
        }
    }
};

// Codebook value tables for byte permutes: tl[i] / th[i] hold the low / high
// bytes of fp16 entries 4i..4i+3.
struct PrmtTable {
    uint32_t tl[4], th[4];
};

// 8 nibbles of eight 3-bit codes (bits 0..23 of v; higher bits ignored).
__device__ __forceinline__ uint32_t spread3(uint32_t v) {
    uint32_t t = (v & 0x00000FFFu) | ((v << 4) & 0x0FFF0000u);
    t = (t & 0x003F003Fu) | ((t << 2) & 0x3F003F00u);
    return (t & 0x07070707u) | ((t << 1) & 0x70707070u);
}

// Lookup of 4 codes given as selector nibbles [x_j, x_j', y_j, y_j'] (3-bit
// indices, bit 3 clear): returns half2(c[x_j], c[y_j]) and half2(c[x_j'], c[y_j']).
template <int VB>
__device__ __forceinline__ void lookup4(uint32_t sel, const PrmtTable &t, uint32_t &ra, uint32_t &rb) {
    uint32_t pl, ph;
    if constexpr (VB <= 3) {
        pl = prmt(t.tl[0], t.tl[1], sel);
        ph = prmt(t.th[0], t.th[1], sel);
    } else {  // 4 bits: two 8-entry tables, chosen per byte by the nibble's bit 3
        const uint32_t s7 = sel & 0x7777u;
        const uint32_t hb = ((sel >> 1) & 0x4444u) | 0x3210u;
        pl = prmt(prmt(t.tl[0], t.tl[1], s7), prmt(t.tl[2], t.tl[3], s7), hb);
        ph = prmt(prmt(t.th[0], t.th[1], s7), prmt(t.th[2], t.th[3], s7), hb);
    }
    ra = prmt(pl, ph, 0x6240u);
    rb = prmt(pl, ph, 0x7351u);
}

// dim(mt, r): the code index (0..15) of accumulator row r (0: row g, 1: row
// g+8) of m-tile mt.  run(): the A registers of one token pair (x, y) for all
// eight m-tiles: ra[mt] for row g, rb[mt] for row g+8.
template <int VB>
struct VUnpack {  // 5..8 bits: shared-memory table, codes (2mt, 2mt+1)
    static constexpr __host__ __device__ int dim(int mt, int r) { return 2 * mt + r; }
    template <int NW>
    static __device__ __forceinline__ uint32_t code(const uint32_t (&x)[NW], int j) {
        const int bit = VB * j, wi = bit >> 5, sh = bit & 31;
        const uint32_t v = (sh + VB <= 32) ? (x[wi] >> sh) : __funnelshift_r(x[wi], x[wi + 1], sh);
        return v & ((1u << VB) - 1u);
    }
    static __device__ __forceinline__ void run(const uint32_t (&x)[VWin<VB>::NW], const uint32_t (&y)[VWin<VB>::NW],
                                               const PrmtTable &, const unsigned short *ctab, uint32_t (&ra)[8],
                                               uint32_t (&rb)[8]) {
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            ra[mt] = static_cast<uint32_t>(ctab[code(x, 2 * mt)]) | (static_cast<uint32_t>(ctab[code(y, 2 * mt)]) << 16);
            rb[mt] = static_cast<uint32_t>(ctab[code(x, 2 * mt + 1)]) |
                     (static_cast<uint32_t>(ctab[code(y, 2 * mt + 1)]) << 16);
        }
    }
};

template <>
struct VUnpack<1> {  // nibble selectors (Z >> e) & 0x1111 with Z = bytes interleaved: codes (e, e+4)
    static constexpr __host__ __device__ int dim(int mt, int r) { return 8 * (mt >> 2) + (mt & 3) + 4 * r; }
    static __device__ __forceinline__ void run(const uint32_t (&x)[1], const uint32_t (&y)[1], const PrmtTable &t,
                                               const unsigned short *, uint32_t (&ra)[8], uint32_t (&rb)[8]) {
        const uint32_t Z = prmt(x[0], y[0], 0x5140u);  // [x.b0, y.b0, x.b1, y.b1]
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            const int sh = (mt >> 2) * 16 + (mt & 3);
            lookup4<1>((Z >> sh) & 0x1111u, t, ra[mt], rb[mt]);
        }
    }
};

template <>
struct VUnpack<2> {  // byte k of both tokens, shift 2e: codes (4k + e, 4k + e + 2)
    static constexpr __host__ __device__ int dim(int mt, int r) { return 4 * (mt >> 1) + (mt & 1) + 2 * r; }
    static __device__ __forceinline__ void run(const uint32_t (&x)[1], const uint32_t (&y)[1], const PrmtTable &t,
                                               const unsigned short *, uint32_t (&ra)[8], uint32_t (&rb)[8]) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint32_t Z = prmt(x[0], y[0], static_cast<uint32_t>(k | ((k + 4) << 4)));
            lookup4<2>(Z & 0x3333u, t, ra[2 * k], rb[2 * k]);
            lookup4<2>((Z >> 2) & 0x3333u, t, ra[2 * k + 1], rb[2 * k + 1]);
        }
    }
};

template <>
struct VUnpack<3> {  // codes spread to nibbles; selector = byte k of both tokens: codes (2mt, 2mt+1)
    static constexpr __host__ __device__ int dim(int mt, int r) { return 2 * mt + r; }
    static __device__ __forceinline__ void run(const uint32_t (&x)[2], const uint32_t (&y)[2], const PrmtTable &t,
                                               const unsigned short *, uint32_t (&ra)[8], uint32_t (&rb)[8]) {
        const uint32_t sx[2] = {spread3(x[0]), spread3(__funnelshift_r(x[0], x[1], 24))};
        const uint32_t sy[2] = {spread3(y[0]), spread3(__funnelshift_r(y[0], y[1], 24))};
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            const int h = mt >> 2, k = mt & 3;
            const uint32_t sel = prmt(sx[h], sy[h], static_cast<uint32_t>(k | ((k + 4) << 4)));
            lookup4<3>(sel, t, ra[mt], rb[mt]);
        }
    }
};

template <>
struct VUnpack<4> {  // nibbles already; selector = byte k of both tokens: codes (2mt, 2mt+1)
    static constexpr __host__ __device__ int dim(int mt, int r) { return 2 * mt + r; }
    static __device__ __forceinline__ void run(const uint32_t (&x)[2], const uint32_t (&y)[2], const PrmtTable &t,
                                               const unsigned short *, uint32_t (&ra)[8], uint32_t (&rb)[8]) {
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            const int h = mt >> 2, k = mt & 3;
            const uint32_t sel = prmt(x[h], y[h], static_cast<uint32_t>(k | ((k + 4) << 4)));
            lookup4<4>(sel, t, ra[mt], rb[mt]);
        }
    }
};

// ------------------------------------------------------------------- kernel
struct ValueTable {
    unsigned short half[256];  // fp16 codebook values of this class's value width
};

constexpr int kPT = kPackedStageTokens;  // 32 tokens per warp: two 16-token tiles

template <int KB, int VB, bool QJL>
struct PackedGeom {
    static constexpr int RK = 16 * KB, RV = 16 * VB;
    static constexpr int offV = kPT * RK;
    static constexpr int offKS = offV + kPT * RV;
    static constexpr int offVS = offKS + kPT * 4;
    static constexpr int offQS = offVS + kPT * 4;
    static constexpr int offQN = offQS + kPT * 16;
    static constexpr int stage = QJL ? offQN + kPT * 4 : offQS;
    static constexpr int fixed = (VB >= 5 ? 512 : 0) + kMaxGqa * kD * 4 + 64;  // codebook, queries, flag, barriers
    // as many stages in flight (2..4) as fit with kPackedCtasPerSm CTAs per SM
    static constexpr int fit = (227 * 1024 / kPackedCtasPerSm - 1024 - fixed) / stage;
    static constexpr int stages = fit > 4 ? 4 : (fit < 2 ? 2 : fit);
    static constexpr int ctab = stages * stage;                  // fp16 codebook (5-8 bits)
    static constexpr int qoff = ctab + (VB >= 5 ? 512 : 0);      // rotated queries [4][128] words, sums [4]
    static constexpr int flag = qoff + kMaxGqa * kD * 4 + 16;
    static constexpr int bar = flag + 16;                        // one mbarrier per stage buffer
    static constexpr int smem = bar + 8 * stages;
};

// Position of a stage in the class's stage sequence (item, batch element,
// stage within the (item, batch) group); with PTRS, the group's base pointers.
template <bool QJL, bool PTRS>
struct StageCursor {
    int item, b, st, n_stages, n_tokens;
    const uint8_t *kc, *vc, *qs;
    const float *ks, *vs, *qn;
    __device__ __forceinline__ void bind(const WorkItem *items) {
        const WorkItem &it = items[item];
        n_stages = it.n_stages;
        n_tokens = it.n_tokens;
        if constexpr (!PTRS) return;
        kc = it.kc + b * it.kstride;
        vc = it.vc + b * it.vstride;
        ks = it.ks + static_cast<size_t>(b) * it.sstride;
        vs = it.vs + static_cast<size_t>(b) * it.sstride;
        if constexpr (QJL) {
            qs = it.qs + static_cast<size_t>(b) * it.qstride * 16;
            qn = it.qn + static_cast<size_t>(b) * it.qstride;
        }
    }
    __device__ __forceinline__ void locate(const WorkItem *items, int lo, int hi, long long s) {
        item = find_stage_item(items, lo, hi, s);
        const long long r = s - items[item].stage_begin;
        const int ns = items[item].n_stages;
        b = static_cast<int>(r / ns);
        st = static_cast<int>(r - static_cast<long long>(b) * ns);
        bind(items);
    }
    // returns true when the next stage starts a new group
    __device__ __forceinline__ bool advance(const WorkItem *items, int B, bool rebind) {
        if (++st < n_stages) return false;
        st = 0;
        if (++b == B) {
            b = 0;
            ++item;
        }
        if (rebind) bind(items);
        return true;
    }
};

// Persistent split-K kernel of one class: gridDim.x CTAs share the class's S
// stages in equal contiguous ranges and stream them through one cp.async
// pipeline that never drains at group boundaries.  Each CTA writes one partial
// per (item, batch) group it touches; the CTA completing a (layer, batch, KV
// head) merges its partials (finish_and_combine).
template <int KB, int VB, bool QJL>
__global__ void __launch_bounds__(kThreads, kPackedCtasPerSm)
    decode_packed_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int item_lo, const int item_hi,
                         const long long S, const __grid_constant__ ValueTable vt) {
    using G = PackedGeom<KB, VB, QJL>;
    constexpr int NS = G::stages;
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int gqa = dims.gqa, B = dims.B;
    const long long s_begin = range_begin(blockIdx.x, S, gridDim.x);
    const int n_st = static_cast<int>(range_begin(blockIdx.x + 1, S, gridDim.x) - s_begin);
    pdl_launch_dependents();

    unsigned short *ctab = reinterpret_cast<unsigned short *>(smem + G::ctab);
    if constexpr (VB >= 5) {
        for (int i = threadIdx.x; i < (1 << VB); i += kThreads) ctab[i] = vt.half[i];
    }
    PrmtTable ptab;
    if constexpr (VB <= 4) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int k = 4 * i + e;
                const uint32_t v = k < (1 << VB) ? vt.half[k] : 0u;
                lo |= (v & 0xFFu) << (8 * e);
                hi |= (v >> 8) << (8 * e);
            }
            ptab.tl[i] = lo;
            ptab.th[i] = hi;
        }
    }

    // ---- loader (thread 0): stage k of this CTA's range into buffer k % NS by
    // TMA bulk copies completing on full[k % NS]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + G::bar);
    StageCursor<QJL, true> lc;
    if (threadIdx.x == 0) {
        lc.locate(ws.items, item_lo, item_hi, s_begin);
#pragma unroll
        for (int i = 0; i < NS; i++) mbar_init(&full[i], 1);
        mbar_init_fence();
    }
    __syncthreads();
    int loads_left = n_st;
    auto load_next = [&](int k) {
        uint64_t *bar = &full[k % NS];
        uint8_t *dst = smem + (k % NS) * G::stage;
        const int t0 = lc.st * kPT;
        const int n = min(kPT, lc.n_tokens - t0);
        // scale runs are rounded up to 16 bytes: rows hold a multiple of 16 tokens
        const unsigned nk = n * G::RK, nv = n * G::RV, ns = (n * 4 + 15) & ~15u;
        const unsigned total = nk + nv + 2 * ns + (QJL ? n * 16 + ns : 0);
        fence_proxy_async();
        mbar_expect_tx(bar, total);
        bulk_g2s(dst, lc.kc + static_cast<size_t>(t0) * G::RK, nk, bar);
        bulk_g2s(dst + G::offV, lc.vc + static_cast<size_t>(t0) * G::RV, nv, bar);
        bulk_g2s(dst + G::offKS, lc.ks + t0, ns, bar);
        bulk_g2s(dst + G::offVS, lc.vs + t0, ns, bar);
        if constexpr (QJL) {
            bulk_g2s(dst + G::offQS, lc.qs + static_cast<size_t>(t0) * 16, n * 16, bar);
            bulk_g2s(dst + G::offQN, lc.qn + t0, ns, bar);
        }
        // rebind only if another stage follows in this CTA's range
        lc.advance(ws.items, B, --loads_left > 0);
    };
    if (threadIdx.x == 0) {
        for (int k = 0; k < NS - 1 && k < n_st; k++) load_next(k);
    }
    if constexpr (QJL) pdl_wait();  // the prep kernel's outputs

    // ---- consumer
    StageCursor<QJL, false> cc;
    cc.locate(ws.items, item_lo, item_hi, s_begin);
    int g_layer = 0, g_head = 0, g_b = 0, g_item = 0;
    long long g_stage0 = 0;  // class stage index of the group's first stage
    uint32_t bq[16], bt[16];
    float qsum = 0.f, tsum = 0.f;
    WarpState st;
    uint32_t *qsh = reinterpret_cast<uint32_t *>(smem + G::qoff);
    float *qs_sum = reinterpret_cast<float *>(qsh + kMaxGqa * kD);
    int *flag = reinterpret_cast<int *>(smem + G::flag);
    constexpr float alpha = 16777216.0f * 2.0f / static_cast<float>(1 << KB);  // 2^(1-KB), times 2^24
    constexpr float beta = 1.0f / static_cast<float>(1 << KB) - 1.0f;
    const float qk_scale = dims.qk_scale;
    // per-thread byte offsets of the key window (codes [32c, 32c+32) of token
    // row g) and of the value window (codes [16g, 16g+16) of token row 2c)
    const int koff = g * G::RK + 4 * KB * c;
    const int voff = 2 * c * G::RV + ((2 * VB * g) & ~3);
    const int vsh = ((2 * VB * g) & 3) * 8;

    // each warp writes its own partial of the current group; then the group's
    // CTA-level count (and possibly the merge)
    auto flush = [&]() {
        const long long gr = static_cast<long long>(g_item) * B + g_b;
        const int slot = ws.grp_part[gr] +
                         kDecodeWarps * static_cast<int>(blockIdx.x - cta_of_stage(g_stage0, S, gridDim.x)) + warp;
        write_warp_partial_pair(st, ws.part + static_cast<size_t>(slot) * (kMaxGqa * kPartStride), gqa,
                                [g](int mt, int r) { return 16 * g + VUnpack<VB>::dim(mt, r); });
        finish_and_combine(dims, ws, g_layer, g_b, g_head, flag);
    };
    // a new group: its identity and the B fragments of its rotated queries
    // (column g: head g/2, part g&1)
    auto start_group = [&]() {
        const WorkItem &it = ws.items[cc.item];
        g_item = cc.item;
        g_b = cc.b;
        g_layer = it.layer;
        g_head = it.head;
        g_stage0 = it.stage_begin + static_cast<long long>(cc.b) * it.n_stages;
        init_state(st);
        const size_t qbase = (static_cast<size_t>(g_layer) * B + g_b) * dims.Hq + g_head * gqa;
        const int head = g >> 1, part = g & 1;
        uint32_t q[16];
        if constexpr (QJL) {
            const uint32_t *qw = ws.qrot + ((qbase + head) * 2 + part) * (kD / 2) + 16 * c;
#pragma unroll
            for (int i = 0; i < 16; i++) q[i] = head < gqa ? qw[i] : 0u;
            gather_b<KUnpack<KB>>(q, bq);
            const uint32_t *tw = ws.qjlt + ((qbase + head) * 2 + part) * (kD / 2) + 16 * c;
#pragma unroll
            for (int i = 0; i < 16; i++) q[i] = head < gqa ? tw[i] : 0u;
            gather_b<KUnpack<1>>(q, bt);
            qsum = c < gqa ? ws.qsum[(qbase + c) * 4] : 0.f;
            tsum = c < gqa ? ws.qsum[(qbase + c) * 4 + 1] : 0.f;
        } else {
            if (warp < gqa) {  // warp w rotates query head w of the group
                float x[4];
                load_q4(ws.q + (qbase + warp) * kD, lane, x);
                warp_rotate(x, ws.layer[g_layer].sign_bits, dims.inv_sqrt_d, lane);
                const float sm = store_hilo(qsh + warp * kD, x, lane);
                if (lane == 0) qs_sum[warp] = sm;
            }
            __syncthreads();
            const uint32_t *qw = qsh + head * kD + part * (kD / 2) + 16 * c;
#pragma unroll
            for (int i = 0; i < 16; i++) q[i] = head < gqa ? qw[i] : 0u;
            gather_b<KUnpack<KB>>(q, bq);
            qsum = c < gqa ? qs_sum[c] : 0.f;
            __syncthreads();
        }
    };
    start_group();
    bool new_group = false;

    for (int k = 0; k < n_st; k++) {
        const bool arrived = mbar_wait(&full[k % NS], (k / NS) & 1);
        // all warps are past stage k-1 (its buffer is free) and agree on errors
        if (__syncthreads_or(!arrived)) {
            if (threadIdx.x == 0) {
                atomicExch(ws.error, 1);
                // let the copies still in flight land before the CTA's shared memory goes away
                for (int j = k; j < n_st && j < k + NS - 1; j++) mbar_wait(&full[j % NS], (j / NS) & 1);
            }
            __syncthreads();
            return;
        }
        if (threadIdx.x == 0 && k + NS - 1 < n_st) load_next(k + NS - 1);
        if (new_group) {
            flush();
            start_group();
        }
        const uint8_t *buf = smem + (k % NS) * G::stage;
        const int n = min(kPT, cc.n_tokens - cc.st * kPT);
        new_group = cc.advance(ws.items, B, k + 1 < n_st);
        const int tA = warp * 32;  // this warp's tiles: tokens [tA, tA + 16) and [tA + 16, tA + 32)
        if (tA >= n) continue;
        const bool has_b = tA + 16 < n;
        // ---- scores of both tiles
        float sc[4];
        const float *kss = reinterpret_cast<const float *>(buf + G::offKS);
        const float *qns = reinterpret_cast<const float *>(buf + G::offQN);
#pragma unroll
        for (int t = 0; t < 2; t++) {
            const int t0 = tA + 16 * t;
            float raw0, raw1;
            qk_raw<KB>(buf + t0 * G::RK + koff, buf + (t0 + 8) * G::RK + koff, bq, raw0, raw1);
            float s0 = kss[t0 + g] * (alpha * raw0 + beta * qsum);
            float s1 = kss[t0 + g + 8] * (alpha * raw1 + beta * qsum);
            if constexpr (QJL) {
                float r0, r1;
                qk_raw<1>(buf + G::offQS + (t0 + g) * 16 + 4 * c, buf + G::offQS + (t0 + g + 8) * 16 + 4 * c, bt, r0,
                          r1);
                constexpr float gam = 1.2533141373155003f / kJl;  // sqrt(pi/2) / jl
                s0 += gam * qns[t0 + g] * (33554432.0f * r0 - tsum);
                s1 += gam * qns[t0 + g + 8] * (33554432.0f * r1 - tsum);
            }
            sc[2 * t] = s0 * qk_scale;
            sc[2 * t + 1] = s1 * qk_scale;
        }
        const float *vss = reinterpret_cast<const float *>(buf + G::offVS);
        const bool okv[4] = {tA + g < n, tA + g + 8 < n, tA + 16 + g < n, tA + 24 + g < n};
        const float vsv[4] = {vss[tA + g], vss[tA + g + 8], vss[tA + 16 + g], vss[tA + 24 + g]};
        uint32_t bp[4];
        softmax_pair(st, sc, okv, vsv, g, c, gqa, bp);
        // ---- values of both tiles
        const uint8_t *vst = buf + G::offV;
#pragma unroll
        for (int t = 0; t < 2; t++) {
            if (t == 1 && !has_b) break;
            const uint8_t *vb = vst + (tA + 16 * t) * G::RV;
            uint32_t x0[VWin<VB>::NW], x1[VWin<VB>::NW], x2[VWin<VB>::NW], x3[VWin<VB>::NW];
            VWin<VB>::load(vb + voff, vsh, x0);
            VWin<VB>::load(vb + voff + G::RV, vsh, x1);
            VWin<VB>::load(vb + voff + 8 * G::RV, vsh, x2);
            VWin<VB>::load(vb + voff + 9 * G::RV, vsh, x3);
            uint32_t ra[8], rb[8], rc[8], rd[8];
            VUnpack<VB>::run(x0, x1, ptab, ctab, ra, rb);
            VUnpack<VB>::run(x2, x3, ptab, ctab, rc, rd);
#pragma unroll
            for (int mt = 0; mt < 8; mt++)
                mma16816(st.acc[mt], ra[mt], rb[mt], rc[mt], rd[mt], bp[2 * t], bp[2 * t + 1]);
        }
    }
    // every thread waits for the previous grid of the call before its last
    // merge, so that this grid's completion implies that of all earlier ones
    pdl_wait();
    flush();
}

template <int KB, int VB, bool QJL>
cudaError_t launch_packed(const DecodeDims &dims, const DecodeWorkspace &ws, int item_lo, int item_hi, int n_ctas,
                          long long n_stages, const unsigned short *value_half, cudaStream_t s, bool pdl) {
    using G = PackedGeom<KB, VB, QJL>;
    static bool configured = false;
    if (!configured) {
        if (G::smem > 48 * 1024) {
            const cudaError_t e = cudaFuncSetAttribute(decode_packed_kernel<KB, VB, QJL>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, G::smem);
            if (e != cudaSuccess) return e;
        }
        configured = true;
    }
    ValueTable vt;
    for (int i = 0; i < 256; i++) vt.half[i] = i < (1 << VB) ? value_half[i] : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = G::smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_packed_kernel<KB, VB, QJL>, dims, ws, item_lo, item_hi, n_stages, vt);
}

}  // namespace dec
}  // namespace tqk

// One translation unit per key width instantiates every value width, with and
// without QJL.
#define TQ_INSTANTIATE_PACKED_KB(KB)                                                                          \
    namespace tqk {                                                                                            \
    PackedLauncher packed_launcher_kb##KB(int vb, bool qjl) {                                                  \
        switch (vb * 2 + (qjl ? 1 : 0)) {                                                                      \
            case 2: return dec::launch_packed<KB, 1, false>;                                                   \
            case 3: return dec::launch_packed<KB, 1, true>;                                                    \
            case 4: return dec::launch_packed<KB, 2, false>;                                                   \
            case 5: return dec::launch_packed<KB, 2, true>;                                                    \
            case 6: return dec::launch_packed<KB, 3, false>;                                                   \
            case 7: return dec::launch_packed<KB, 3, true>;                                                    \
            case 8: return dec::launch_packed<KB, 4, false>;                                                   \
            case 9: return dec::launch_packed<KB, 4, true>;                                                    \
            case 10: return dec::launch_packed<KB, 5, false>;                                                  \
            case 11: return dec::launch_packed<KB, 5, true>;                                                   \
            case 12: return dec::launch_packed<KB, 6, false>;                                                  \
            case 13: return dec::launch_packed<KB, 6, true>;                                                   \
            case 14: return dec::launch_packed<KB, 7, false>;                                                  \
            case 15: return dec::launch_packed<KB, 7, true>;                                                   \
            case 16: return dec::launch_packed<KB, 8, false>;                                                  \
            case 17: return dec::launch_packed<KB, 8, true>;                                                   \
            default: return nullptr;                                                                           \
        }                                                                                                      \
    }                                                                                                          \
    }
