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
//   Q.K  mma.m16n8k16: A = 16 tokens x 16 dims of raw key codes left at their
//        bit offset s inside an fp16 half (code * 2^(s-24), a subnormal, so one
//        AND extracts two codes), B = the GQA group's 4 query heads as fp16
//        hi/lo column pairs, each element scaled by 2^(kA-s), so that every
//        product is q * code * 2^(kA-24).  Thread (g, c) owns dims
//        [32c, 32c + 32) of a record; which two codes share an A register is
//        chosen per bit width (KUnpack) and the B fragment uses the same map.
//   P.V  mma.m16n8k16: A = 16 dims x 16 tokens of values, B = probabilities
//        (<= 2^8 with a lazy running max) times the value scale in fp16, one
//        column per query head.  Thread (g, c) owns dims [16g, 16g + 16).  An A
//        register pairs one dim of two tokens; its decoding depends on the
//        value width (VDec):
//          1 bit   the codebook is +-c1, affine in the code: A holds the code
//                  bit as a subnormal and the record is finished as
//                  c1 * (2 acc - sum of weights);
//          2, 3    one shared-memory load per register from a table of fp16
//                  pairs (c[x], c[y]) indexed by both tokens' codes, one
//                  column of the table per lane (no bank conflicts);
//          4       byte permutes (PRMT) on register-resident tables;
//          5-8     per-code loads from a shared-memory codebook.
#pragma once

#include <type_traits>

#include "tq_decode_common.cuh"

namespace tqk {
namespace dec {

// bits of the fp16 power of two 2^k (0 <= k <= 15)
__host__ __device__ constexpr uint32_t half_pow2_bits(int k) { return static_cast<uint32_t>(15 + k) << 10; }

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// ------------------------------------------------------------------- keys
// run(): 16 A registers from the thread's KB-word window (codes 0..31 of its
// 32-dim slice); register r feeds k-step r/2 (r even: a0/a1 rows, r odd:
// a2/a3).  dim(r, half): the code index (0..31) in the low (0) / high (1) fp16
// half; shift(r, half): its bit offset s inside the half (the half holds
// code * 2^(s-24)).  kA: the largest shift; the B fragment holds q * 2^(kA-s).
template <int KB>
struct KUnpack {  // 5, 6, 7 bits: pairs (j, j+16) from 16-bit slices, shifted down
    static constexpr int kA = 0;
    static constexpr __host__ __device__ int dim(int r, int half) { return r + 16 * half; }
    static constexpr __host__ __device__ int shift(int, int) { return 0; }
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
struct KUnpack<1> {  // codes (r, r+16) at bit r (r < 10) or, after >> 10, bit r - 10
    static constexpr int kA = 9;
    static constexpr __host__ __device__ int dim(int r, int half) { return r + 16 * half; }
    static constexpr __host__ __device__ int shift(int r, int) { return r < 10 ? r : r - 10; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[1], uint32_t (&a)[16]) {
        const uint32_t t = w[0] >> 10;
#pragma unroll
        for (int r = 0; r < 16; r++) a[r] = (r < 10 ? w[0] : t) & (0x00010001u << shift(r, 0));
    }
};

template <>
struct KUnpack<2> {  // word i: codes (16i + e, 16i + 8 + e), e < 5 in place, e >= 5 after >> 10
    static constexpr int kA = 8;
    static constexpr __host__ __device__ int dim(int r, int half) { return 16 * (r >> 3) + (r & 7) + 8 * half; }
    static constexpr __host__ __device__ int shift(int r, int) { return (r & 7) < 5 ? 2 * (r & 7) : 2 * (r & 7) - 10; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[2], uint32_t (&a)[16]) {
        const uint32_t t[2] = {w[0] >> 10, w[1] >> 10};
#pragma unroll
        for (int r = 0; r < 16; r++) a[r] = ((r & 7) < 5 ? w[r >> 3] : t[r >> 3]) & (0x00030003u << shift(r, 0));
    }
};

template <>
struct KUnpack<3> {  // byte-aligned sources from PRMT; code j sits at bit (3j mod 8) of its half
    static constexpr int kA = 7;
    static constexpr __host__ __device__ int dim(int r, int half) { return (r < 8 ? r : r + 8) + 8 * half; }
    static constexpr __host__ __device__ int shift(int r, int half) { return (3 * dim(r, half)) & 7; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[3], uint32_t (&a)[16]) {
        // sources (bytes of the 12-byte window in the low half | high half):
        // S0 (0,1 | 3,4): codes 0-2 | 8-10; S1 (1,2 | 4,5): 3-5 | 11-13;
        // S2 (2 | 5): 6-7 | 14-15; S3 (6,7 | 9,10): 16-18 | 24-26;
        // S4 (7,8 | 10,11): 19-21 | 27-29; S5 (8 | 11): 22-23 | 30-31
        const uint32_t S[6] = {prmt(w[0], w[1], 0x4310u), prmt(w[0], w[1], 0x5421u), prmt(w[0], w[1], 0x6532u),
                               prmt(w[1], w[2], 0x6532u), prmt(w[1], w[2], 0x7643u), prmt(w[2], w[2], 0x3310u)};
        constexpr int src[16] = {0, 0, 0, 1, 1, 1, 2, 2, 3, 3, 3, 4, 4, 4, 5, 5};
#pragma unroll
        for (int r = 0; r < 16; r++) a[r] = S[src[r]] & (0x00070007u << shift(r, 0));
    }
};

template <>
struct KUnpack<4> {  // word i: codes (8i + e, 8i + 4 + e); e = 0, 1 in place, e = 2, 3 after >> 8
    static constexpr int kA = 4;
    static constexpr __host__ __device__ int dim(int r, int half) { return 8 * (r >> 2) + (r & 3) + 4 * half; }
    static constexpr __host__ __device__ int shift(int r, int) { return (r & 1) ? 4 : 0; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[4], uint32_t (&a)[16]) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t t = w[i] >> 8;
            a[4 * i] = w[i] & 0x000F000Fu;
            a[4 * i + 1] = w[i] & 0x00F000F0u;
            a[4 * i + 2] = t & 0x000F000Fu;
            a[4 * i + 3] = t & 0x00F000F0u;
        }
    }
};

template <>
struct KUnpack<8> {  // bytes (2e, 2e+1) of word i zero-extended: codes (4i + 2e, 4i + 2e + 1)
    static constexpr int kA = 0;
    static constexpr __host__ __device__ int dim(int r, int half) { return 4 * (r >> 1) + 2 * (r & 1) + half; }
    static constexpr __host__ __device__ int shift(int, int) { return 0; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[8], uint32_t (&a)[16]) {
#pragma unroll
        for (int r = 0; r < 16; r++) a[r] = prmt(w[r >> 1], 0u, (r & 1) ? 0x4342u : 0x4140u);
    }
};

// QJL sign bits (1 bit per projection): pairs (r, r+16) shifted down to bit 0.
struct SignUnpack {
    static constexpr int kA = 0;
    static constexpr __host__ __device__ int dim(int r, int half) { return r + 16 * half; }
    static constexpr __host__ __device__ int shift(int, int) { return 0; }
    static __device__ __forceinline__ void run(const uint32_t (&w)[1], uint32_t (&a)[16]) {
#pragma unroll
        for (int r = 0; r < 16; r++) a[r] = (w[0] >> r) & 0x00010001u;
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

// Raw Q.K of tokens g and g+8 for head c (units of 2^(KU::kA - 24) code units).
template <typename KU, int NW, bool TWO = true>
__device__ __forceinline__ void qk_raw(const uint8_t *rec0, const uint8_t *rec1, const uint32_t (&bq)[16],
                                       float &raw0, float &raw1) {
    uint32_t w0[NW], w1[NW], a0[16], a1[16];
    lds_words(w0, rec0);
    lds_words(w1, rec1);
    KU::run(w0, a0);
    KU::run(w1, a1);
    if constexpr (TWO) {  // two chains for ILP
        float e[4] = {0.f, 0.f, 0.f, 0.f}, o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
            mma16816(e, a0[2 * kk], a1[2 * kk], a0[2 * kk + 1], a1[2 * kk + 1], bq[2 * kk], bq[2 * kk + 1]);
            mma16816(o, a0[2 * kk + 2], a1[2 * kk + 2], a0[2 * kk + 3], a1[2 * kk + 3], bq[2 * kk + 2],
                     bq[2 * kk + 3]);
        }
        raw0 = (e[0] + e[1]) + (o[0] + o[1]);
        raw1 = (e[2] + e[3]) + (o[2] + o[3]);
    } else {  // one chain: two adds less per tile row pair
        float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; kk++)
            mma16816(e, a0[2 * kk], a1[2 * kk], a0[2 * kk + 1], a1[2 * kk + 1], bq[2 * kk], bq[2 * kk + 1]);
        raw0 = e[0] + e[1];
        raw1 = e[2] + e[3];
    }
}

// Token pairs (head_dim 64): rows g, g+8 are virtual records (2 v, 2 v + 1);
// the E columns take q against all 128 virtual dims, the O columns q with the
// odd half negated (nmask = 0x80008000 on the lanes c >= 2 holding it), so
// that E + O and E - O are twice the even and odd tokens' raw Q.K.
template <typename KU, int NW>
__device__ __forceinline__ void qk_raw2(const uint8_t *rec0, const uint8_t *rec1, const uint32_t (&bq)[16],
                                        uint32_t nmask, float (&raw)[4]) {
    uint32_t w0[NW], w1[NW], a0[16], a1[16];
    lds_words(w0, rec0);
    lds_words(w1, rec1);
    KU::run(w0, a0);
    KU::run(w1, a1);
    float e[4] = {0.f, 0.f, 0.f, 0.f}, o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
        mma16816(e, a0[2 * kk], a1[2 * kk], a0[2 * kk + 1], a1[2 * kk + 1], bq[2 * kk], bq[2 * kk + 1]);
        mma16816(o, a0[2 * kk], a1[2 * kk], a0[2 * kk + 1], a1[2 * kk + 1], bq[2 * kk] ^ nmask,
                 bq[2 * kk + 1] ^ nmask);
    }
    raw[0] = e[0] + e[1];  // row g: E
    raw[1] = o[0] + o[1];  // row g: O
    raw[2] = e[2] + e[3];  // row g + 8: E
    raw[3] = o[2] + o[3];  // row g + 8: O
}

// B fragment (16 registers) of a natural-order fp16 vector slice: words q[0..15]
// hold dims 2i, 2i+1 of the thread's 32-dim slice; register r pairs dims
// KU::dim(r, 0) and KU::dim(r, 1), each scaled by 2^(kA - shift) (exact).
template <typename KU>
__device__ __forceinline__ void gather_b(const uint32_t (&q)[16], uint32_t (&b)[16]) {
#pragma unroll
    for (int r = 0; r < 16; r++) {
        const int d0 = KU::dim(r, 0), d1 = KU::dim(r, 1);
        const uint32_t sel = ((d0 & 1) ? 0x32u : 0x10u) | (((d1 & 1) ? 0x76u : 0x54u) << 8);
        b[r] = prmt(q[d0 >> 1], q[d1 >> 1], sel);
        if constexpr (KU::kA > 0) {
            const uint32_t f = half_pow2_bits(KU::kA - KU::shift(r, 0)) |
                               (half_pow2_bits(KU::kA - KU::shift(r, 1)) << 16);
            const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&b[r]),
                                      *reinterpret_cast<const __half2 *>(&f));
            b[r] = *reinterpret_cast<const uint32_t *>(&v);
        }
    }
}

// ------------------------------------------------------------------- values
// Window of the thread's 16 value codes (bits [16g VB, 16g VB + 16 VB) of the
// record) as little-endian words, for the 5- to 8-bit decoders.
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

// Per-thread constants of the value decoders.
struct VCtx {
    int off;                     // byte offset of the thread's window in token row 2c of a tile
    int sh;                      // funnel shift (0/16) or PRMT selector of the window
    uint32_t tab;                // shared address of this lane's column of the pair table
    PrmtTable pt;                // 4-bit codebook bytes
    const unsigned short *ctab;  // 5- to 8-bit codebook in shared memory
};

// Byte offset of pair-table entry F[POS .. POS + BITS) with entries 2^TS bytes
// apart (a multiply or a high multiply, both off the integer-logic pipe).
template <int POS, int BITS, int TS>
__device__ __forceinline__ uint32_t pair_off(uint32_t F) {
    const uint32_t f = F & (((1u << BITS) - 1u) << POS);
    if constexpr (POS <= TS) return f * (1u << (TS - POS));
    else return __umulhi(f, 1u << (32 - POS + TS));
}

// pair(): the A registers of one token pair (x = the row at p, y = the next
// row) for all eight m-tiles: ra[mt] for accumulator row g (dim(mt, 0)),
// rb[mt] for row g+8 (dim(mt, 1)); the low half of each register is token x.
template <int VB, int TS>
struct VDec {  // 5..8 bits: shared-memory codebook, codes (2mt, 2mt+1)
    static constexpr bool kLinear = false;
    static constexpr __host__ __device__ int dim(int mt, int r) { return 2 * mt + r; }
    template <int NW>
    static __device__ __forceinline__ uint32_t code(const uint32_t (&x)[NW], int j) {
        const int bit = VB * j, wi = bit >> 5, sh = bit & 31;
        const uint32_t v = (sh + VB <= 32) ? (x[wi] >> sh) : __funnelshift_r(x[wi], x[wi + 1], sh);
        return v & ((1u << VB) - 1u);
    }
    static __device__ __forceinline__ void pair(const uint8_t *p, int RV, const VCtx &cx, uint32_t (&ra)[8],
                                                uint32_t (&rb)[8]) {
        uint32_t x[VWin<VB>::NW], y[VWin<VB>::NW];
        VWin<VB>::load(p + cx.off, cx.sh, x);
        VWin<VB>::load(p + cx.off + RV, cx.sh, y);
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            ra[mt] = static_cast<uint32_t>(cx.ctab[code(x, 2 * mt)]) |
                     (static_cast<uint32_t>(cx.ctab[code(y, 2 * mt)]) << 16);
            rb[mt] = static_cast<uint32_t>(cx.ctab[code(x, 2 * mt + 1)]) |
                     (static_cast<uint32_t>(cx.ctab[code(y, 2 * mt + 1)]) << 16);
        }
    }
};

template <int TS>
struct VDec<1, TS> {  // code j at bit j (j < 10) or, after >> 10, bit j - 10: dims (mt, mt + 8)
    static constexpr bool kLinear = true;
    static constexpr __host__ __device__ int dim(int mt, int r) { return mt + 8 * r; }
    static constexpr __host__ __device__ int shift(int j) { return j < 10 ? j : j - 10; }
    static __device__ __forceinline__ void pair(const uint8_t *p, int RV, const VCtx &cx, uint32_t (&ra)[8],
                                                uint32_t (&rb)[8]) {
        const uint32_t wx = *reinterpret_cast<const uint32_t *>(p + cx.off);
        const uint32_t wy = *reinterpret_cast<const uint32_t *>(p + cx.off + RV);
        const uint32_t Z = prmt(wx, wy, static_cast<uint32_t>(cx.sh));  // x's 16 codes | y's 16 codes
        const uint32_t Z2 = Z >> 10;
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            ra[mt] = Z & (0x00010001u << mt);
            rb[mt] = (mt < 2 ? Z : Z2) & (0x00010001u << shift(mt + 8));
        }
    }
    // 2^(24 - s): the accumulator of code j holds the weighted bit sum times 2^(s - 24)
    static __device__ __forceinline__ float unscale(int mt, int r) {
        return __uint_as_float(static_cast<uint32_t>(127 + 24 - shift(dim(mt, r))) << 23);
    }
};

template <int TS>
struct VDec<2, TS> {  // pair table of 16 entries; E/O fields of 4 bits: dims (2mt, 2mt+1)
    static constexpr bool kLinear = false;
    static constexpr __host__ __device__ int dim(int mt, int r) { return 2 * mt + r; }
    static __device__ __forceinline__ uint32_t field(uint32_t F, int j) {
        switch (j) {
            case 0: return pair_off<0, 4, TS>(F);
            case 1: return pair_off<4, 4, TS>(F);
            case 2: return pair_off<8, 4, TS>(F);
            case 3: return pair_off<12, 4, TS>(F);
            case 4: return pair_off<16, 4, TS>(F);
            case 5: return pair_off<20, 4, TS>(F);
            case 6: return pair_off<24, 4, TS>(F);
            default: return pair_off<28, 4, TS>(F);
        }
    }
    static __device__ __forceinline__ void pair(const uint8_t *p, int RV, const VCtx &cx, uint32_t (&ra)[8],
                                                uint32_t (&rb)[8]) {
        const uint32_t wx = *reinterpret_cast<const uint32_t *>(p + cx.off);
        const uint32_t wy = *reinterpret_cast<const uint32_t *>(p + cx.off + RV);
        constexpr uint32_t M = 0x33333333u;
        const uint32_t E = (wx & M) | ((wy << 2) & ~M);  // field j: x_{2j} | y_{2j} << 2
        const uint32_t O = ((wx >> 2) & M) | (wy & ~M);  // field j: x_{2j+1} | y_{2j+1} << 2
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            ra[mt] = lds32(cx.tab + field(E, mt));
            rb[mt] = lds32(cx.tab + field(O, mt));
        }
    }
};

template <int TS>
struct VDec<3, TS> {  // pair table of 64 entries; E/O fields of 6 bits: dims (2mt, 2mt+1)
    static constexpr bool kLinear = false;
    static constexpr __host__ __device__ int dim(int mt, int r) { return 2 * mt + r; }
    static __device__ __forceinline__ uint32_t field(uint32_t F, int j) {
        switch (j) {
            case 0: return pair_off<0, 6, TS>(F);
            case 1: return pair_off<6, 6, TS>(F);
            case 2: return pair_off<12, 6, TS>(F);
            case 3: return pair_off<18, 6, TS>(F);
            default: return pair_off<24, 6, TS>(F);
        }
    }
    static __device__ __forceinline__ void pair(const uint8_t *p, int RV, const VCtx &cx, uint32_t (&ra)[8],
                                                uint32_t (&rb)[8]) {
        // the 48-bit window starts cx.sh bits into the word at p + cx.off
        const uint32_t *px = reinterpret_cast<const uint32_t *>(p + cx.off);
        const uint32_t *py = reinterpret_cast<const uint32_t *>(p + cx.off + RV);
        const uint32_t x0 = __funnelshift_r(px[0], px[1], cx.sh), y0 = __funnelshift_r(py[0], py[1], cx.sh);
        const uint32_t x1 = __funnelshift_r(x0, px[1] >> cx.sh, 30);  // codes 10..15
        const uint32_t y1 = __funnelshift_r(y0, py[1] >> cx.sh, 30);
        constexpr uint32_t M = 0x071C71C7u;  // 3-bit fields at 6j
        const uint32_t E0 = (x0 & M) | ((y0 << 3) & ~M), O0 = ((x0 >> 3) & M) | (y0 & ~M);
        const uint32_t E1 = (x1 & M) | ((y1 << 3) & ~M), O1 = ((x1 >> 3) & M) | (y1 & ~M);
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            ra[mt] = lds32(cx.tab + (mt < 5 ? field(E0, mt) : field(E1, mt - 5)));
            rb[mt] = lds32(cx.tab + (mt < 5 ? field(O0, mt) : field(O1, mt - 5)));
        }
    }
};

// Lookup of 4 codes given as selector nibbles [x_j, x_j', y_j, y_j'] (4-bit
// indices): half2(c[x_j], c[y_j]) and half2(c[x_j'], c[y_j']); two 8-entry
// tables chosen per byte by the nibble's bit 3.
__device__ __forceinline__ void lookup4(uint32_t sel, const PrmtTable &t, uint32_t &ra, uint32_t &rb) {
    const uint32_t s7 = sel & 0x7777u;
    const uint32_t hb = ((sel >> 1) & 0x4444u) | 0x3210u;
    const uint32_t pl = prmt(prmt(t.tl[0], t.tl[1], s7), prmt(t.tl[2], t.tl[3], s7), hb);
    const uint32_t ph = prmt(prmt(t.th[0], t.th[1], s7), prmt(t.th[2], t.th[3], s7), hb);
    ra = prmt(pl, ph, 0x6240u);
    rb = prmt(pl, ph, 0x7351u);
}

template <int TS>
struct VDec<4, TS> {  // nibbles; selector = byte k of both tokens: codes (2mt, 2mt+1)
    static constexpr bool kLinear = false;
    static constexpr __host__ __device__ int dim(int mt, int r) { return 2 * mt + r; }
    static __device__ __forceinline__ void pair(const uint8_t *p, int RV, const VCtx &cx, uint32_t (&ra)[8],
                                                uint32_t (&rb)[8]) {
        const uint2 x = *reinterpret_cast<const uint2 *>(p + cx.off);
        const uint2 y = *reinterpret_cast<const uint2 *>(p + cx.off + RV);
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
            const int k = mt & 3;
            const uint32_t sel = prmt(mt < 4 ? x.x : x.y, mt < 4 ? y.x : y.y, static_cast<uint32_t>(k | ((k + 4) << 4)));
            lookup4(sel, cx.pt, ra[mt], rb[mt]);
        }
    }
};

// ------------------------------------------------------------------- kernel
struct ValueTable {
    unsigned short half[256];  // fp16 codebook values of this class's value width and law
    float c1;                  // binary32 centroid 1 of a 1-bit codebook (= -centroid 0)
};

template <int KB, int VB, bool QJL, int NH = 1, int NP = 1>
struct PackedGeom {
    static constexpr int PT = packed_stage_tokens(KB, VB, QJL, NH, NP);  // tokens per stage, a multiple of 64
    static constexpr int CTAS = packed_ctas_per_sm(KB, VB, QJL, NH, NP);
    static constexpr int RK = 16 * KB * NH / NP, RV = 16 * VB * NH / NP;  // bytes of a token's key / value record
    static constexpr int RKR = RK * NP, RVR = RV * NP;  // bytes of a tile row (NP tokens)
    static constexpr int offV = PT * RK;
    static constexpr int offKS = offV + PT * RV;
    static constexpr int offVS = offKS + PT * 4;
    static constexpr int offQS = offVS + PT * 4;
    static constexpr int offQN = offQS + PT * 16;
    static constexpr int stage = QJL ? offQN + PT * 4 : offQS;
    static constexpr int budget = 227 * 1024 / CTAS - 1024;
    // flag, barriers (the rotated queries come from the prep kernel); NH > 1:
    // the raw-score exchange, two buffers of a float4 per thread
    static constexpr int xbytes = NH > 1 ? 2 * kThreads * 16 : 0;
    static constexpr int qbytes = 16 + 64 + xbytes;
    static constexpr int pair_entries = (VB == 2 || VB == 3) ? (1 << (2 * VB)) : 0;
    // pair table: one column per lane (32 copies) if that still leaves 3
    // stages in flight at the class's CTAs per SM, or as many as 16 copies
    // would; else 16 (2-way bank conflicts)
    static constexpr int fit32 = (budget - qbytes - pair_entries * 128) / stage;
    static constexpr int fit16 = (budget - qbytes - pair_entries * 64) / stage;
    static constexpr int copies = (pair_entries == 0 || fit32 >= 3 || fit32 >= fit16) ? 32 : 16;
    static constexpr int tab_bytes = pair_entries * copies * 4;
    static constexpr int TS = copies == 32 ? 7 : 6;  // log2 of the table's entry stride
    static constexpr int fixed = (VB >= 5 ? 512 : 0) + tab_bytes + qbytes;
    // as many stages in flight (2..4) as fit with the class's CTAs per SM
    static constexpr int fit = (budget - fixed) / stage;
    static constexpr int stages = fit > 4 ? 4 : (fit < 2 ? 2 : fit);
    static constexpr int ctab = stages * stage;               // fp16 codebook (5-8 bits)
    static constexpr int ptab = ctab + (VB >= 5 ? 512 : 0);   // pair table (2, 3 bits)
    static constexpr int qoff = ptab + tab_bytes;             // end of the tables
    static constexpr int flag = qoff;
    static constexpr int bar = flag + 16;                     // one mbarrier per stage buffer
    static constexpr int xch = (bar + 8 * stages + 15) & ~15;  // NH > 1: the exchange buffers
    static constexpr int smem = NH > 1 ? xch + xbytes : bar + 8 * stages;
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
    // stage s of the launch, in item `it` (the host's per-CTA table)
    __device__ __forceinline__ void locate(const WorkItem *items, int it, long long s) {
        item = it;
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
// stages in equal contiguous ranges and stream them through one bulk-copy
// pipeline that never drains at group boundaries.  Each warp writes one
// partial per (item, batch) group its CTA touches; the CTA completing a
// (layer, batch, KV head) merges the partials (finish_and_combine).
//
// NH > 1 (head_dim 128 NH): a token's key (value) record is NH consecutive
// 128-dim sub-records of 16 KB (16 VB) bytes, the LSB-first code stream cut at
// dims 128 j.  NH warps share each 32-token block: warp w scores and sums
// sub-record w mod NH with the 128-dim machinery, the NH warps add their raw
// Q.K partials through shared memory (a named barrier per block, the same
// order on every warp, so that all take identical softmax decisions), and
// each writes its sub-record's partial (record w mod NH of its group).
//
// NP = 2 (head_dim 64): a tile row is a token pair, read as one 128-dim
// record (qk_raw2, softmax_pair2, write_warp_partial_pair2, combine_np2).
template <int KB, int VB, bool QJL, int NH = 1, int NP = 1>
__global__ void __launch_bounds__(kThreads, packed_ctas_per_sm(KB, VB, QJL, NH, NP))
    decode_packed_kernel(const DecodeDims dims, const DecodeWorkspace ws, const int *__restrict__ cta_item,
                         const long long S, const __grid_constant__ ValueTable vt) {
    static_assert(NH == 1 || (!QJL && (NH == 2 || NH == 4)), "QJL sketches at head_dim 128 only");
    static_assert(NP == 1 || (!QJL && NH == 1 && NP == 2), "token pairs: head_dim 64, no QJL");
    using G = PackedGeom<KB, VB, QJL, NH, NP>;
    using KU = KUnpack<KB>;
    using VD = VDec<VB, G::TS>;
    constexpr int NS = G::stages;
    constexpr int kPT = G::PT;
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int sub = NH > 1 ? warp % NH : 0;  // the warp's 128-dim sub-record
    const int gqa = dims.gqa, B = dims.B;
    const long long s_begin = range_begin(blockIdx.x, S, gridDim.x);
    const int n_st = static_cast<int>(range_begin(blockIdx.x + 1, S, gridDim.x) - s_begin);
    pdl_launch_dependents();

    // ---- value decoder constants and tables
    VCtx vx;
    vx.ctab = reinterpret_cast<const unsigned short *>(smem + G::ctab);
    vx.tab = smem_u32(smem + G::ptab) + 4 * (lane & (G::copies - 1));
    if constexpr (VB == 1) {
        vx.off = 2 * c * G::RVR + 16 * VB * sub + 4 * (g >> 1);
        vx.sh = (g & 1) ? 0x7632 : 0x5410;  // PRMT: x's halfword g | y's halfword g
    } else if constexpr (VB == 3) {
        vx.off = 2 * c * G::RVR + 16 * VB * sub + 4 * ((3 * g) >> 1);
        vx.sh = (g & 1) * 16;
    } else {
        vx.off = 2 * c * G::RVR + 16 * VB * sub + ((2 * VB * g) & ~3);
        vx.sh = ((2 * VB * g) & 3) * 8;
    }
    if constexpr (VB >= 5) {
        unsigned short *ct = reinterpret_cast<unsigned short *>(smem + G::ctab);
        for (int i = threadIdx.x; i < (1 << VB); i += kThreads) ct[i] = vt.half[i];
    }
    if constexpr (G::pair_entries > 0) {
        uint32_t *pt = reinterpret_cast<uint32_t *>(smem + G::ptab);
        for (int i = threadIdx.x; i < G::pair_entries * G::copies; i += kThreads) {
            const int e = i / G::copies;
            pt[i] = static_cast<uint32_t>(vt.half[e & ((1 << VB) - 1)]) |
                    (static_cast<uint32_t>(vt.half[e >> VB]) << 16);
        }
    }
    if constexpr (VB == 4) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const uint32_t v = vt.half[4 * i + e];
                lo |= (v & 0xFFu) << (8 * e);
                hi |= (v >> 8) << (8 * e);
            }
            vx.pt.tl[i] = lo;
            vx.pt.th[i] = hi;
        }
    }

    // ---- loader (thread 0): stage k of this CTA's range into buffer k % NS by
    // TMA bulk copies completing on full[k % NS]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + G::bar);
    StageCursor<QJL, true> lc;
    if (threadIdx.x == 0) {
        lc.locate(ws.items, cta_item[blockIdx.x], s_begin);
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
        // token pairs: an odd count rounds up to 16 bytes inside the row
        const unsigned nk = NP == 1 ? n * G::RK : (n * G::RK + 15) & ~15u;
        const unsigned nv = NP == 1 ? n * G::RV : (n * G::RV + 15) & ~15u;
        const unsigned ns = (n * 4 + 15) & ~15u;
        const unsigned total = nk + nv + 2 * ns + (QJL ? n * 16 + ns : 0);
        fence_proxy_async();
        mbar_expect_tx(bar, total);
        // the cache streams through L2 once: evict it first
        const uint64_t pol = policy_evict_first();
        bulk_g2s_hint(dst, lc.kc + static_cast<size_t>(t0) * G::RK, nk, bar, pol);
        bulk_g2s_hint(dst + G::offV, lc.vc + static_cast<size_t>(t0) * G::RV, nv, bar, pol);
        bulk_g2s_hint(dst + G::offKS, lc.ks + t0, ns, bar, pol);
        bulk_g2s_hint(dst + G::offVS, lc.vs + t0, ns, bar, pol);
        if constexpr (QJL) {
            bulk_g2s_hint(dst + G::offQS, lc.qs + static_cast<size_t>(t0) * 16, n * 16, bar, pol);
            bulk_g2s_hint(dst + G::offQN, lc.qn + t0, ns, bar, pol);
        }
        // rebind only if another stage follows in this CTA's range
        lc.advance(ws.items, B, --loads_left > 0);
    };
    if (threadIdx.x == 0) {
        for (int k = 0; k < NS - 1 && k < n_st; k++) load_next(k);
    }
    pdl_wait();  // the prep kernel's rotated queries (its grid precedes every packed class)

    // ---- consumer
    StageCursor<QJL, false> cc;
    cc.locate(ws.items, cta_item[blockIdx.x], s_begin);
    int g_layer = 0, g_head = 0, g_b = 0;
    int g_slot = 0;  // the warp's partial-record slot of the group
    uint32_t bq[16], bt[16];
    float qsum = 0.f, tsum = 0.f, aq = 0.f;
    // classes with the 168-register budget (3 CTAs per SM) fold the score
    // scale into the group's constants (aq and beta qsum times the scale), one
    // multiply less per score, and sum Q.K in one mma chain (two adds less per
    // pair of tile rows); the 128-register classes keep both apart (their
    // registers spill otherwise)
    constexpr bool kFoldScale = G::CTAS == 3;
    float aqs = 0.f, bqs = 0.f;
    WarpState st;
    int *flag = reinterpret_cast<int *>(smem + G::flag);
    // raw = (q / 2^e) . code * 2^(kA - 24) and q . yhat = m (alpha q.code + beta sum q)
    constexpr float alphaA = static_cast<float>(1 << (24 - KU::kA)) * 2.0f / static_cast<float>(1 << KB);
    constexpr float beta = 1.0f / static_cast<float>(1 << KB) - 1.0f;
    const float qk_scale = dims.qk_scale;
    const float c1 = vt.c1;
    // byte offset of the thread's key window: codes [32c, 32c+32) of token row
    // g's sub-record
    const int koff = g * G::RKR + 16 * KB * sub + 4 * KB * c;
    const uint32_t nmask = (NP == 2 && c >= 2) ? 0x80008000u : 0u;  // token pairs: the odd half's sign

    int xpar = 0;  // exchange buffer of the warp's next block (NH > 1)
    // spilled: the warp's record of the current group holds an earlier part of
    // it, relative to the max m_ref (of head c, on lane c)
    bool spilled = false;
    float m_ref = 0.f;
    // the warp's state into its record slot of the current group: written at
    // the group's first spill or flush, folded in at later ones
    auto write_record = [&]() {
        auto dim_of = [g](int mt, int r) { return 16 * g + VD::dim(mt, r); };
        auto fin = [c1](int mt, int r, float acc, float W) {
            if constexpr (VD::kLinear) return c1 * (2.0f * acc * VDec<1, 7>::unscale(mt, r) - W);
            else return acc;
        };
        float *rec = ws.part + static_cast<size_t>(g_slot) * (kMaxGqa * kPartStride);
        const float dm = st.m - m_ref;
        if (!spilled) {
            if constexpr (NP == 2) write_warp_partial_pair2(st, rec, gqa, dim_of, fin);
            else write_warp_partial_pair(st, rec, gqa, dim_of, fin);
        } else if (__any_sync(0xffffffffu, c < gqa && !(dm <= 64.f))) {
            merge_warp_partial<NP, VD>(st, rec, gqa, fin);
        } else {
            fold_warp_partial<NP, VD>(st, rec, gqa, fin, ex2(dm));
            return;
        }
        m_ref = st.m;
    };
    // a new group: its identity and the B fragments of its rotated queries
    // (column g: head g/2, part g&1), each head divided by a power of two 2^e
    // that brings its largest coordinate into [0.5, 1)
    auto start_group = [&]() {
        const WorkItem &it = ws.items[cc.item];
        g_b = cc.b;
        g_layer = it.layer;
        g_head = it.head;
        // the group's CTAs write consecutive slots of kDecodeWarps, by CTA
        const long long stage0 = it.stage_begin + static_cast<long long>(cc.b) * it.n_stages;
        g_slot = ws.grp_part[static_cast<long long>(cc.item) * B + cc.b] +
                 kDecodeWarps * static_cast<int>(blockIdx.x - cta_of_stage(stage0, S, gridDim.x)) + warp;
        init_state(st);
        spilled = false;
        const size_t qbase = (static_cast<size_t>(g_layer) * B + g_b) * dims.Hq + g_head * gqa;
        const int head = g >> 1, part = g & 1;
        uint32_t q[16];
        if constexpr (QJL) {
            const uint32_t *qw = ws.qrot + ((qbase + head) * 2 + part) * (kD / 2) + 16 * c;
#pragma unroll
            for (int i = 0; i < 16; i++) q[i] = head < gqa ? qw[i] : 0u;
            gather_b<KU>(q, bq);
            const uint32_t *tw = ws.qjlt + ((qbase + head) * 2 + part) * (kD / 2) + 16 * c;
#pragma unroll
            for (int i = 0; i < 16; i++) q[i] = head < gqa ? tw[i] : 0u;
            gather_b<SignUnpack>(q, bt);
            qsum = c < gqa ? ws.qsum[(qbase + c) * 4] : 0.f;
            tsum = c < gqa ? ws.qsum[(qbase + c) * 4 + 1] : 0.f;
            aq = c < gqa ? alphaA * ws.qsum[(qbase + c) * 4 + 2] : 0.f;
        } else if constexpr (NP == 2) {  // 64 dims: lanes c and c + 2 take the same 32
            const uint32_t *qw = ws.qrot + ((qbase + head) * 2 + part) * (kD / 4) + 16 * (c & 1);
#pragma unroll
            for (int i = 0; i < 16; i++) q[i] = head < gqa ? qw[i] : 0u;
            gather_b<KU>(q, bq);
            qsum = c < gqa ? ws.qsum[(qbase + c) * 4] : 0.f;
            aq = c < gqa ? alphaA * ws.qsum[(qbase + c) * 4 + 2] : 0.f;
        } else {  // the prep kernel rotated the queries
            const uint32_t *qw = ws.qrot + ((qbase + head) * 2 + part) * (NH * kD / 2) + 64 * sub + 16 * c;
#pragma unroll
            for (int i = 0; i < 16; i++) q[i] = head < gqa ? qw[i] : 0u;
            gather_b<KU>(q, bq);
            qsum = c < gqa ? ws.qsum[(qbase + c) * 4] : 0.f;
            aq = c < gqa ? alphaA * ws.qsum[(qbase + c) * 4 + 2] : 0.f;
        }
        if constexpr (kFoldScale) {
            aqs = aq * qk_scale;
            bqs = beta * qsum * qk_scale;
        }
    };
    // the warp's two 16-token tiles: tokens [tA, tA + 32) of the stage buffer
    auto tiles = [&](const uint8_t *buf, int tA, int n, auto full_tag) {
        constexpr bool FULL = decltype(full_tag)::value;
        const float *kss = reinterpret_cast<const float *>(buf + G::offKS);
        const float *vss = reinterpret_cast<const float *>(buf + G::offVS);
        uint32_t bp[4];
        if constexpr (NP == 2) {
            // virtual rows tA + 16 t + g (+ 8): tokens 2 row, 2 row + 1
            float s8[8], vs8[8];
            bool ok8[8];
            const float ha = 0.5f * aq;
#pragma unroll
            for (int t = 0; t < 2; t++) {
                const int t0 = tA + 16 * t, r0 = t0 + g;
                float raw[4];
                qk_raw2<KU, KB>(buf + t0 * G::RKR + koff, buf + (t0 + 8) * G::RKR + koff, bq, nmask, raw);
#pragma unroll
                for (int r = 0; r < 2; r++) {
                    const float E = raw[2 * r], O = raw[2 * r + 1];
#pragma unroll
                    for (int par = 0; par < 2; par++) {
                        const int tok = 2 * (r0 + 8 * r) + par;
                        const int i = 4 * t + 2 * r + par;
                        s8[i] = kss[tok] * (ha * (par ? E - O : E + O) + beta * qsum) * qk_scale;
                        ok8[i] = FULL || tok < n;
                        vs8[i] = vss[tok];
                    }
                }
            }
            softmax_pair2<FULL, VD::kLinear>(st, s8, ok8, vs8, g, c, bp);
        } else {
        float sc[4];
        if constexpr (NH > 1) {
            // this sub-record's raw Q.K of tokens g, g+8 of both tiles, summed
            // over the NH sub-records in the order 0..NH-1 by every warp
            float r[4];
            qk_raw<KU, KB, !kFoldScale>(buf + tA * G::RK + koff, buf + (tA + 8) * G::RK + koff, bq, r[0], r[1]);
            qk_raw<KU, KB, !kFoldScale>(buf + (tA + 16) * G::RK + koff, buf + (tA + 24) * G::RK + koff, bq, r[2],
                                        r[3]);
            float4 *xb = reinterpret_cast<float4 *>(smem + G::xch) + xpar * kThreads + (warp - sub) * 32 + lane;
            xb[sub * 32] = make_float4(r[0], r[1], r[2], r[3]);
            named_barrier(1 + warp / NH, 32 * NH);
            float4 a = xb[0];
#pragma unroll
            for (int j = 1; j < NH; j++) {
                const float4 o = xb[32 * j];
                a.x += o.x;
                a.y += o.y;
                a.z += o.z;
                a.w += o.w;
            }
            xpar ^= 1;
            const float raw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int t = 0; t < 2; t++) {
                const int t0 = tA + 16 * t;
                if constexpr (kFoldScale) {
                    sc[2 * t] = kss[t0 + g] * (aqs * raw[2 * t] + bqs);
                    sc[2 * t + 1] = kss[t0 + g + 8] * (aqs * raw[2 * t + 1] + bqs);
                } else {
                    sc[2 * t] = kss[t0 + g] * (aq * raw[2 * t] + beta * qsum) * qk_scale;
                    sc[2 * t + 1] = kss[t0 + g + 8] * (aq * raw[2 * t + 1] + beta * qsum) * qk_scale;
                }
            }
        } else {
#pragma unroll
        for (int t = 0; t < 2; t++) {
            const int t0 = tA + 16 * t;
            float raw0, raw1;
            qk_raw<KU, KB, !kFoldScale>(buf + t0 * G::RK + koff, buf + (t0 + 8) * G::RK + koff, bq, raw0, raw1);
            float s0, s1;
            if constexpr (kFoldScale) {
                s0 = kss[t0 + g] * (aqs * raw0 + bqs);
                s1 = kss[t0 + g + 8] * (aqs * raw1 + bqs);
            } else {
                s0 = kss[t0 + g] * (aq * raw0 + beta * qsum);
                s1 = kss[t0 + g + 8] * (aq * raw1 + beta * qsum);
            }
            if constexpr (QJL) {
                const float *qns = reinterpret_cast<const float *>(buf + G::offQN);
                float r0, r1;
                qk_raw<SignUnpack, 1>(buf + G::offQS + (t0 + g) * 16 + 4 * c,
                                      buf + G::offQS + (t0 + g + 8) * 16 + 4 * c, bt, r0, r1);
                constexpr float gam = 1.2533141373155003f / kJl;  // sqrt(pi/2) / jl
                const float gqs = kFoldScale ? gam * qk_scale : gam;
                s0 += gqs * qns[t0 + g] * (33554432.0f * r0 - tsum);
                s1 += gqs * qns[t0 + g + 8] * (33554432.0f * r1 - tsum);
            }
            sc[2 * t] = kFoldScale ? s0 : s0 * qk_scale;
            sc[2 * t + 1] = kFoldScale ? s1 : s1 * qk_scale;
        }
        }
        bool okv[4];
        if constexpr (FULL) {
            okv[0] = okv[1] = okv[2] = okv[3] = true;
        } else {
            okv[0] = tA + g < n;
            okv[1] = tA + g + 8 < n;
            okv[2] = tA + 16 + g < n;
            okv[3] = tA + 24 + g < n;
        }
        const float vsv[4] = {vss[tA + g], vss[tA + g + 8], vss[tA + 16 + g], vss[tA + 24 + g]};
        softmax_pair<FULL, VD::kLinear>(st, sc, okv, vsv, g, c, bp);
        }
        // ---- values of both tiles (rows: tokens, or token pairs for NP = 2)
        const uint8_t *vst = buf + G::offV;
        const int nrows = NP == 1 ? n : (n + 1) / 2;
#pragma unroll
        for (int t = 0; t < 2; t++) {
            if (!FULL && t == 1 && tA + 16 >= nrows) break;
            const uint8_t *vrow = vst + (tA + 16 * t) * G::RVR;
            uint32_t ra[8], rb[8], rc[8], rd[8];
            VD::pair(vrow, G::RVR, vx, ra, rb);               // rows 2c, 2c+1
            VD::pair(vrow + 8 * G::RVR, G::RVR, vx, rc, rd);  // rows 2c+8, 2c+9
#pragma unroll
            for (int mt = 0; mt < 8; mt++)
                mma16816(st.acc[mt], ra[mt], rb[mt], rc[mt], rd[mt], bp[2 * t], bp[2 * t + 1]);
        }
    };
    __syncthreads();  // codebook and pair table written
    start_group();
    bool new_group = false;
    // stages between spills (a power of two): a warp accumulates 16-token
    // tiles at kPT NH / (16 NP kDecodeWarps) per stage, 64 between spills
    constexpr int kSpill = (64 * 16 * NP * kDecodeWarps) / (kPT * NH) > 0 ? (64 * 16 * NP * kDecodeWarps) / (kPT * NH) : 1;
    static_assert((kSpill & (kSpill - 1)) == 0, "spill cadence: a power of two");

    // one pass per stage, and a last one (k = n_st) for the final merge
    for (int k = 0;; k++) {
        const bool last = k == n_st;
        if (!last) {
            const bool arrived = mbar_wait(&full[k % NS], (k / NS) & 1, dims.wait_polls);
            // all warps are past stage k-1 (its buffer is free) and agree on errors
            if (__syncthreads_or(!arrived)) {
                if (threadIdx.x == 0) {
                    atomicExch(ws.error, 1);
                    // let the copies still in flight land before the CTA's shared
                    // memory goes away (always with the full bound)
                    for (int j = k; j < n_st && j < k + NS - 1; j++) mbar_wait(&full[j % NS], (j / NS) & 1);
                }
                __syncthreads();
                return;
            }
            if (threadIdx.x == 0 && k + NS - 1 < n_st) load_next(k + NS - 1);
        } else {
            // every thread waits for the previous grid of the call before its
            // last merge, so that this grid's completion implies that of all
            // earlier ones
            pdl_wait();
        }
        // the one place where the warps' states leave their registers: at the
        // end of a group or of the range (flush), and every kSpill stages of
        // the range (~64 tiles of each warp) for the group in progress (spill).
        // CTAs spill at staggered stages, so that the folds of all CTAs do not
        // meet in L2 at once.  (Rare: marked unlikely, so that this code stays
        // off the loop's straight path.)
        const bool spill_due = k > 0 && ((k - 1 + static_cast<int>(blockIdx.x)) & (kSpill - 1)) == kSpill - 1;
        if (__builtin_expect(new_group || last || spill_due, 0)) {
            write_record();
            if (new_group || last) {
                finish_and_combine<NH, NP>(dims, ws, g_layer, g_b, g_head, flag);
                if (last) break;
                start_group();
            } else {
                restart_sums(st);
                spilled = true;
            }
        }
        const uint8_t *buf = smem + (k % NS) * G::stage;
        const int n = min(kPT, cc.n_tokens - cc.st * kPT);
        new_group = cc.advance(ws.items, B, k + 1 < n_st);
        // warp w takes tokens [32 w, 32 w + 32) of every 128 of the stage
        // (NH > 1: block w / NH of every 128 / NH, sub-record w mod NH; NP = 2:
        // rows of token pairs)
        const int nrows = NP == 1 ? n : (n + 1) / 2;
        for (int tA = (warp / NH) * 32; tA < nrows; tA += 32 * (kDecodeWarps / NH)) {
            if (NP * (tA + 32) <= n) tiles(buf, tA, n, std::true_type{});
            else tiles(buf, tA, n, std::false_type{});
        }
    }
}

template <int KB, int VB, bool QJL, int NH = 1, int NP = 1>
cudaError_t launch_packed(const DecodeDims &dims, const DecodeWorkspace &ws, const int *cta_item, int n_ctas,
                          long long n_stages, const unsigned short *value_half, float value_c1, cudaStream_t s,
                          bool pdl) {
    using G = PackedGeom<KB, VB, QJL, NH, NP>;
    static bool configured = false;
    if (!configured) {
        if (G::smem > 48 * 1024) {
            const cudaError_t e = cudaFuncSetAttribute(decode_packed_kernel<KB, VB, QJL, NH, NP>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, G::smem);
            if (e != cudaSuccess) return e;
        }
        configured = true;
    }
    ValueTable vt;
    for (int i = 0; i < 256; i++) vt.half[i] = i < (1 << VB) ? value_half[i] : 0;
    vt.c1 = value_c1;
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
    return cudaLaunchKernelEx(&cfg, decode_packed_kernel<KB, VB, QJL, NH, NP>, dims, ws, cta_item, n_stages, vt);
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

// head_dim 128 nh (nh = 2, 4) and head_dim 64 (token pairs), no QJL: one
// translation unit per key width instantiates every value width.
#define TQ_INSTANTIATE_WIDE_KB(KB)                                                                            \
    namespace tqk {                                                                                            \
    PackedLauncher packed_launcher_wide_kb##KB(int vb, int nh) {                                               \
        switch (vb * 8 + nh) {                                                                                 \
            case 10: return dec::launch_packed<KB, 1, false, 2>;                                               \
            case 12: return dec::launch_packed<KB, 1, false, 4>;                                               \
            case 18: return dec::launch_packed<KB, 2, false, 2>;                                               \
            case 20: return dec::launch_packed<KB, 2, false, 4>;                                               \
            case 26: return dec::launch_packed<KB, 3, false, 2>;                                               \
            case 28: return dec::launch_packed<KB, 3, false, 4>;                                               \
            case 34: return dec::launch_packed<KB, 4, false, 2>;                                               \
            case 36: return dec::launch_packed<KB, 4, false, 4>;                                               \
            case 42: return dec::launch_packed<KB, 5, false, 2>;                                               \
            case 44: return dec::launch_packed<KB, 5, false, 4>;                                               \
            case 50: return dec::launch_packed<KB, 6, false, 2>;                                               \
            case 52: return dec::launch_packed<KB, 6, false, 4>;                                               \
            case 58: return dec::launch_packed<KB, 7, false, 2>;                                               \
            case 60: return dec::launch_packed<KB, 7, false, 4>;                                               \
            case 66: return dec::launch_packed<KB, 8, false, 2>;                                               \
            case 68: return dec::launch_packed<KB, 8, false, 4>;                                               \
            default: return nullptr;                                                                           \
        }                                                                                                      \
    }                                                                                                          \
    PackedLauncher packed_launcher_narrow_kb##KB(int vb) {                                                     \
        switch (vb) {                                                                                          \
            case 1: return dec::launch_packed<KB, 1, false, 1, 2>;                                             \
            case 2: return dec::launch_packed<KB, 2, false, 1, 2>;                                             \
            case 3: return dec::launch_packed<KB, 3, false, 1, 2>;                                             \
            case 4: return dec::launch_packed<KB, 4, false, 1, 2>;                                             \
            case 5: return dec::launch_packed<KB, 5, false, 1, 2>;                                             \
            case 6: return dec::launch_packed<KB, 6, false, 1, 2>;                                             \
            case 7: return dec::launch_packed<KB, 7, false, 1, 2>;                                             \
            case 8: return dec::launch_packed<KB, 8, false, 1, 2>;                                             \
            default: return nullptr;                                                                           \
        }                                                                                                      \
    }                                                                                                          \
    }
