// tq_internal.h -- private declarations shared by the host code and the kernels
// of the rotated + quantized KV library.  Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/tq.h"
#include "tq_decode_geometry.h"

namespace tqk {

constexpr int kD = 128;          // head_dim the kernels implement
constexpr int kMaxH = TQ_MAX_HEADS;
constexpr int kMaxGqa = 4;       // query heads per KV head (MMA columns: 2 per head)
constexpr int kJl = 128;         // QJL sketch length the kernels implement

// Codebooks for 1..8 bits in one flat table: level k of b bits at kCbOff[b] + k,
// threshold k of b bits at kCbOff[b] + k as well (threshold table has one unused
// slot per width).  sum_{b=1..8} 2^b = 510 entries.
constexpr int kCbTotal = 510;
__host__ __device__ constexpr int cb_off(int bits) { return (1 << bits) - 2; }

struct Codebooks {
    float centroid[kCbTotal];
    float threshold[kCbTotal];
};

// ----------------------------------------------------------------- compress
struct CompressParams {
    const uint16_t *K, *V;
    int64_t sb, sh, st;          // element strides of K and V
    int B, H, T, t_begin, capacity;
    uint8_t *kcodes, *vcodes;
    float *kscale, *vscale;
    uint8_t *qjl_signs;
    float *qjl_norm;
    const float *S;              // jl x d (device) or nullptr
    int nq;
    uint32_t kblock, vblock;     // bytes per batch element (all heads, capacity tokens)
    uint32_t koff[kMaxH], voff[kMaxH];  // per-head byte offset inside a batch block
    uint8_t kbits[kMaxH], vbits[kMaxH];
    int8_t qrank[kMaxH];         // -1: no QJL
    uint32_t sign_bits[kD / 32];
    float inv_sqrt_d;            // binary32(1/sqrt(d))
    const float *Q;              // dense rotation (d x d, device, y = Q x) or nullptr: the SRHT of sign_bits
    uint8_t *vqjl_signs;         // value-residual sketches (heads with vrank >= 0)
    float *vqjl_norm;
    int nv;
    int8_t vrank[kMaxH];         // -1: no value sketch
    float thr[kCbTotal];         // value thresholds, flat by bit width
    float cent[kCbTotal];        // value centroids, flat by bit width (value sketches)
    int n_sel;                   // compress_kernel: the heads it compresses, sel[0..n_sel)
    uint8_t sel[kMaxH];
};

constexpr int kRowsBuckets = 1024;  // buckets of a value quotient: sign, exponent, one mantissa bit
constexpr int kRowsMaxD = 512;      // head_dim up to which the one-thread-per-slice compressor runs

// Keys or values of the heads of one bit width, one thread per 128-dim slice
// (tq_compress_rows*.cu): launches of an SRHT compression without QJL sketches
// at head_dim 128, 256 or 512.
struct RowsParams {
    const uint16_t *X;           // K or V, element (b, h, t, i) at b*sb + h*sh + t*st + i
    int64_t sb, sh, st;
    int B, H, T, t_begin, capacity;
    uint8_t *codes;              // kcodes or vcodes
    float *scale;                // kscale or vscale
    uint32_t block;              // bytes per batch element of the code buffer
    uint32_t off[kMaxH];         // per-head byte offset inside a batch block
    int n_heads;                 // heads of this launch (all of one width)
    uint8_t head[kMaxH];         // their indices
    int nh;                      // 128-dim slices per vector (head_dim / 128: 1, 2 or 4)
    int np;                      // tokens per thread (2 at head_dim 64, else 1)
    uint32_t in_mask[kRowsMaxD / 2];  // word i: the input sign bits of coordinates 2i (bit 15), 2i + 1 (bit 31)
    float out_scale[kRowsMaxD];  // coordinate i: -binary32(1/sqrt(d)) if D_i = -1, else +
    float thr[255];              // values: the width's thresholds, ascending
    // values of <= 3 bits: bucket b = (bit pattern of u) >> 22 holds k_base and
    // the bucket's one threshold t_c (+inf if none) as bits: code = k_base + [t_c < u].
    // 4 bits (bucket4_ok): bucket b = (bit pattern of u) >> 21 (sign, exponent,
    // two mantissa bits) holds k_base << 21 | t', t' the low 21 bits of the
    // bucket's one threshold, complemented in negative buckets (2^21 - 1 if
    // none): code = k_base + [t' < x], x the low 21 bits of u, complemented if
    // u < 0 (both share u's top 11 bits, so that this is [t_c < u])
    struct Bucket { uint32_t t, k; };
    union {
        Bucket bucket[kRowsBuckets];
        uint32_t bucket4[2 * kRowsBuckets];
    };
    int bucket4_ok;
};
cudaError_t launch_compress_rows(const RowsParams &p, int bits, bool values, cudaStream_t s);
cudaError_t launch_compress_rows_nh2(const RowsParams &p, int bits, bool values, cudaStream_t s);
cudaError_t launch_compress_rows_nh4(const RowsParams &p, int bits, bool values, cudaStream_t s);
cudaError_t launch_compress_rows_np2(const RowsParams &p, int bits, bool values, cudaStream_t s);

// ----------------------------------------------------------------- dequantize
struct DequantParams {
    int B, H, t_begin, n, capacity;
    const uint8_t *kcodes, *vcodes;
    const float *kscale, *vscale;
    uint32_t kblock, vblock;
    uint32_t koff[kMaxH], voff[kMaxH];
    uint8_t kbits[kMaxH], vbits[kMaxH];
    uint32_t sign_bits[kD / 32];
    float inv_sqrt_d;
    const float *Q;              // dense rotation or nullptr (SRHT)
    float *k_rot, *v_rot, *k_orig, *v_orig;
    float centroid[kCbTotal];
};

// ----------------------------------------------------------------- requantize
// Tier demotion: tokens [s_t0, s_t0 + dst.T) of a source packed segment,
// dequantized in the rotated space and compressed again into positions
// [dst.t_begin, dst.t_begin + dst.T) of the destination segment `dst` (whose K
// and V pointers are unused).
struct RequantParams {
    CompressParams dst;
    const uint8_t *skcodes, *svcodes;
    const float *skscale, *svscale;
    uint32_t skblock, svblock;
    uint32_t skoff[kMaxH], svoff[kMaxH];
    uint8_t skbits[kMaxH], svbits[kMaxH];
    int scapacity, s_t0;
    float centroid[kCbTotal];    // value centroids, flat by bit width
};

// ----------------------------------------------------------------- decode
// One work item per (layer, segment, KV head) of a decode call; its CTAs are
// (batch element, token chunk) pairs.  Stored in the workspace.
struct alignas(16) WorkItem {
    const uint8_t *kc, *vc;   // packed codes of (b=0, head, t=0); fp16 segments: K / V of (b=0, head, t=0)
    const float *ks, *vs;     // scales of (b=0, head, t=0) (packed)
    const uint8_t *qs;        // QJL sign records of (b=0, head's rank, t=0)
    const float *qn;          // QJL norms
    uint64_t kstride, vstride;  // bytes between batch elements
    uint32_t sstride;         // floats between batch elements in the scale arrays (H * cap)
    uint32_t qstride;         // records between batch elements in the QJL arrays (nq * cap)
    long long stage_begin;    // packed: first 64-token stage of (this item, b = 0) within its class launch
    int n_stages;             // packed: 64-token stages per batch element
    int kind;                 // TQ_SEG_PACKED / TQ_SEG_FP16
    int layer, head;
    int n_tokens;
    int chunk, n_chunks;      // fp16: tokens per CTA (multiple of 64) and CTAs per batch element
    int cta_begin;            // fp16: first CTA within its launch
    int kb, vb, qjl, vlaw;  // vlaw: value codebook law (host side only)
    float *mass;              // attention mass of (b=0, head, t=0), batch stride sstride; null: none
    int mass_cta_begin;       // first CTA of the item in the attention-mass launch
    const uint8_t *vqs;       // value-residual sketches of (b=0, head's rank, t=0); null: none
    const float *vqn;         // their norms
    uint32_t vqstride;        // records between batch elements (nv * cap)
    int vqjl_cta_begin;       // first CTA of the item in the value-sketch launch
};

struct LayerPlan {
    uint32_t sign_bits[TQ_MAX_HEAD_DIM / 32];  // the SRHT's sign bits (head_dim / 32 words used)
    const float *dense;                    // dense rotation (d x d, y = Q x) or nullptr: the SRHT
    int has_qjl;
    int has_vqjl;                          // some packed item of the layer sketches its values
    int qjl_mode;                          // TQ_QJL_UNBIASED / TQ_QJL_SIGN_PAIR
    int n_items[kMaxH];                    // items of each KV head
    int item[kMaxH][TQ_MAX_SEGMENTS];      // their indices in the WorkItem array
};

struct DecodeDims {
    int L, B, H, Hq, gqa;
    int any_qjl;         // QJL layers: the prep kernel writes S R q
    int any_prep;        // the prep kernel ran (QJL or dense-rotation layers read R q from it)
    float qk_scale;      // log2(e) / sqrt(d)
    float inv_sqrt_d;    // binary32(1/sqrt(d)) used by the rotations
    int wait_polls;      // polls of a split-K CTA's wait for its own copies before it gives up
    int nh;              // 128-dim sub-records per head vector (head_dim / 128: 1, 2 or 4)
    int np;              // tokens per 128-dim tile row (2 at head_dim 64, else 1)
};

// Workspace: [WorkItem x n][LayerPlan x L][group tables][counters][q prep]
// [partials] (256-aligned parts; everything before the q prep is uploaded by
// every call, counters as zeros).  A group is (item, batch element), index
// item * B + b; its partial records are grp_part[g] .. grp_part[g] + grp_nparts[g] - 1.
struct DecodeWorkspace {
    WorkItem *items;
    LayerPlan *layer;
    int *grp_part;     // [items * B]
    int *grp_nparts;   // [items * B]
    int *lbh_total;    // [L][B][H]: CTA portions of (layer, batch, KV head) over all its items
    int *counter;      // [L][B][H]: CTA portions of (layer, batch, KV head) finished so far
    int *error;        // set non-zero by a kernel that gave up waiting for its copies
    uint32_t *qrot;    // [L][B][Hq][2][d/2] half2 words: hi, lo of R q (QJL calls only)
    uint32_t *qjlt;    // [L][B][Hq][2][d/2] half2 words: hi, lo of S R q (QJL calls only)
    float *qsum;       // [L][B][Hq][4]: sum(R q), sum(S R q), 2^e of the stored R q / 2^e (QJL calls only)
    float *part;       // [parts][kMaxGqa][4 + d]: m (log2 units), l, pad, pad, acc
    float *ml;         // [L][B][Hq][2]: merged max (log2 units) and sum, or null (no mass, no value sketch)
    float *z;          // [L][B][Hq][d]: sum_t p_t rho_t s_t of the value sketches (null: none)
    const uint16_t *q; // the caller's queries, fp16 [L][B][Hq][d]
    float *out;        // the caller's output, [L][B][Hq][d]
    // per-CTA work item of each launch (host-computed, one load instead of a
    // search): the split-K classes' tables (each launch gets its own offset),
    // the attention-mass and the value-sketch launches'
    const int *cta_item;
    const int *mass_cta_item;
    const int *vqjl_cta_item;
};

// Stage geometry of the split-K kernels: the fp16 kernel takes 64 tokens per
// stage (16 per warp); the packed kernels take 128 or 256 per stage (each warp
// 32 tokens, two 16-token tiles, of every 128), see packed_stage_tokens.
constexpr int kStageTokens = 64;
constexpr int kDecodeWarps = 4;
constexpr int kStages = 4;

// A launch of the split-K kernel of one class over items [item_lo, item_hi).
// Packed classes run persistent CTAs over n_stages 128-token stages (n_ctas of
// them, each taking an equal contiguous range); fp16 runs one CTA per chunk.
struct ClassLaunch {
    int kb, vb, qjl;   // kb == 16: fp16 segments
    int law;           // value codebook law
    int item_lo, item_hi, n_ctas;
    long long n_stages;
    int cta_off;       // this launch's per-CTA item table within DecodeWorkspace::cta_item
};

typedef cudaError_t (*PackedLauncher)(const DecodeDims &, const DecodeWorkspace &, const int *cta_item,
                                      int n_ctas, long long n_stages, const unsigned short *value_half,
                                      float value_c1,
                                      cudaStream_t s, bool pdl);
PackedLauncher packed_launcher_kb1(int vb, bool qjl);
PackedLauncher packed_launcher_kb2(int vb, bool qjl);
PackedLauncher packed_launcher_kb3(int vb, bool qjl);
PackedLauncher packed_launcher_kb4(int vb, bool qjl);
PackedLauncher packed_launcher_kb5(int vb, bool qjl);
PackedLauncher packed_launcher_kb6(int vb, bool qjl);
PackedLauncher packed_launcher_kb7(int vb, bool qjl);
PackedLauncher packed_launcher_kb8(int vb, bool qjl);
// head_dim 128 nh (nh = 2, 4), no QJL: one launcher table per key width
PackedLauncher packed_launcher_wide_kb1(int vb, int nh);
PackedLauncher packed_launcher_wide_kb2(int vb, int nh);
PackedLauncher packed_launcher_wide_kb3(int vb, int nh);
PackedLauncher packed_launcher_wide_kb4(int vb, int nh);
PackedLauncher packed_launcher_wide_kb5(int vb, int nh);
PackedLauncher packed_launcher_wide_kb6(int vb, int nh);
PackedLauncher packed_launcher_wide_kb7(int vb, int nh);
PackedLauncher packed_launcher_wide_kb8(int vb, int nh);
// head_dim 64 (token pairs), no QJL
PackedLauncher packed_launcher_narrow_kb1(int vb);
PackedLauncher packed_launcher_narrow_kb2(int vb);
PackedLauncher packed_launcher_narrow_kb3(int vb);
PackedLauncher packed_launcher_narrow_kb4(int vb);
PackedLauncher packed_launcher_narrow_kb5(int vb);
PackedLauncher packed_launcher_narrow_kb6(int vb);
PackedLauncher packed_launcher_narrow_kb7(int vb);
PackedLauncher packed_launcher_narrow_kb8(int vb);

// ----------------------------------------------------------------- other head dims
// Compression, dequantization and decode attention for head dimensions other
// than kD (powers of two 16..1024; tq_generic.cu).  No QJL sketches, dense
// rotations or attention-mass outputs on this path.
constexpr int kMaxD = TQ_MAX_HEAD_DIM;

struct GenCompressParams {
    const uint16_t *K, *V;
    int64_t sb, sh, st;          // element strides of K and V
    int B, H, T, t_begin, capacity;
    uint8_t *kcodes, *vcodes;
    float *kscale, *vscale;
    uint32_t kblock, vblock;
    uint32_t koff[kMaxH], voff[kMaxH];
    uint8_t kbits[kMaxH], vbits[kMaxH];
    uint32_t sign_bits[kMaxD / 32];
    float inv_sqrt_d;
    float thr[kCbTotal];         // value thresholds, flat by bit width
};

struct GenDequantParams {
    int B, H, t_begin, n, capacity;
    const uint8_t *kcodes, *vcodes;
    const float *kscale, *vscale;
    uint32_t kblock, vblock;
    uint32_t koff[kMaxH], voff[kMaxH];
    uint8_t kbits[kMaxH], vbits[kMaxH];
    uint32_t sign_bits[kMaxD / 32];
    float inv_sqrt_d;
    float *k_rot, *v_rot, *k_orig, *v_orig;
    float centroid[kCbTotal];
};

struct GenDecodeParams {
    int L, B, H, Hq, gqa;
    float qk_scale;              // log2(e) / sqrt(d)
    float inv_sqrt_d;
    const WorkItem *items;       // one per (layer, segment, KV head) with tokens
    const LayerPlan *layer;      // each (layer, KV head)'s items
    const uint32_t *signs;       // [L][kMaxD / 32] sign bits of each layer's rotation
    const uint16_t *q;           // fp16 [L][B][Hq][d]
    float *out;                  // [L][B][Hq][d]
    float centroid[kCbTotal];    // value centroids, flat by bit width
};

cudaError_t launch_gen_compress(const GenCompressParams &p, int d, cudaStream_t s);
cudaError_t launch_gen_dequant(const GenDequantParams &p, int d, cudaStream_t s);
cudaError_t launch_gen_decode(const GenDecodeParams &p, int d, cudaStream_t s);

// Records a CUDA error for tq_last_cuda_error() and returns TQ_ERR_CUDA.
tq_status record_cuda_error(cudaError_t e);

// Device address of the static decode scratch array on the current device
// (tq_static.cu); looked up on the first use per device.
tq_status static_workspace(void **out);

// Launchers (defined in the .cu files).  Return cudaGetLastError().
cudaError_t launch_compress(const CompressParams &p, cudaStream_t s);
// Dense rotation (p.Q set, no QJL heads): the tensor-core kernel.  Returns
// cudaErrorInvalidValue when the input strides cannot be described to TMA.
cudaError_t launch_compress_dense(const CompressParams &p, cudaStream_t s);
cudaError_t read_compress_dense_error(int *flag);
cudaError_t clear_compress_dense_error();
cudaError_t launch_dequant(const DequantParams &p, cudaStream_t s);
cudaError_t launch_requantize(const RequantParams &p, cudaStream_t s);
cudaError_t launch_decode_kernels(const DecodeDims &dims, const DecodeWorkspace &ws, const ClassLaunch *classes,
                                  int n_classes, const float *S, const unsigned short *const *value_half,
                                  const float *value_c1,
                                  cudaStream_t s, cudaEvent_t ev_start, cudaEvent_t ev_stop, int *n_launched);

}  // namespace tqk
