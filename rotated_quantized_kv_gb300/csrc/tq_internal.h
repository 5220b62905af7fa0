// tq_internal.h -- private declarations shared by the host code and the kernels
// of the rotated + quantized KV library.  Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/tq.h"

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
    float thr[kCbTotal];         // value thresholds, flat by bit width
};

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
    float *k_rot, *v_rot, *k_orig, *v_orig;
    float centroid[kCbTotal];
};

// ----------------------------------------------------------------- decode
// One entry per (layer, segment) of a decode call, stored in the workspace.
struct alignas(16) SegPlan {
    const uint8_t *kcodes, *vcodes;  // packed codes, or fp16 K / V for fp16 segments
    const float *kscale, *vscale;
    const uint8_t *qjl_signs;
    const float *qjl_norm;
    int kind;          // TQ_SEG_PACKED / TQ_SEG_FP16
    int layer;
    int n_tokens;
    int capacity;
    int chunk;         // tokens per CTA (multiple of 64)
    int n_chunks;
    int cta_begin;     // first CTA of this segment within its kind's launch
    int part_begin;    // first partial record of this segment
    int nq;
    uint32_t kblock, vblock;
    uint32_t koff[kMaxH], voff[kMaxH];
    uint8_t kbits[kMaxH], vbits[kMaxH];
    int8_t qrank[kMaxH];
};

struct LayerPlan {
    int seg_begin, seg_end;          // this layer's packed segments in the SegPlan array
    int f16_begin, f16_end;          // this layer's fp16 segments
    int has_qjl;
    uint32_t sign_bits[kD / 32];
};

struct DecodeDims {
    int L, B, H, Hq, gqa;
    int n_seg;
    int n_packed_ctas, n_fp16_ctas;  // CTAs of the two split-K kernels
    int n_parts;                      // partial records (one per CTA)
    float qk_scale;                   // log2(e) / sqrt(d)
    float inv_sqrt_d;                 // binary32(1/sqrt(d)) used by the rotations
};

// Workspace: [SegPlan x n_seg][LayerPlan x L][q prep][partials] (16-aligned parts).
struct DecodeWorkspace {
    SegPlan *seg;
    LayerPlan *layer;
    uint32_t *qrot;    // [L][B][Hq][2][d/2] half2 words: hi, lo of R q
    uint32_t *qorig;   // [L][B][Hq][2][d/2] half2 words: hi, lo of q
    uint32_t *qjlt;    // [L][B][Hq][2][d/2] half2 words: hi, lo of S R q
    float *qsum;       // [L][B][Hq][4]: sum(R q), sum(S R q)
    float *part;       // [n_parts][kMaxGqa][2 + d]: m (log2 units), l, acc
};

// Packed-kernel stage geometry: 64 tokens per stage, 16 per warp.
constexpr int kStageTokens = 64;
constexpr int kDecodeWarps = 4;
constexpr int kStages = 4;

size_t packed_stage_bytes(int kb_max, int vb_max, bool qjl);

// Records a CUDA error for tq_last_cuda_error() and returns TQ_ERR_CUDA.
tq_status record_cuda_error(cudaError_t e);

// Launchers (defined in the .cu files).  Return cudaGetLastError().
cudaError_t launch_compress(const CompressParams &p, cudaStream_t s);
cudaError_t launch_dequant(const DequantParams &p, cudaStream_t s);
cudaError_t launch_decode_kernels(const DecodeDims &dims, const DecodeWorkspace &ws, int n_packed_seg,
                                  int kb_max, int vb_max, bool any_qjl, const uint16_t *q,
                                  const float *S, const unsigned short *centroid_half, float *out,
                                  cudaStream_t s, cudaEvent_t ev_start, cudaEvent_t ev_stop);

}  // namespace tqk
