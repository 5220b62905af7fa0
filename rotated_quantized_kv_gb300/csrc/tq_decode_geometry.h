// tq_decode_geometry.h -- stage geometry of the packed split-K decode classes
// (shared by the host planner and the kernels).
#pragma once

#include <cuda_runtime.h>

namespace tqk {

// Stage geometry of a packed split-K class, chosen by the bytes a token-head
// carries.  Light classes (<= 144 B: K4V4 and narrower at head_dim 128) do
// little work per token, so the per-stage costs (the CTA barrier, the copy
// issue, the cursor) weigh more: they run 256-token stages (512 at <= 64 B:
// K2V1, K1V2, ...) at 3 resident CTAs per SM.  Heavier classes run 128-token
// stages at 4 CTAs per SM, except with QJL sketches, whose operands take more
// registers (3 CTAs per SM).  Registers and shared memory of each
// instantiation are sized for its CTAs per SM.
//
// nh: 128-dim sub-records per record (head_dim = 128 nh).  With nh > 1 the
// warps of a CTA split each 32-token block by sub-record, so a warp holds the
// registers of one 128-dim slice and the class runs at 3 CTAs per SM; token
// records above 284 B (8-bit keys and values at head_dim 256) take 64-token
// stages so that two stages still fit.
__host__ __device__ constexpr int packed_token_bytes(int kb, int vb, bool qjl, int nh = 1) {
    return 16 * nh * (kb + vb) + 8 + (qjl ? 20 : 0);
}
__host__ __device__ constexpr bool packed_light(int kb, int vb, bool qjl, int nh = 1) {
    return packed_token_bytes(kb, vb, qjl, nh) <= 144;
}
//
// np = 2 (head_dim 64): a tile row is a pair of tokens read as one 128-dim
// record, so a stage holds twice the tokens of the 128-dim class of the same
// widths (the same bytes), at 3 CTAs per SM.
__host__ __device__ constexpr int packed_stage_tokens(int kb, int vb, bool qjl, int nh = 1, int np = 1) {
    return np > 1                                       ? np * packed_stage_tokens(kb, vb, qjl, 1, 1)
           : packed_token_bytes(kb, vb, qjl, nh) <= 64  ? 512
           : packed_light(kb, vb, qjl, nh)              ? 256
           : packed_token_bytes(kb, vb, qjl, nh) <= 284 ? 128
                                                        : 64;
}
__host__ __device__ constexpr int packed_ctas_per_sm(int kb, int vb, bool qjl, int nh = 1, int np = 1) {
    return (np > 1 || nh > 1 || qjl || packed_light(kb, vb, qjl, nh)) ? 3 : 4;
}

}  // namespace tqk
