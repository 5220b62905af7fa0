// tq_mass.h -- geometry shared by the host plan and the passes that rescore
// packed tokens after a decode call (attention mass, QJL on values).
#pragma once

#include <cuda_runtime.h>

namespace tqk {

// Tokens per CTA of the rescoring passes: each of its 4 warps takes a quarter
// in 16-token tiles, so that the per-CTA query preparation is amortised.
constexpr int kMassTokens = 4096;

// Each warp of a rescoring CTA stages 64-token steps of its records through two
// shared-memory buffers; one buffer holds the key records (16 kb bytes each),
// their scales, and for QJL or value-sketch items the 16-byte sign records and
// norms.  Host and kernels size it for the widest key width of the launch.
constexpr int kMassStep = 64;
constexpr int mass_stage_bytes(int max_kb, bool key_sketch, bool value_sketch) {
    return kMassStep * (16 * max_kb + 4 + (key_sketch ? 20 : 0) + (value_sketch ? 20 : 0));
}

struct DecodeDims;
struct DecodeWorkspace;

// Attention mass of every item with a mass pointer (n_ctas CTAs in all, each
// finding its item in the workspace's per-CTA table), after the decode kernels
// of the call; stage_bytes from mass_stage_bytes for the launch's items.
cudaError_t launch_attention_mass(const DecodeDims &dims, const DecodeWorkspace &ws, int n_ctas, int stage_bytes,
                                  cudaStream_t s);
// QJL on values: z of every item with a value sketch (n_ctas CTAs), then
// out += R (sqrt(pi/2)/jl S^T z) for the query heads of layers that have one.
cudaError_t launch_value_qjl(const DecodeDims &dims, const DecodeWorkspace &ws, int n_ctas, int stage_bytes,
                             const float *S, cudaStream_t s);

}  // namespace tqk
