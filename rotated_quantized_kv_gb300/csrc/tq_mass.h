// tq_mass.h -- geometry shared by the host plan and the passes that rescore
// packed tokens after a decode call (attention mass, QJL on values).
#pragma once

namespace tqk {

// Tokens per CTA of the rescoring passes: each of its 4 warps takes a quarter
// in 16-token tiles, so that the per-CTA query preparation is amortised.
constexpr int kMassTokens = 4096;

}  // namespace tqk
