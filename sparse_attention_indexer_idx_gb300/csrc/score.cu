// Dispatch of the indexer score to its kernel family.  The choice depends only
// on (dtype pair, H, D), so every path that scores a (query, key) pair exactly
// -- dense, seed, survivor -- lands on the same arithmetic.
#include "internal.h"

namespace idx {

constexpr bool kTensorScoreEnabled = true;

bool score_uses_tensor_cores(const idx_problem& p) {
  const bool dt = p.q_dtype == IDX_BF16 && (p.k_dtype == IDX_BF16 || p.k_dtype == IDX_FP8_E4M3);
  const bool hs = p.H == 16 || p.H == 32 || p.H == 64 || p.H == 128;
  return dt && hs && p.D == 128 && kTensorScoreEnabled;
}

cudaError_t launch_score(const idx_problem& p, float* scores, int64_t ld, cudaStream_t st, const int32_t* row_mask) {
  if (score_uses_tensor_cores(p)) return launch_score_tc(p, scores, ld, row_mask, st);
  return launch_score_simt(p, scores, ld, row_mask, st);
}

}  // namespace idx
