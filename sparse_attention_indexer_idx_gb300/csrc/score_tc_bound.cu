// DoSA bound-scan instantiations of the tensor-core kernel (score_tc.cuh):
// 32 prepared vectors per query (R retained heads + the negative aggregate),
// 8 queries per tile over shared keys, one query per tile over per-row keys;
// shared bf16 keys with R <= 16 take the group layout (16 vectors per query and
// one block of the 8 aggregates: N = 144).
#include "score_tc.cuh"

namespace idx {

bool bound_group_layout(const idx_problem& p, int R) {
  return p.key_off == nullptr && p.k_dtype == IDX_BF16 && R <= 16;
}

cudaError_t launch_bound(const idx_problem& prep, const float* wfold, const float* coef, const float* tau,
                         const float* knorm, const uint32_t* seedbits, int64_t seed_stride, uint32_t* candbits,
                         int64_t cb_stride, int R, const int32_t* row_mask, cudaStream_t st) {
  TcArgs a{};
  a.p = prep;
  a.wfold = wfold;
  a.coef = coef;
  a.tau = tau;
  a.knorm = knorm;
  a.seedbits = seedbits;
  a.seed_stride = seed_stride;
  a.candbits = candbits;
  a.cb_stride = cb_stride;
  a.R = R;
  a.row_mask = row_mask;
  const bool shared = prep.key_off == nullptr;
  if (shared && !knorm) return cudaErrorInvalidValue;
  if (prep.k_dtype == IDX_FP8_E4M3)
    return shared ? launch_tc<TcCfg<IDX_FP8_E4M3, 32, 4, kBound>>(a, st)
                  : launch_tc<TcCfg<IDX_FP8_E4M3, 32, 1, kBound>>(a, st);
  if (!shared) return launch_tc<TcCfg<IDX_BF16, 32, 1, kBound>>(a, st);
  return bound_group_layout(prep, R) ? launch_tc<TcCfg<IDX_BF16, 16, 8, kBound>>(a, st)
                                     : launch_tc<TcCfg<IDX_BF16, 32, 8, kBound>>(a, st);
}

}  // namespace idx
