// Gathered-key instantiations of the tensor-core score kernel (score_tc.cuh):
// exact scores of per-row key lists, one row per group (N = H), the same MMA
// shape per (query, key) pair as the dense per-row instantiation.
#include "score_tc.cuh"

namespace idx {

template <int KDT>
static cudaError_t gather_for(const TcArgs& a, cudaStream_t st) {
  switch (a.p.H) {
    case 16: return launch_tc<TcCfg<KDT, 16, 1, kGather>>(a, st);
    case 32: return launch_tc<TcCfg<KDT, 32, 1, kGather>>(a, st);
    case 64: return launch_tc<TcCfg<KDT, 64, 1, kGather>>(a, st);
    case 128: return launch_tc<TcCfg<KDT, 128, 1, kGather>>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_score_gather(const idx_problem& p, const int32_t* list, const int32_t* cnt, int64_t gld,
                                float* scores, int64_t ld, const int32_t* row_mask, cudaStream_t st) {
  TcArgs a{};
  a.p = p;
  a.scores = scores;
  a.ld = ld;
  a.list = list;
  a.cnt = cnt;
  a.gld = gld;
  a.row_mask = row_mask;
  return p.k_dtype == IDX_FP8_E4M3 ? gather_for<IDX_FP8_E4M3>(a, st) : gather_for<IDX_BF16>(a, st);
}

}  // namespace idx
