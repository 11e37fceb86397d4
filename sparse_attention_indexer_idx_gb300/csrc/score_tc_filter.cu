// bf16-key kFilter instantiations of the tensor-core score kernel (score_tc.cuh):
// the dense score of every visible key, kept as (id, score) only when it
// reaches the row's threshold.  One query per group.
#include "score_tc.cuh"

namespace idx {

cudaError_t launch_score_filter_fp8(const TcArgs& a, cudaStream_t st);

cudaError_t launch_score_filter(const idx_problem& p, const float* tau, int32_t* cand, float* cand_sc,
                                int32_t* cand_cnt, int64_t cap, int32_t* status, const int32_t* row_mask,
                                cudaStream_t st) {
  TcArgs a{};
  a.p = p;
  a.tau = tau;
  a.cand = cand;
  a.cand_sc = cand_sc;
  a.cand_cnt = cand_cnt;
  a.cap = cap;
  a.status = status;
  a.row_mask = row_mask;
  if (p.k_dtype == IDX_FP8_E4M3) return launch_score_filter_fp8(a, st);
  switch (p.H) {
    case 16: return launch_tc<TcCfg<IDX_BF16, 16, 1, kFilter>>(a, st);
    case 32: return launch_tc<TcCfg<IDX_BF16, 32, 1, kFilter>>(a, st);
    case 64: return launch_tc<TcCfg<IDX_BF16, 64, 1, kFilter>>(a, st);
    case 128: return launch_tc<TcCfg<IDX_BF16, 128, 1, kFilter>>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace idx
