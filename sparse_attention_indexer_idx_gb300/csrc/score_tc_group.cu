// Shared-candidate-stream instantiations of the tensor-core score kernel
// (score_tc.cuh, kGroup): four consecutive queries over one key sequence score
// one list of keys together (N = 4 x H for bf16 keys, 4 x 2H for FP8), with
// the same MMA shape and epilogue chain per (query, key) pair as every other
// instantiation, and keep (id, score) per query when the score reaches tau.
#include "score_tc.cuh"

namespace idx {

bool group_stream_supported(const idx_problem& p) {
  if (p.key_off != nullptr || !score_uses_tensor_cores(p)) return false;
  if (p.k_dtype == IDX_FP8_E4M3) return p.H == 16 || p.H == 32;
  return p.H == 16 || p.H == 32 || p.H == 64;
}

cudaError_t launch_score_group(const idx_problem& p, const int32_t* list, const int32_t* cnt, int64_t gld,
                               const uint32_t* seedbits, int64_t seed_stride, const float* tau, int32_t* status,
                               int32_t* out_ids, float* out_sc, int32_t* out_cnt, int64_t out_ld, int64_t cap,
                               cudaStream_t st) {
  TcArgs a{};
  a.p = p;
  a.list = list;
  a.cnt = cnt;
  a.gld = gld;
  a.seedbits = seedbits;
  a.seed_stride = seed_stride;
  a.tau = tau;
  a.status = status;
  a.cand = out_ids;
  a.cand_sc = out_sc;
  a.cand_cnt = out_cnt;
  a.cand_ld = out_ld;
  a.cap = cap;
  if (!group_stream_supported(p)) return cudaErrorInvalidValue;
  if (p.k_dtype == IDX_FP8_E4M3) {
    return p.H == 16 ? launch_tc<TcCfg<IDX_FP8_E4M3, 16, 4, kGroup>>(a, st)
                     : launch_tc<TcCfg<IDX_FP8_E4M3, 32, 4, kGroup>>(a, st);
  }
  switch (p.H) {
    case 16: return launch_tc<TcCfg<IDX_BF16, 16, 4, kGroup>>(a, st);
    case 32: return launch_tc<TcCfg<IDX_BF16, 32, 4, kGroup>>(a, st);
    default: return launch_tc<TcCfg<IDX_BF16, 64, 4, kGroup>>(a, st);
  }
}

}  // namespace idx
