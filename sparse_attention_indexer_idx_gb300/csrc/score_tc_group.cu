// Shared-candidate-stream instantiations of the tensor-core score kernel
// (score_tc.cuh, kGroup): four consecutive queries over one key sequence score
// one list of keys together (N = 4 x H for bf16 keys, 4 x 2H for FP8), with
// the same MMA shape and epilogue chain per (query, key) pair as every other
// instantiation; scores are written by list position.
#include "score_tc.cuh"

namespace idx {

bool group_stream_supported(const idx_problem& p) {
  if (p.key_off != nullptr || !score_uses_tensor_cores(p)) return false;
  if (p.k_dtype == IDX_FP8_E4M3) return p.H == 16 || p.H == 32;
  return p.H == 16 || p.H == 32 || p.H == 64;
}

cudaError_t launch_score_group(const idx_problem& p, const int32_t* list, const int32_t* cnt, int64_t gld,
                               float* scores, int64_t ld, cudaStream_t st) {
  TcArgs a{};
  a.p = p;
  a.list = list;
  a.cnt = cnt;
  a.gld = gld;
  a.scores = scores;
  a.ld = ld;
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
