// FP8-e4m3-key instantiations of the tensor-core score kernel (score_tc.cuh).
#include "score_tc.cuh"

namespace idx {

cudaError_t launch_score_tc_fp8(const idx_problem& p, float* scores, int64_t ld, cudaStream_t st) {
  const bool shared = p.key_off == nullptr;
  switch (p.H) {
    case 16: return shared ? launch_tc<TcCfg<IDX_FP8_E4M3, 16, 16>>(p, scores, ld, st)
                           : launch_tc<TcCfg<IDX_FP8_E4M3, 16, 1>>(p, scores, ld, st);
    case 32: return shared ? launch_tc<TcCfg<IDX_FP8_E4M3, 32, 8>>(p, scores, ld, st)
                           : launch_tc<TcCfg<IDX_FP8_E4M3, 32, 1>>(p, scores, ld, st);
    case 64: return shared ? launch_tc<TcCfg<IDX_FP8_E4M3, 64, 4>>(p, scores, ld, st)
                           : launch_tc<TcCfg<IDX_FP8_E4M3, 64, 1>>(p, scores, ld, st);
    case 128: return shared ? launch_tc<TcCfg<IDX_FP8_E4M3, 128, 2>>(p, scores, ld, st)
                            : launch_tc<TcCfg<IDX_FP8_E4M3, 128, 1>>(p, scores, ld, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace idx
