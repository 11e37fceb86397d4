// FP8-e4m3-key dense instantiations of the tensor-core score kernel (score_tc.cuh).
#include "score_tc.cuh"

namespace idx {

cudaError_t launch_score_tc_fp8(const TcArgs& a, cudaStream_t st) {
  const bool shared = a.p.key_off == nullptr;
  switch (a.p.H) {
    case 16: return shared ? launch_tc<TcCfg<IDX_FP8_E4M3, 16, 8, kScore>>(a, st)
                           : launch_tc<TcCfg<IDX_FP8_E4M3, 16, 1, kScore>>(a, st);
    case 32: return shared ? launch_tc<TcCfg<IDX_FP8_E4M3, 32, 4, kScore>>(a, st)
                           : launch_tc<TcCfg<IDX_FP8_E4M3, 32, 1, kScore>>(a, st);
    case 64: return shared ? launch_tc<TcCfg<IDX_FP8_E4M3, 64, 2, kScore>>(a, st)
                           : launch_tc<TcCfg<IDX_FP8_E4M3, 64, 1, kScore>>(a, st);
    case 128: return shared ? launch_tc<TcCfg<IDX_FP8_E4M3, 128, 1, kScore>>(a, st)
                            : launch_tc<TcCfg<IDX_FP8_E4M3, 128, 1, kScore>>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace idx
