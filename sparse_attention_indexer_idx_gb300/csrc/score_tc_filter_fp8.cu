// FP8-e4m3-key kFilter instantiations of the tensor-core score kernel (score_tc.cuh).
#include "score_tc.cuh"

namespace idx {

cudaError_t launch_score_filter_fp8(const TcArgs& a, cudaStream_t st) {
  switch (a.p.H) {
    case 16: return launch_tc<TcCfg<IDX_FP8_E4M3, 16, 1, kFilter>>(a, st);
    case 32: return launch_tc<TcCfg<IDX_FP8_E4M3, 32, 1, kFilter>>(a, st);
    case 64: return launch_tc<TcCfg<IDX_FP8_E4M3, 64, 1, kFilter>>(a, st);
    case 128: return launch_tc<TcCfg<IDX_FP8_E4M3, 128, 1, kFilter>>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace idx
