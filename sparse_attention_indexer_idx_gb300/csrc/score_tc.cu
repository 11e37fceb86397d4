#include "internal.h"
namespace idx {
cudaError_t launch_score_tc(const idx_problem&, float*, int64_t, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace idx
