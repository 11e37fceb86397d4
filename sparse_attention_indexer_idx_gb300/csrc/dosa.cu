#include "internal.h"
namespace idx {
size_t dosa_ws(const idx_problem&, int, const dosa_params&, int) { return 0; }
cudaError_t launch_dosa(const idx_problem&, int, const dosa_params&, const int32_t*, int, int32_t*, float*, int32_t*,
                        dosa_stats*, void*, size_t, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace idx
