// Exact top-K over dense score rows (see topk.cuh for the method).
#include "internal.h"
#include "topk.cuh"

namespace idx {

constexpr int kTopkThreads = 1024;

// One thread block per row.  When `p` is given, row m's length is its visible
// key count (rows with a bad extent are empty); otherwise lens[m], clamped to
// [0, max_len].
__global__ void __launch_bounds__(kTopkThreads) topk_dense_kernel(const float* __restrict__ scores, int64_t ld,
                                                                   const int32_t* __restrict__ lens,
                                                                   idx_problem p, int use_p, int max_len, int K,
                                                                   int32_t* __restrict__ out_ids,
                                                                   float* __restrict__ out_scores) {
  __shared__ TopkShared<kTopkThreads> sh;
  extern __shared__ uint64_t sel[];
  const int64_t m = blockIdx.x;
  int len;
  if (use_p) {
    int64_t off;
    row_extent(p, m, &off, &len);
  } else {
    len = lens[m];
    len = len < 0 ? 0 : (len > max_len ? max_len : len);
  }
  DenseScoreRow row{scores + m * ld, len};
  block_topk<kTopkThreads>(sh, sel, row, K, out_ids + m * (int64_t)K, out_scores ? out_scores + m * (int64_t)K : nullptr,
                           false);
}

static int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

cudaError_t launch_topk_dense(const float* scores, int64_t ld, const int32_t* lens, const idx_problem* p_or_null,
                              int64_t M, int max_len, int K, int32_t* out_ids, float* out_scores, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  size_t smem = (size_t)next_pow2(K) * sizeof(uint64_t);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(topk_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(IDX_MAX_K * sizeof(uint64_t)));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  idx_problem p{};
  if (p_or_null) p = *p_or_null;
  topk_dense_kernel<<<(unsigned)M, kTopkThreads, smem, st>>>(scores, ld, lens, p, p_or_null ? 1 : 0, max_len, K,
                                                             out_ids, out_scores);
  return cudaGetLastError();
}

}  // namespace idx
