// Indexer score on CUDA cores: s(k) = sum_h w_h ReLU(q_h . k)
// ("DoSA：用安全上界减少 Indexer 的完整打分", section 3).
//
// Used for fp32 inputs and for bf16 shapes the tensor-core kernel does not
// cover.  One thread per (row, key); the row's queries and weights are staged
// in shared memory.  Each dot is an fp32 fused-multiply-add chain over
// d = 0..D-1 and the head sum a chain over h = 0..H-1, so a (query, key)
// score has the same bits whichever launch computes it.
#include "internal.h"

namespace idx {

constexpr int kSimtThreads = 128;

template <int KDT>
__device__ __forceinline__ float load_key(const void* keys, int64_t idx) {
  if (KDT == IDX_F32) return __ldg((const float*)keys + idx);
  const uint16_t b = __ldg((const unsigned short*)keys + idx);
  return __uint_as_float((uint32_t)b << 16);
}

// Score of key `key` (row-relative) of row m against the staged queries.
template <int KDT>
__device__ __forceinline__ float simt_pair_score(const idx_problem& p, const float* qs, int64_t krow_elem) {
  const int H = p.H, D = p.D;
  float s = 0.0f;
  for (int h = 0; h < H; ++h) {
    const float* qh = qs + h * D;
    float dot = 0.0f;
    for (int d = 0; d < D; ++d) dot = __fmaf_rn(qh[d], load_key<KDT>(p.keys, krow_elem + d), dot);
    s = __fmaf_rn(qs[H * D + h], fmaxf(dot, 0.0f), s);
  }
  return s;
}

template <int QDT>
__device__ __forceinline__ void stage_query(const idx_problem& p, int64_t m, float* qs) {
  const int H = p.H, D = p.D;
  for (int i = threadIdx.x; i < H * D; i += blockDim.x) {
    float v;
    if (QDT == IDX_F32) {
      v = ((const float*)p.q)[m * H * D + i];
    } else {
      v = __uint_as_float((uint32_t)((const unsigned short*)p.q)[m * H * D + i] << 16);
    }
    qs[i] = v;
  }
  for (int h = threadIdx.x; h < H; h += blockDim.x) qs[H * D + h] = p.w[m * H + h];
}

template <int QDT, int KDT>
__global__ void __launch_bounds__(kSimtThreads) score_simt_kernel(idx_problem p, float* __restrict__ scores,
                                                                   int64_t ld, const int32_t* __restrict__ row_mask) {
  extern __shared__ float qs[];   // [H*D] queries then [H] weights
  for (int64_t m = blockIdx.y; m < p.M; m += gridDim.y) {
    int64_t off;
    int len;
    bool ok = row_extent(p, m, &off, &len);
    if (!ok && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&g_device_error, DEVERR_BAD_ROW);
    if (row_mask && !row_mask[m]) len = 0;
    if ((int64_t)blockIdx.x * kSimtThreads >= len) continue;   // uniform over the block
    __syncthreads();
    stage_query<QDT>(p, m, qs);
    __syncthreads();
    const int key = blockIdx.x * kSimtThreads + threadIdx.x;
    if (key < len) scores[m * ld + key] = simt_pair_score<KDT>(p, qs, (off + key) * (int64_t)p.D);
  }
}

cudaError_t launch_score_simt(const idx_problem& p, float* scores, int64_t ld, const int32_t* row_mask,
                              cudaStream_t st) {
  if (p.M <= 0 || p.max_key_len <= 0) return cudaSuccess;
  dim3 grid((unsigned)((p.max_key_len + kSimtThreads - 1) / kSimtThreads), (unsigned)(p.M < 65535 ? p.M : 65535));
  size_t smem = (size_t)(p.H * p.D + p.H) * sizeof(float);
  cudaError_t e;
  if (p.q_dtype == IDX_F32 && p.k_dtype == IDX_F32) {
    e = cudaFuncSetAttribute(score_simt_kernel<IDX_F32, IDX_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    score_simt_kernel<IDX_F32, IDX_F32><<<grid, kSimtThreads, smem, st>>>(p, scores, ld, row_mask);
  } else {
    e = cudaFuncSetAttribute(score_simt_kernel<IDX_BF16, IDX_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    score_simt_kernel<IDX_BF16, IDX_BF16><<<grid, kSimtThreads, smem, st>>>(p, scores, ld, row_mask);
  }
  return cudaGetLastError();
}

}  // namespace idx
