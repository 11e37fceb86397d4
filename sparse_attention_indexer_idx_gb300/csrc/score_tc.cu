// bf16-key dense instantiations of the tensor-core score kernel (score_tc.cuh)
// and the tensor-map helper shared with the other instantiations.
#include <cudaTypedefs.h>

#include "score_tc.cuh"

namespace idx {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_score_tc_fp8(const TcArgs& a, cudaStream_t st);

cudaError_t launch_score_tc(const idx_problem& p, float* scores, int64_t ld, const int32_t* row_mask,
                            cudaStream_t st) {
  TcArgs a{};
  a.p = p;
  a.scores = scores;
  a.ld = ld;
  a.row_mask = row_mask;
  if (p.k_dtype == IDX_FP8_E4M3) return launch_score_tc_fp8(a, st);
  const bool shared = p.key_off == nullptr;
  switch (p.H) {
    case 16: return shared ? launch_tc<TcCfg<IDX_BF16, 16, 16, kScore>>(a, st)
                           : launch_tc<TcCfg<IDX_BF16, 16, 1, kScore>>(a, st);
    case 32: return shared ? launch_tc<TcCfg<IDX_BF16, 32, 8, kScore>>(a, st)
                           : launch_tc<TcCfg<IDX_BF16, 32, 1, kScore>>(a, st);
    case 64: return shared ? launch_tc<TcCfg<IDX_BF16, 64, 4, kScore>>(a, st)
                           : launch_tc<TcCfg<IDX_BF16, 64, 1, kScore>>(a, st);
    case 128: return shared ? launch_tc<TcCfg<IDX_BF16, 128, 2, kScore>>(a, st)
                            : launch_tc<TcCfg<IDX_BF16, 128, 1, kScore>>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace idx
