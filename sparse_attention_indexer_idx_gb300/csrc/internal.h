// Library-internal declarations shared by the .cu files of libidx.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/idx.h"
#include "common.cuh"

namespace idx {

constexpr int kTile = 128;  // keys per tensor-core tile (one TMEM lane each)

// Number of streaming multiprocessors of the current device (cached).
int sm_count();

// Records the message returned by idx_last_error_string() and returns st.
idx_status fail(idx_status st, const char* fmt, ...);

// Visible extent of row m: false (and len 0) when the extent does not fit the
// key buffer or exceeds max_key_len.
__device__ __forceinline__ bool row_extent(const idx_problem& p, int64_t m, int64_t* off, int* len) {
  int32_t L = p.key_len[m];
  int64_t o = p.key_off ? p.key_off[m] : 0;
  bool ok = L >= 0 && L <= p.max_key_len && o >= 0 && o + (int64_t)L <= p.n_keys;
  *off = ok ? o : 0;
  *len = ok ? L : 0;
  return ok;
}

// ---- launchers (host) -------------------------------------------------------
cudaError_t launch_witness_merge(int32_t* ids, int64_t rows, int topk, const int32_t* ctx, int keep, int S, int B,
                                 cudaStream_t st);
cudaError_t launch_witness_indices(const int32_t* ids, int64_t rows, int topk, const int32_t* ctx, int S,
                                   int32_t* out, cudaStream_t st);

// Exact top-K of dense score rows; ws holds topk_dense_ws() bytes (0 when every
// row fits one chunk).  Rows come from lens[m] (clamped to [0, max_len]) or,
// when p_or_null is given, from the problem's visible extents.
size_t topk_dense_ws(int64_t M, int max_len, int K);
// id_map (optional, [M, id_ld]): position i of row m stands for key id
// id_map[m*id_ld + i] (id_ld 0: one map shared by all rows).  row_mask
// (optional): rows with row_mask[m] == 0 are neither read nor written.
cudaError_t launch_topk_dense(const float* scores, int64_t ld, const int32_t* lens, const idx_problem* p_or_null,
                              int64_t M, int max_len, int K, int32_t* out_ids, float* out_scores, void* ws,
                              cudaStream_t st, const int32_t* id_map = nullptr, int64_t id_ld = 0,
                              const int32_t* row_mask = nullptr);

// Scores of every visible key (the kernel family depends only on dtype/H/D).
// row_mask (optional, device [M]): rows with row_mask[m] == 0 are skipped.
cudaError_t launch_score(const idx_problem& p, float* scores, int64_t ld, cudaStream_t st,
                         const int32_t* row_mask = nullptr);
bool score_uses_tensor_cores(const idx_problem& p);
cudaError_t launch_score_simt(const idx_problem& p, float* scores, int64_t ld, const int32_t* row_mask,
                              cudaStream_t st);
cudaError_t launch_score_tc(const idx_problem& p, float* scores, int64_t ld, const int32_t* row_mask,
                            cudaStream_t st);
// Exact scores of per-row key lists (tensor-core shapes only): scores[m*ld + i]
// for list position i < cnt[m] of row m, keys key_off[m] + list[m*gld + i].
cudaError_t launch_score_gather(const idx_problem& p, const int32_t* list, const int32_t* cnt, int64_t gld,
                                float* scores, int64_t ld, const int32_t* row_mask, cudaStream_t st);
// Shared candidate stream: group g = rows 4g..4g+3 over one key sequence scores
// the keys list[g*gld + i], i < cnt[g], for its four rows: scores[m*ld + i]
// (m = 4g + q).  Shared keys, tensor-core shapes with 4 queries per MMA tile.
bool group_stream_supported(const idx_problem& p);
cudaError_t launch_score_group(const idx_problem& p, const int32_t* list, const int32_t* cnt, int64_t gld,
                               float* scores, int64_t ld, cudaStream_t st);
// DoSA bound scan over prepared vectors prep.q = [M, 32, 128] bf16: bit k of
// candbits row m (cb_stride words, at least ceil(max_key_len / 128) * 4) is set
// iff key k is a candidate; words of tiles past a row's group are not written.
// Shared keys (key_off == NULL) need knorm [n_keys] = ||k|| rounded up (codes
// for FP8); per-row keys take ||k|| from the key tile (knorm unused).
// Prepared rows R..30 and their folded weights must be zero.  With
// bound_group_layout(p, R) the prepared rows are laid out per group of 8
// queries: 144 rows at group * 144, query q's vector r < 16 at q * 16 + r, its
// aggregate at 128 + q (rows 136..143 zero).
bool bound_group_layout(const idx_problem& p, int R);
cudaError_t launch_bound(const idx_problem& prep, const float* wfold, const float* coef, const float* tau,
                         const float* knorm, const uint32_t* seedbits, int64_t seed_stride, uint32_t* candbits,
                         int64_t cb_stride, int R, const int32_t* row_mask, cudaStream_t st);

size_t block_select_ws(int64_t Q, int n_kv, int64_t L, const block_sparse_config& c);
// tensor_route: allow the tensor-core route (block_tc.cu) when it applies; ws
// must then hold block_select_ws() bytes, which covers both routes.
cudaError_t launch_block_select(const float* q, const float* k, const int32_t* pos, int64_t Q, int n_kv, int D,
                                int64_t L, const block_sparse_config& c, int32_t* out, int out_width,
                                int32_t* out_count, void* ws, cudaStream_t st, block_select_stats* stats,
                                bool tensor_route, const cudaEvent_t* ev = nullptr);
cudaError_t launch_block_positions(const int32_t* blocks, const int32_t* counts, int64_t rows, int W,
                                   const int32_t* qpos, int n_kv, int64_t L, int bs, int32_t* out, int ow,
                                   int32_t* out_count, cudaStream_t st);
bool block_select_tc_applies(int D, const block_sparse_config& c, int64_t Q, int n_kv, int64_t L);
size_t block_select_tc_ws(int64_t Q, int n_kv, int64_t L, const block_sparse_config& c);
cudaError_t launch_block_select_tc(const float* q, const float* k, const int32_t* pos, int64_t Q, int n_kv,
                                   int64_t L, const block_sparse_config& c, int32_t* out, int out_width,
                                   int32_t* out_count, void* ws, block_select_stats* stats, cudaStream_t st,
                                   const cudaEvent_t* ev = nullptr);

size_t topk_prior_ws(const idx_problem& p, int K, int P, int64_t cap);
cudaError_t launch_topk_prior(const idx_problem& p, int K, const int32_t* prior, int P, int64_t cap,
                              int32_t* out_ids, float* out_scores, int32_t* row_status, topk_prior_stats* stats,
                              void* ws, cudaStream_t st, const cudaEvent_t* ev = nullptr);

size_t dosa_ws(const idx_problem& p, int K, const dosa_params& dp, int seed_ld);
// Byte offsets of the pruned path's intermediate arrays in the workspace
// (false where dosa_topk takes the unpruned path for every row).
bool dosa_layout(const idx_problem& p, int K, const dosa_params& dp, int seed_ld, dosa_ws_layout* out);
cudaError_t launch_dosa(const idx_problem& p, int K, const dosa_params& dp, const int32_t* seed_ids, int seed_ld,
                        int32_t* out_ids, float* out_scores, int32_t* row_status, dosa_stats* stats, void* ws,
                        size_t ws_bytes, cudaStream_t st);

// ---- workspace carving -------------------------------------------------------
struct WsCarver {
  char* base;
  size_t used = 0;
  explicit WsCarver(void* b) : base((char*)b) {}
  template <class T>
  T* take(size_t count) {
    size_t off = (used + 255) & ~size_t(255);
    used = off + count * sizeof(T);
    return base ? (T*)(base + off) : nullptr;
  }
};

}  // namespace idx
