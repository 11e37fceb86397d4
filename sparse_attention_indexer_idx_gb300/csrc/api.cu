// C-ABI entry points of libidx: argument validation on the host, workspace
// carving and dispatch to the kernels.  Nothing here computes on the host.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <vector>
#include <cstring>
#include <string>

#include "internal.h"

namespace idx {

static std::vector<uint32_t (*)()>& error_words() {
  static std::vector<uint32_t (*)()> v;
  return v;
}
static std::mutex g_error_words_mu;

void register_error_word(uint32_t (*take)()) {
  std::lock_guard<std::mutex> lk(g_error_words_mu);
  error_words().push_back(take);
}

static std::vector<cudaError_t (*)(uint64_t)>& wait_limit_setters() {
  static std::vector<cudaError_t (*)(uint64_t)> v;
  return v;
}

void register_wait_limit_setter(cudaError_t (*set)(uint64_t)) {
  std::lock_guard<std::mutex> lk(g_error_words_mu);
  wait_limit_setters().push_back(set);
}

static thread_local std::string g_last_error;

idx_status fail(idx_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

static idx_status cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return IDX_OK;
  return fail(IDX_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// SM count of the calling thread's current device, cached per device (the
// kernels size their grids by it, and a process may switch devices).
int sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (cached) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

static idx_status check_problem(const idx_problem* p) {
  if (!p) return fail(IDX_ERR_INVALID_ARG, "problem is NULL");
  if (p->M < 0 || p->H <= 0 || p->D <= 0 || p->n_keys < 0 || p->max_key_len < 0)
    return fail(IDX_ERR_INVALID_ARG, "negative or zero size (M=%lld H=%d D=%d n_keys=%lld max_key_len=%d)",
                (long long)p->M, p->H, p->D, (long long)p->n_keys, p->max_key_len);
  // bounds that keep every size derived from the problem (the M x max_key_len
  // scores, workspaces, key offsets) far inside 64-bit arithmetic (checked by
  // division, so the check itself cannot wrap)
  if (p->M > ((int64_t)1 << 40) || p->n_keys > ((int64_t)1 << 46) ||
      (p->max_key_len > 0 && p->M > ((int64_t)1 << 56) / p->max_key_len))
    return fail(IDX_ERR_UNSUPPORTED, "problem too large (M=%lld max_key_len=%d n_keys=%lld)", (long long)p->M,
                p->max_key_len, (long long)p->n_keys);
  if (p->M > 0 && (!p->q || !p->w || !p->key_len))
    return fail(IDX_ERR_INVALID_ARG, "q, w and key_len must be non-NULL");
  if (p->n_keys > 0 && !p->keys) return fail(IDX_ERR_INVALID_ARG, "keys is NULL");
  if (p->H > 128) return fail(IDX_ERR_UNSUPPORTED, "H=%d above 128", p->H);
  const bool f32 = p->q_dtype == IDX_F32 && p->k_dtype == IDX_F32;
  const bool bf16 = p->q_dtype == IDX_BF16 && p->k_dtype == IDX_BF16;
  const bool fp8 = p->q_dtype == IDX_BF16 && p->k_dtype == IDX_FP8_E4M3;
  if (!(f32 || bf16 || fp8))
    return fail(IDX_ERR_UNSUPPORTED, "dtype pair (q %d, keys %d) not supported", p->q_dtype, p->k_dtype);
  if (fp8 && !p->key_scale) return fail(IDX_ERR_INVALID_ARG, "FP8 keys need key_scale");
  if (!fp8 && p->key_scale) return fail(IDX_ERR_INVALID_ARG, "key_scale is only for FP8 keys");
  if ((f32 || bf16) && p->D > 256) return fail(IDX_ERR_UNSUPPORTED, "D=%d above 256", p->D);
  if ((int64_t)p->H * p->D > 16384) return fail(IDX_ERR_UNSUPPORTED, "H*D above 16384");
  if (fp8 && !score_uses_tensor_cores(*p))
    return fail(IDX_ERR_UNSUPPORTED, "FP8 keys need D=128 and H in {16,32,64,128}");
  if (!p->key_off && p->max_key_len > p->n_keys)
    return fail(IDX_ERR_INVALID_ARG, "shared keys: max_key_len %d exceeds n_keys %lld", p->max_key_len,
                (long long)p->n_keys);
  return IDX_OK;
}

}  // namespace idx

using namespace idx;

extern "C" {

const char* idx_last_error_string(void) { return g_last_error.c_str(); }

uint32_t idx_device_error(void) {
  cudaDeviceSynchronize();
  uint32_t v = 0;
  std::lock_guard<std::mutex> lk(g_error_words_mu);
  for (auto take : error_words()) v |= take();
  return v;
}

idx_status idx_set_wait_limit_ns(uint64_t ns) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e, "idx_set_wait_limit_ns");
  std::lock_guard<std::mutex> lk(g_error_words_mu);
  for (auto set : wait_limit_setters()) {
    e = set(ns);
    if (e != cudaSuccess) return cuda_status(e, "idx_set_wait_limit_ns");
  }
  return IDX_OK;
}

idx_status idx_score(const idx_problem* p, float* scores, int64_t ld_scores, void* stream) {
  idx_status st = check_problem(p);
  if (st) return st;
  if (ld_scores < p->max_key_len) return fail(IDX_ERR_INVALID_ARG, "ld_scores < max_key_len");
  if (p->M > 0 && p->max_key_len > 0 && !scores) return fail(IDX_ERR_INVALID_ARG, "scores is NULL");
  return cuda_status(launch_score(*p, scores, ld_scores, (cudaStream_t)stream), "idx_score");
}

size_t idx_topk_workspace_size(const idx_problem* p, int32_t K) {
  if (!p || p->M <= 0) return 0;
  WsCarver c(nullptr);
  c.take<float>((size_t)p->M * (size_t)(p->max_key_len > 0 ? p->max_key_len : 1));
  c.take<char>(topk_dense_ws(p->M, p->max_key_len, K < 1 ? 1 : K));
  return c.used + 256;
}

idx_status idx_topk(const idx_problem* p, int32_t K, int32_t* out_ids, float* out_scores, void* ws, size_t ws_bytes,
                    void* stream) {
  idx_status st = check_problem(p);
  if (st) return st;
  if (K < 1 || K > IDX_MAX_K) return fail(IDX_ERR_INVALID_ARG, "K=%d outside [1, %d]", K, IDX_MAX_K);
  if (p->M > 0 && !out_ids) return fail(IDX_ERR_INVALID_ARG, "out_ids is NULL");
  if (ws_bytes < idx_topk_workspace_size(p, K)) return fail(IDX_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (p->M > 0 && !ws) return fail(IDX_ERR_INVALID_ARG, "workspace is NULL");
  if (p->M == 0) return IDX_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t ld = p->max_key_len > 0 ? p->max_key_len : 1;
  WsCarver c(ws);
  float* scores = c.take<float>((size_t)p->M * (size_t)ld);
  char* lists = c.take<char>(topk_dense_ws(p->M, p->max_key_len, K));
  cudaError_t e = launch_score(*p, scores, ld, s);
  if (e != cudaSuccess) return cuda_status(e, "idx_topk/score");
  e = launch_topk_dense(scores, ld, nullptr, p, p->M, p->max_key_len, K, out_ids, out_scores, lists, s);
  return cuda_status(e, "idx_topk/select");
}

size_t idx_topk_prior_workspace_size(const idx_problem* p, int32_t K, int32_t prior_ld,
                                     int32_t candidate_capacity) {
  if (!p || p->M <= 0 || K < 1 || prior_ld < 1 || candidate_capacity < 1) return 0;
  return topk_prior_ws(*p, K, prior_ld, candidate_capacity);
}

static idx_status topk_prior_impl(const idx_problem* p, int32_t K, const int32_t* prior_ids, int32_t prior_ld,
                                  int32_t candidate_capacity, int32_t* out_ids, float* out_scores,
                                  int32_t* row_status, topk_prior_stats* stats, void* ws, size_t ws_bytes,
                                  void* stream, const cudaEvent_t* ev) {
  idx_status st = check_problem(p);
  if (st) return st;
  if (K < 1 || K > IDX_MAX_K) return fail(IDX_ERR_INVALID_ARG, "K=%d outside [1, %d]", K, IDX_MAX_K);
  if (prior_ld < 1) return fail(IDX_ERR_INVALID_ARG, "prior_ld=%d below 1", prior_ld);
  if (candidate_capacity < K)
    return fail(IDX_ERR_INVALID_ARG, "candidate_capacity=%d below K=%d", candidate_capacity, K);
  if (p->M == 0) return IDX_OK;
  if (!out_ids || !prior_ids) return fail(IDX_ERR_INVALID_ARG, "NULL pointer");
  if (ws_bytes < idx_topk_prior_workspace_size(p, K, prior_ld, candidate_capacity))
    return fail(IDX_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (!ws) return fail(IDX_ERR_INVALID_ARG, "workspace is NULL");
  return cuda_status(launch_topk_prior(*p, K, prior_ids, prior_ld, candidate_capacity, out_ids, out_scores,
                                       row_status, stats, ws, (cudaStream_t)stream, ev),
                     "idx_topk_prior");
}

idx_status idx_topk_prior(const idx_problem* p, int32_t K, const int32_t* prior_ids, int32_t prior_ld,
                          int32_t candidate_capacity, int32_t* out_ids, float* out_scores, int32_t* row_status,
                          topk_prior_stats* stats, void* ws, size_t ws_bytes, void* stream) {
  return topk_prior_impl(p, K, prior_ids, prior_ld, candidate_capacity, out_ids, out_scores, row_status, stats, ws,
                         ws_bytes, stream, nullptr);
}

idx_status idx_topk_prior_events(const idx_problem* p, int32_t K, const int32_t* prior_ids, int32_t prior_ld,
                                 int32_t candidate_capacity, int32_t* out_ids, float* out_scores,
                                 int32_t* row_status, topk_prior_stats* stats, void* ws, size_t ws_bytes,
                                 void* const* events, int32_t n_events, void* stream) {
  if (!events || n_events < 6) return fail(IDX_ERR_INVALID_ARG, "idx_topk_prior_events needs 6 events");
  cudaEvent_t ev[6];
  for (int i = 0; i < 6; ++i) ev[i] = (cudaEvent_t)events[i];
  return topk_prior_impl(p, K, prior_ids, prior_ld, candidate_capacity, out_ids, out_scores, row_status, stats, ws,
                         ws_bytes, stream, ev);
}

size_t idx_topk_scores_workspace_size(int64_t M, int32_t max_len, int32_t K) {
  if (M <= 0 || max_len <= 0) return 0;
  return topk_dense_ws(M, max_len, K < 1 ? 1 : K);
}

idx_status idx_topk_scores(const float* scores, int64_t ld, const int32_t* lens, int64_t M, int32_t max_len,
                           int32_t K, int32_t* out_ids, float* out_scores, void* ws, size_t ws_bytes,
                           void* stream) {
  if (M < 0 || max_len < 0 || ld < max_len) return fail(IDX_ERR_INVALID_ARG, "bad sizes");
  if (K < 1 || K > IDX_MAX_K) return fail(IDX_ERR_INVALID_ARG, "K=%d outside [1, %d]", K, IDX_MAX_K);
  if (M > 0 && (!lens || !out_ids || (max_len > 0 && !scores))) return fail(IDX_ERR_INVALID_ARG, "NULL pointer");
  const size_t need = idx_topk_scores_workspace_size(M, max_len, K);
  if (ws_bytes < need) return fail(IDX_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (need > 0 && !ws) return fail(IDX_ERR_INVALID_ARG, "workspace is NULL");
  if (M == 0) return IDX_OK;
  return cuda_status(launch_topk_dense(scores, ld, lens, nullptr, M, max_len, K, out_ids, out_scores, ws,
                                       (cudaStream_t)stream),
                     "idx_topk_scores");
}

size_t dosa_topk_workspace_size(const idx_problem* p, int32_t K, const dosa_params* dp, int32_t seed_ld) {
  if (!p || !dp || p->M <= 0) return 0;
  return dosa_ws(*p, K, *dp, seed_ld);
}

idx_status dosa_topk(const idx_problem* p, int32_t K, const dosa_params* dp, const int32_t* seed_ids,
                     int32_t seed_ld, int32_t* out_ids, float* out_scores, int32_t* row_status, dosa_stats* stats,
                     void* ws, size_t ws_bytes, void* stream) {
  idx_status st = check_problem(p);
  if (st) return st;
  if (!dp) return fail(IDX_ERR_INVALID_ARG, "params is NULL");
  if (K < 1 || K > IDX_MAX_K) return fail(IDX_ERR_INVALID_ARG, "K=%d outside [1, %d]", K, IDX_MAX_K);
  if (dp->n_seed < 0 || dp->retained_heads < 1 || dp->n_sample < 1 || dp->candidate_capacity < 0 ||
      !(dp->act_freq_min >= 0.0f && dp->act_freq_min <= 1.0f) || !(dp->margin_gamma >= 0.0f))
    return fail(IDX_ERR_INVALID_ARG, "bad dosa_params");
  if (seed_ids && seed_ld < 1) return fail(IDX_ERR_INVALID_ARG, "seed_ld < 1");
  if (p->M > 0 && !out_ids) return fail(IDX_ERR_INVALID_ARG, "out_ids is NULL");
  if (ws_bytes < dosa_topk_workspace_size(p, K, dp, seed_ids ? seed_ld : 0))
    return fail(IDX_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (p->M == 0) return IDX_OK;
  if (!ws) return fail(IDX_ERR_INVALID_ARG, "workspace is NULL");
  return cuda_status(launch_dosa(*p, K, *dp, seed_ids, seed_ids ? seed_ld : 0, out_ids, out_scores, row_status,
                                 stats, ws, ws_bytes, (cudaStream_t)stream),
                     "dosa_topk");
}

idx_status dosa_workspace_layout(const idx_problem* p, int32_t K, const dosa_params* dp, int32_t seed_ld,
                                 dosa_ws_layout* out) {
  idx_status st = check_problem(p);
  if (st) return st;
  if (!dp || !out) return fail(IDX_ERR_INVALID_ARG, "NULL pointer");
  if (K < 1 || K > IDX_MAX_K) return fail(IDX_ERR_INVALID_ARG, "K=%d outside [1, %d]", K, IDX_MAX_K);
  if (!dosa_layout(*p, K, *dp, seed_ld > 0 ? seed_ld : 0, out))
    return fail(IDX_ERR_UNSUPPORTED, "dosa_topk takes the unpruned path for this shape");
  return IDX_OK;
}

idx_status witness_merge(int32_t* topk_ids, int64_t rows, int32_t topk, const int32_t* context_lens,
                         int64_t n_context_lens, int32_t keep, int32_t num_segments, int32_t max_replacements,
                         void* stream) {
  if (num_segments == 0) return IDX_OK;
  if (num_segments < 0 || num_segments > IDX_MAX_SEGMENTS)
    return fail(IDX_ERR_SEGMENTS_OUT_OF_RANGE, "num_segments=%d outside [1, %d]", num_segments, IDX_MAX_SEGMENTS);
  if (keep < 0 || keep > topk) return fail(IDX_ERR_KEEP_OUT_OF_RANGE, "keep=%d outside [0, topk=%d]", keep, topk);
  if (rows < 0 || topk < 0 || max_replacements < 0) return fail(IDX_ERR_INVALID_ARG, "negative size");
  if (n_context_lens < rows)
    return fail(IDX_ERR_ROWS_MISMATCH, "%lld context lengths for %lld rows", (long long)n_context_lens,
                (long long)rows);
  const int32_t B = max_replacements < topk - keep ? max_replacements : topk - keep;
  if (B <= 0 || rows == 0) return IDX_OK;
  if (!topk_ids || !context_lens) return fail(IDX_ERR_INVALID_ARG, "NULL pointer");
  return cuda_status(launch_witness_merge(topk_ids, rows, topk, context_lens, keep, num_segments, B,
                                          (cudaStream_t)stream),
                     "witness_merge");
}

idx_status witness_indices(const int32_t* learned, int64_t rows, int32_t topk, const int32_t* context_lens,
                           int64_t n_context_lens, int32_t num_segments, int32_t* out, void* stream) {
  if (num_segments <= 0 || num_segments > IDX_MAX_SEGMENTS)
    return fail(IDX_ERR_SEGMENTS_OUT_OF_RANGE, "num_segments=%d outside [1, %d]", num_segments, IDX_MAX_SEGMENTS);
  if (rows < 0 || topk < 0) return fail(IDX_ERR_INVALID_ARG, "negative size");
  if (n_context_lens < rows)
    return fail(IDX_ERR_ROWS_MISMATCH, "%lld context lengths for %lld rows", (long long)n_context_lens,
                (long long)rows);
  if (rows == 0) return IDX_OK;
  if ((topk > 0 && !learned) || !context_lens || !out) return fail(IDX_ERR_INVALID_ARG, "NULL pointer");
  return cuda_status(launch_witness_indices(learned, rows, topk, context_lens, num_segments, out,
                                            (cudaStream_t)stream),
                     "witness_indices");
}

size_t block_select_workspace_size(int64_t Q, int32_t n_kv, int64_t L, const block_sparse_config* cfg) {
  if (!cfg || Q <= 0 || n_kv <= 0 || L <= 0) return 0;
  return block_select_ws(Q, n_kv, L, *cfg);
}

static idx_status block_select_impl(const float* index_q, const float* index_k, const int32_t* query_pos, int64_t Q,
                                    int32_t n_kv, int32_t D, int64_t L, const block_sparse_config* cfg, int32_t* out,
                                    int32_t out_width, int32_t* out_count, block_select_stats* stats, void* ws,
                                    size_t ws_bytes, void* stream, const cudaEvent_t* ev) {
  if (!cfg) return fail(IDX_ERR_INVALID_ARG, "config is NULL");
  if (Q < 0 || n_kv < 0 || D <= 0 || L < 0 || cfg->block_size < 0 || cfg->top_blocks < 0 || cfg->init_blocks < 0 ||
      cfg->local_blocks < 0)
    return fail(IDX_ERR_INVALID_ARG, "negative size or config field");
  const int64_t need_w = cfg->top_blocks > (int64_t)cfg->init_blocks + cfg->local_blocks
                             ? cfg->top_blocks
                             : (int64_t)cfg->init_blocks + cfg->local_blocks;
  if (out_width < need_w || out_width > IDX_MAX_K)
    return fail(IDX_ERR_INVALID_ARG, "out_width=%d must be in [max(top, init+local)=%lld, %d]", out_width,
                (long long)need_w, IDX_MAX_K);
  if (D > 256) return fail(IDX_ERR_UNSUPPORTED, "D=%d above 256", D);
  if (D == 128 && (((uintptr_t)index_q | (uintptr_t)index_k) & 15))
    return fail(IDX_ERR_INVALID_ARG, "index_q/index_k must be 16-byte aligned");
  if (Q * n_kv == 0) return IDX_OK;
  if (!index_q || !query_pos || !out || (L > 0 && !index_k)) return fail(IDX_ERR_INVALID_ARG, "NULL pointer");
  if (ws_bytes < block_select_workspace_size(Q, n_kv, L, cfg))
    return fail(IDX_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (block_select_workspace_size(Q, n_kv, L, cfg) > 0 && !ws) return fail(IDX_ERR_INVALID_ARG, "workspace is NULL");
  return cuda_status(launch_block_select(index_q, index_k, query_pos, Q, n_kv, D, L, *cfg, out, out_width, out_count,
                                         ws, (cudaStream_t)stream, stats, true, ev),
                     "block_select");
}

idx_status block_select(const float* index_q, const float* index_k, const int32_t* query_pos, int64_t Q,
                        int32_t n_kv, int32_t D, int64_t L, const block_sparse_config* cfg, int32_t* out,
                        int32_t out_width, int32_t* out_count, block_select_stats* stats, void* ws,
                        size_t ws_bytes, void* stream) {
  return block_select_impl(index_q, index_k, query_pos, Q, n_kv, D, L, cfg, out, out_width, out_count, stats, ws,
                           ws_bytes, stream, nullptr);
}

idx_status block_select_events(const float* index_q, const float* index_k, const int32_t* query_pos, int64_t Q,
                               int32_t n_kv, int32_t D, int64_t L, const block_sparse_config* cfg, int32_t* out,
                               int32_t out_width, int32_t* out_count, block_select_stats* stats, void* ws,
                               size_t ws_bytes, void* const* events, int32_t n_events, void* stream) {
  if (!events || n_events < 6) return fail(IDX_ERR_INVALID_ARG, "block_select_events needs 6 events");
  cudaEvent_t ev[6];
  for (int i = 0; i < 6; ++i) ev[i] = (cudaEvent_t)events[i];
  return block_select_impl(index_q, index_k, query_pos, Q, n_kv, D, L, cfg, out, out_width, out_count, stats, ws,
                           ws_bytes, stream, ev);
}

idx_status block_positions(const int32_t* blocks, const int32_t* counts, int64_t Q, int32_t n_kv, int32_t W,
                           const int32_t* query_pos, int64_t L, int32_t block_size, int32_t* out, int32_t out_width,
                           int32_t* out_count, void* stream) {
  if (Q < 0 || n_kv <= 0 || W < 0 || L < 0 || block_size < 0)
    return fail(IDX_ERR_INVALID_ARG, "negative size, or n_kv <= 0");
  if (W > IDX_MAX_K) return fail(IDX_ERR_INVALID_ARG, "W=%d above %d", W, IDX_MAX_K);
  if ((int64_t)out_width < (int64_t)W * block_size || out_width < 0)
    return fail(IDX_ERR_INVALID_ARG, "out_width=%d below W*block_size=%lld", out_width, (long long)W * block_size);
  if (Q * n_kv == 0) return IDX_OK;
  if ((W > 0 && !blocks) || !query_pos || (out_width > 0 && !out)) return fail(IDX_ERR_INVALID_ARG, "NULL pointer");
  return cuda_status(launch_block_positions(blocks, counts, Q * n_kv, W, query_pos, n_kv, L, block_size, out,
                                            out_width, out_count, (cudaStream_t)stream),
                     "block_positions");
}

}  // extern "C"
