/*
 * libidx -- sparse-attention indexer hot path on one GB300 (sm_103a).
 *
 * Plain C ABI.  Every pointer named "device" is a CUDA device pointer owned by
 * the caller; the library never allocates device memory on these paths and
 * never synchronises the host: all work is enqueued on the caller's stream
 * (`stream` is a cudaStream_t; NULL is the legacy default stream).  Entry points
 * that need scratch memory take (ws, ws_bytes) and have a *_workspace_size()
 * query; the workspace is caller-owned device memory, at least 256-byte
 * aligned, and may be reused across calls that do not overlap on the GPU.
 *
 * Every argument that the host can see is validated before anything is
 * launched; a call that returns an error has enqueued nothing and written
 * nothing.  Values that live in device memory (key_len, key_off, context
 * lengths, query positions) cannot be checked by the host: a row whose extent
 * falls outside the key buffer or above max_key_len is treated as a row with
 * no visible keys and sets IDX_DEVERR_BAD_ROW in the device error word
 * (idx_device_error()).  Inputs are assumed finite; NaN scores are undefined.
 *
 * Notation follows the pages: M query rows, H index heads, D head dim, K the
 * top-K, L_r the visible keys of row r, S the segment count.
 */
#ifndef IDX_H_
#define IDX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------- status codes */
typedef int32_t idx_status;
enum {
  IDX_OK = 0,
  /* The three refusals of the segment-witness merge ("Segment Witnesses",
   * section "Refusals"): context lengths do not cover every row; segment count
   * zero (where there is no off switch) or above 64; retained prefix wider
   * than the row. */
  IDX_ERR_ROWS_MISMATCH = 1,
  IDX_ERR_SEGMENTS_OUT_OF_RANGE = 2,
  IDX_ERR_KEEP_OUT_OF_RANGE = 3,
  IDX_ERR_INVALID_ARG = 4,          /* null pointer, negative size, K too large, ... */
  IDX_ERR_UNSUPPORTED = 5,          /* dtype / shape combination not implemented */
  IDX_ERR_WORKSPACE_TOO_SMALL = 6,
  IDX_ERR_CUDA = 7                  /* a CUDA call failed; see idx_last_error_string() */
};

/* Device error word bits (idx_device_error). */
enum {
  IDX_DEVERR_WAIT_TIMEOUT = 1,      /* a pipeline wait hit its time limit; the kernel returned early */
  IDX_DEVERR_BAD_ROW = 2,           /* a row's key extent was outside the key buffer */
  IDX_DEVERR_CAPACITY = 4           /* an internal buffer overflowed; affected rows were recomputed */
};

/* Element types. */
enum { IDX_F32 = 0, IDX_BF16 = 1, IDX_FP8_E4M3 = 2 };

enum { IDX_MAX_SEGMENTS = 64, IDX_MAX_K = 4096 };

/* Human-readable text of the last host-side error of this thread. */
const char* idx_last_error_string(void);

/* Synchronises the device, returns the device error word and clears it. */
uint32_t idx_device_error(void);

/* Every wait inside a tensor-core pipeline (a warp waiting for a tile, an
 * accumulator or a free slot) gives up after a time limit: the kernel then
 * stops its pipeline, waits (with a fixed 2 s limit) for the copies and MMAs
 * it has in flight, frees its tensor memory, returns, and sets
 * IDX_DEVERR_WAIT_TIMEOUT; that call's output is undefined and later calls
 * are unaffected.  This sets the limit, in nanoseconds, for every kernel of
 * the library on the current device (after synchronising it); 0 gives up at
 * the first wait that is not already complete (for tests of the failure
 * path).  IDX_DEFAULT_WAIT_LIMIT_NS is the default. */
#define IDX_DEFAULT_WAIT_LIMIT_NS 2000000000ull
idx_status idx_set_wait_limit_ns(uint64_t ns);

/* ----------------------------------------------------------- the problem ---
 * One batch of indexer rows ("DoSA：用安全上界减少 Indexer 的完整打分",
 * section 3: one index key per position, shared by every head of a query).
 *
 *   q        device [M, H, D], q_dtype IDX_F32 or IDX_BF16, row-major.
 *   w        device [M, H] float32 head weights (either sign).
 *   keys     device [n_keys, D], k_dtype IDX_F32, IDX_BF16 or IDX_FP8_E4M3,
 *            row-major, rows 16-byte aligned for the bf16/fp8 paths.
 *   key_scale device [n_keys] float32 per-token dequantisation scale (> 0),
 *            required for IDX_FP8_E4M3 and NULL otherwise; the score of an FP8
 *            key k = scale * code is scale * sum_h w_h ReLU(q_h . code).
 *   key_off  device [M] int64, or NULL.  NULL: every row reads one shared key
 *            sequence starting at keys[0] (causal prefill; row m sees keys
 *            0..key_len[m]-1).  Non-NULL: row m reads its own keys
 *            keys[key_off[m] .. key_off[m]+key_len[m]-1] (decode).
 *   key_len  device [M] int32, L_r >= 0; key ids are row-relative, 0..L_r-1.
 *   max_key_len host-side bound on every key_len[m] (sizes grids/workspaces).
 *
 * Sizes: M <= 2^40, n_keys <= 2^46 and M * max_key_len <= 2^56, so that every
 * size derived from them stays inside 64-bit arithmetic; larger problems are
 * refused with IDX_ERR_UNSUPPORTED before any device work.
 *
 * Supported: (F32 q, F32 keys) any H <= 128, D <= 256 on CUDA cores;
 * (BF16 q, BF16 keys) and (BF16 q, FP8 keys) with D = 128 and H in
 * {16, 32, 64, 128} on the tensor cores; (BF16 q, BF16 keys) other shapes on
 * CUDA cores.  The same combination always takes the same kernels, so every
 * exact score of a (query, key) pair has the same bits on every path.
 */
typedef struct idx_problem {
  const void* q;
  int32_t q_dtype;
  const float* w;
  int64_t M;
  int32_t H;
  int32_t D;
  const void* keys;
  int32_t k_dtype;
  const float* key_scale;
  int64_t n_keys;
  const int64_t* key_off;
  const int32_t* key_len;
  int32_t max_key_len;
} idx_problem;

/* ---------------------------------------------------------------- idx_score
 * Indexer score s(k) = sum_h w_h ReLU(q_h . k) for every visible key
 * ("DoSA：用安全上界减少 Indexer 的完整打分", section 3, the equation for s(k)).
 * scores: device [M, ld_scores] float32; row m receives s for ids
 * 0..key_len[m]-1; entries at and beyond key_len[m] are not written.
 * ld_scores >= max_key_len.  No workspace. */
idx_status idx_score(const idx_problem* p, float* scores, int64_t ld_scores, void* stream);

/* ---------------------------------------------------------------- idx_topk
 * Exact top-K of every row under the total order (score desc, key id asc)
 * (same page, section 1 and the note after section 2: the final choice is by
 * the original scorer, and equal ids need one consistent total order).
 * out_ids: device [M, K] int32, sorted in that order; rows with fewer than K
 * visible keys are padded with -1.  out_scores: device [M, K] float32 or NULL,
 * padded with -inf; -0.0 is reported as +0.0.  1 <= K <= IDX_MAX_K. */
size_t idx_topk_workspace_size(const idx_problem* p, int32_t K);
idx_status idx_topk(const idx_problem* p, int32_t K, int32_t* out_ids, float* out_scores, void* ws,
                    size_t ws_bytes, void* stream);

/* ---------------------------------------------------------- idx_topk_scores
 * The top-K step alone, on score rows the caller already has: row m is
 * scores[m*ld .. m*ld + lens[m]-1] (device float32, lens device int32, clamped
 * to [0, max_len]), ids are positions in the row.  Same order, padding and K
 * limit as idx_topk.  The workspace holds, per row and per 16384 scores of
 * max_len, a candidate count and 4096 candidate slots of 8 bytes: about
 * M * max_len * 2 bytes. */
size_t idx_topk_scores_workspace_size(int64_t M, int32_t max_len, int32_t K);
idx_status idx_topk_scores(const float* scores, int64_t ld, const int32_t* lens, int64_t M, int32_t max_len,
                           int32_t K, int32_t* out_ids, float* out_scores, void* ws, size_t ws_bytes,
                           void* stream);

/* --------------------------------------------------------------- dosa_topk
 * DoSA safe-upper-bound pruning ("DoSA：用安全上界减少 Indexer 的完整打分",
 * sections 2, 3.1, 3.2 and 4): per row, seeds fully scored give the threshold
 * tau (K-th best seed score) and the seed top-K; every other visible key gets
 * an upper bound U from R retained heads (omitted positive heads bounded via an
 * anchor and residual norm, section 3.1; omitted negative heads active on at
 * least act_freq_min of n_sample seed samples deducted through the ReLU of
 * their |w|-weighted aggregate, section 3.2) plus a rounding margin; keys with
 * U < tau are dropped; the rest are scored exactly, those with s >= tau merged
 * with the seed top-K and the final K chosen by (score desc, id asc).
 * Output contract: identical, bit for bit, to idx_topk on the same inputs.
 *
 * seed_ids: device [M, seed_ld] int32 (row-relative ids, -1 padded) or NULL:
 * NULL selects the built-in rule -- with key_off == NULL (shared keys) the
 * cold rule of section 4 (four evenly spaced representative queries, keys
 * ranked by how many representative top-K lists hold them, then by their best
 * representative score, then id; n_seed seeds from the common visible prefix),
 * otherwise floor(i L_r / n) for i < n = min(L_r, n_seed).  A row with fewer
 * than K distinct visible seeds, or whose candidate list overflows
 * candidate_capacity, is computed on the unpruned path (row_status 1 resp. 2);
 * so is a row whose bound, evaluated by the planner on n_sample evenly spaced
 * visible keys, predicts more than 1.25 x candidate_capacity candidates: it
 * skips the bound scan (row_status 3).  The output does not depend on which
 * rows take the unpruned path.
 * group_stream != 0 (shared keys, H 16/32/64 with bf16 keys or 16/32 with FP8
 * keys; section 4 of the same page): rows in groups of four; a candidate kept
 * by at least two rows of a group and visible to all four is scored once for
 * the four (one tensor-core tile), the other candidates on their own rows;
 * only scores >= tau are written.  Same output either way.
 * row_status: device [M] int32 or NULL.  stats: device dosa_stats or NULL
 * (counters are added to, not overwritten). */
typedef struct dosa_params {
  int32_t n_seed;             /* seeds per row (12288 for prefill) */
  int32_t retained_heads;     /* R (16 / 20) */
  int32_t n_sample;           /* seed samples for the activation statistics (128) */
  float act_freq_min;         /* 0.5 */
  float margin_gamma;         /* relative rounding margin (2^-10) */
  int32_t candidate_capacity; /* per-row candidate list length */
  int32_t group_stream;       /* 1: shared candidate stream for groups of four rows (shared keys) */
} dosa_params;

typedef struct dosa_stats {
  unsigned long long pairs;       /* visible (query, key) pairs decided */
  unsigned long long seeds;       /* seed pairs fully scored */
  unsigned long long candidates;  /* keys with U >= tau (rescored) */
  unsigned long long survivors;   /* rescored keys with s >= tau */
  unsigned long long fallback_rows;
  unsigned long long skipped_rows;  /* rows whose bound scan was skipped (predicted overflow) */
  unsigned long long group_keys;  /* shared stream: keys scored once for a group of four rows */
  unsigned long long solo_keys;   /* shared stream: candidates scored on their own row */
} dosa_stats;

size_t dosa_topk_workspace_size(const idx_problem* p, int32_t K, const dosa_params* dp, int32_t seed_ld);
idx_status dosa_topk(const idx_problem* p, int32_t K, const dosa_params* dp, const int32_t* seed_ids,
                     int32_t seed_ld, int32_t* out_ids, float* out_scores, int32_t* row_status,
                     dosa_stats* stats, void* ws, size_t ws_bytes, void* stream);

/* Where dosa_topk leaves the intermediate results of the pruned path inside
 * its workspace (after the call completes), for tests and diagnostics: byte
 * offsets from the workspace start.  Layouts, with M rows and H heads:
 *   seed_list   int32 [seed_rows, seed_ld] ascending seed ids (seed_rows = 1
 *               for the shared cold-rule seeds, else M), seed_count int32
 *               [seed_rows];
 *   rep_count   uint32 [rep_ld] (cold rule only): per key, how many
 *               representative top-K lists hold it; rep_scores float32
 *               [n_reps, rep_ld] the representatives' scores, n_reps = the
 *               distinct floor(i (M-1) / 3), i = 0..3;
 *   tau         float32 [M]; status int32 [M] (bit 0: too few seeds, bit 1:
 *               candidate overflow, bit 2: bound scan skipped);
 *   plan_head   int32 [M, H]: r >= 0 the head's position among the retained
 *               heads, 1024 + j an omitted positive head anchored on head j,
 *               -2 an omitted negative head in the aggregate set A, -1 any
 *               other omitted head; plan_beta, plan_dnorm float32 [M, H]: beta
 *               and ||q_h - beta q_j|| (rounded up) of the anchored heads;
 *   wfold       float32 [M, 32] folded retained weights; coef float32 [M] =
 *               c + rounding margin;
 *   qprep       bf16 [M, 32, D] prepared vectors (row r < R: the retained head
 *               at position r, row 31: the aggregate a_A rounded to bf16), or
 *               with group_layout the bound's layout: per group of 8 rows 144
 *               rows, row m's vector r at (m/8)*144 + (m%8)*16 + r and its
 *               aggregate at (m/8)*144 + 128 + m%8.
 * Rows whose status has bit 0 set have no plan.  Returns IDX_ERR_UNSUPPORTED
 * for shapes where dosa_topk runs the unpruned path for every row. */
typedef struct dosa_ws_layout {
  int64_t seed_list, seed_count, rep_count, rep_scores, tau, status;
  int64_t plan_head, plan_beta, plan_dnorm, wfold, coef, qprep;
  int64_t seed_ld, rep_ld, seed_rows;
  int32_t group_layout;
  int32_t reserved;
} dosa_ws_layout;

idx_status dosa_workspace_layout(const idx_problem* p, int32_t K, const dosa_params* dp, int32_t seed_ld,
                                 dosa_ws_layout* out);

/* ----------------------------------------------------------- idx_topk_prior
 * Decode top-K with recent selections as a prior ("DoSA：用安全上界减少 Indexer 的
 * 完整打分": the decode path keeps full scoring; the keys of recent selections
 * set a threshold that shrinks the score write-back and the top-K input).
 * prior_ids: device [M, prior_ld] int32, row m's recent selections (row-
 * relative ids, e.g. the previous steps' top-K; negative, out-of-range and
 * repeated entries are ignored).  With I the remaining ids, n = min(K, L_m)
 * and tau_m the n-th largest current score over I, a row with |I| >= n has its
 * top-K among {s >= tau_m}: every visible key is scored, only those are kept
 * (up to candidate_capacity per row) and ranked.  Rows without such a prior,
 * or whose candidates exceed the capacity, take the unpruned path.  A prior
 * wider than K gives a tighter tau_m.  The output is identical to idx_topk's
 * on the same inputs.
 *   row_status: device [M] int32 or NULL: 0 ranked from candidates, 1 no
 *   usable prior, 2 candidate overflow.  stats: device topk_prior_stats or
 *   NULL (added to).  Tensor-core score shapes only use the prior (others run
 *   the unpruned path for every row). */
typedef struct topk_prior_stats {
  unsigned long long rows_filtered; /* rows ranked from their candidates */
  unsigned long long candidates;    /* candidates of those rows */
  unsigned long long dense_rows;    /* rows that took the unpruned path */
} topk_prior_stats;

size_t idx_topk_prior_workspace_size(const idx_problem* p, int32_t K, int32_t prior_ld,
                                     int32_t candidate_capacity);
idx_status idx_topk_prior(const idx_problem* p, int32_t K, const int32_t* prior_ids, int32_t prior_ld,
                          int32_t candidate_capacity, int32_t* out_ids, float* out_scores, int32_t* row_status,
                          topk_prior_stats* stats, void* ws, size_t ws_bytes, void* stream);
/* idx_topk_prior, recording CUDA events (cudaEvent_t handles, host array of
 * n_events >= 6, created by the caller) on `stream` for profiling: before the
 * prior check, after it, after the prior scores and tau, after the filtered
 * scoring, after the candidate top-K, after the unpruned rows and counters. */
idx_status idx_topk_prior_events(const idx_problem* p, int32_t K, const int32_t* prior_ids, int32_t prior_ld,
                                 int32_t candidate_capacity, int32_t* out_ids, float* out_scores,
                                 int32_t* row_status, topk_prior_stats* stats, void* ws, size_t ws_bytes,
                                 void* const* events, int32_t n_events, void* stream);

/* ------------------------------------------------------------ witness_merge
 * Segment-witness covering pass, in place ("Segment Witnesses", sections
 * "Object" and "Implementation rule and contracts").  Row r of topk_ids
 * (device [rows, topk] int32, row-relative offsets, negative = padding) with
 * context length L_r = context_lens[r] (device int32): S_eff = min(S, L_r);
 * occupancy O = {min(floor(x S_eff / L_r), S-1) : x >= 0 in the row};
 * witnesses e_s = ceil(s L_r / S_eff) for s < S_eff not in O, in ascending s,
 * overwrite slots keep, keep+1, ... up to B = min(max_replacements,
 * topk - keep) slots; further witnesses are dropped, slots without a witness
 * keep their value; rows with L_r <= 0 are unchanged.  The serving form is
 * keep = max(topk - S, 0), max_replacements = S.
 * Checks in order: S == 0 -> no-op (the off switch); S > 64 ->
 * IDX_ERR_SEGMENTS_OUT_OF_RANGE; keep > topk or keep < 0 ->
 * IDX_ERR_KEEP_OUT_OF_RANGE; n_context_lens < rows -> IDX_ERR_ROWS_MISMATCH;
 * B <= 0 or rows == 0 -> no-op.  A refused call leaves the buffer untouched. */
idx_status witness_merge(int32_t* topk_ids, int64_t rows, int32_t topk, const int32_t* context_lens,
                         int64_t n_context_lens, int32_t keep, int32_t num_segments, int32_t max_replacements,
                         void* stream);

/* The witness table alone ("Segment Witnesses", Rust API
 * topology_witness_indices): out device [rows, S] int32, out[r][s] = e_s when
 * segment s < S_eff of row r is unoccupied, else -1.  S == 0 or S > 64 ->
 * IDX_ERR_SEGMENTS_OUT_OF_RANGE; n_context_lens < rows -> ROWS_MISMATCH. */
idx_status witness_indices(const int32_t* learned, int64_t rows, int32_t topk, const int32_t* context_lens,
                           int64_t n_context_lens, int32_t num_segments, int32_t* out, void* stream);

/* ------------------------------------------------------------- block_select
 * MiniMax-M3 block-sparse selection ("ferrox_core/block_sparse.rs":
 * block_sparse_select, select_for_head, dot).  For query i at position
 * query_pos[i] (device int32 >= 0) and KV head h: n_blocks = min(pos/bs + 1,
 * ceil(L/bs)) (0 when bs == 0); blocks [0, init) and [n_blocks - local,
 * n_blocks) are forced; budget = max(top, #forced); every other block scores
 * the max over its positions p < min((b+1) bs, L, pos+1) of the raw dot
 * q.k_p, summed in sequence in f32 (products and sums rounded one by one);
 * the best budget - #forced of them by (score desc, block asc) join the forced
 * ones; the selection is written ascending.
 *   index_q device [Q, n_kv, D] float32, index_k device [L, D] float32.
 *   out device [Q, n_kv, out_width] int32, -1 padded; out_count device
 *   [Q, n_kv] int32 or NULL.  out_width >= max(top, init + local).
 * Block size 0 gives empty selections.
 *
 * With block_size 128, D = 128 and top_blocks <= 512 the block maxima are
 * first computed on the tensor cores: every query row q and key block are
 * rounded to fp16 under exact power-of-two scales (q~ = sigma fp16(q/sigma),
 * k~ = s_b fp16(k/s_b), the largest magnitude in [2^14, 2^15)), multiplied on
 * tcgen05 kind::f16 with fp32 accumulation, and each block maximum A_b
 * carries the certified error bound
 *   e_b = ||q~|| max_p ||k_p - k~_p|| + ||q - q~|| max_p ||k_p||
 *         + 2^-12 ||q|| max_p ||k_p|| (+ 2^-118),
 * the maxima over the block's visible positions, every factor rounded up (the
 * last term covers the fp32 accumulation and the page's sequential sum).  A
 * block whose interval [A_b - e_b, A_b + e_b] lies clear of the selection cut
 * is decided by it, the others are scored in the page's order.  The selection
 * is the same either way.  stats: device block_select_stats or NULL, added to (that route only).
 * Workspace: block_select_workspace_size(), about Q * n_kv * ceil(L/bs) * 8
 * bytes. */
typedef struct block_sparse_config {
  int32_t block_size;   /* 128: also the KV page size */
  int32_t top_blocks;   /* 32 */
  int32_t init_blocks;  /* 1 */
  int32_t local_blocks; /* 2 */
} block_sparse_config;

typedef struct block_select_stats {
  unsigned long long pairs;           /* (query, head) pairs whose selection needed scores */
  unsigned long long blocks_bounded;  /* their non-forced blocks, all bounded */
  unsigned long long blocks_rescored; /* of those, scored in the page's order */
  unsigned long long fallback_pairs;  /* pairs that rescored every non-forced block */
  float max_bound_use;                /* largest |A_b - E_b| / e_b over rescored blocks (max-combined) */
  float reserved;
} block_select_stats;

size_t block_select_workspace_size(int64_t Q, int32_t n_kv, int64_t L, const block_sparse_config* cfg);
idx_status block_select(const float* index_q, const float* index_k, const int32_t* query_pos, int64_t Q,
                        int32_t n_kv, int32_t D, int64_t L, const block_sparse_config* cfg, int32_t* out,
                        int32_t out_width, int32_t* out_count, block_select_stats* stats, void* ws,
                        size_t ws_bytes, void* stream);

/* block_select, recording CUDA events (cudaEvent_t handles, host array of
 * n_events >= 6, each created by the caller) on `stream` between its kernels,
 * for profiling: events[0] before the first kernel; on the tensor-core route
 * events[1..5] after the prep, block-maxima, classify, rescoring and resolve
 * kernels; on the CUDA-core route only events[0] and events[5].  Same
 * arguments and result as block_select otherwise. */
idx_status block_select_events(const float* index_q, const float* index_k, const int32_t* query_pos, int64_t Q,
                               int32_t n_kv, int32_t D, int64_t L, const block_sparse_config* cfg, int32_t* out,
                               int32_t out_width, int32_t* out_count, block_select_stats* stats, void* ws,
                               size_t ws_bytes, void* const* events, int32_t n_events, void* stream);

/* --------------------------------------------------------- block_positions
 * The positions a block selection covers ("ferrox_core/block_sparse.rs":
 * positions_of_blocks): row r = i * n_kv + h (query i, KV head h) lists
 * blocks[r * W + j] for j < counts[r] (counts NULL: all W); negative entries
 * are ignored.  Its output is the union over those blocks b of the positions
 * [b * block_size, min((b + 1) * block_size, L, query_pos[i] + 1)),
 * ascending, without repeats -- the block_select output of one row maps to
 * the positions sparse attention reads.
 *   blocks device [Q * n_kv, W] int32 (W <= IDX_MAX_K); counts device
 *   [Q * n_kv] int32 or NULL; query_pos device [Q] int32.
 *   out device [Q * n_kv, out_width] int32, -1 padded, out_width >= W *
 *   block_size (every block covers at most block_size positions);
 *   out_count device [Q * n_kv] int32 or NULL.
 * Block size 0 gives empty rows. */
idx_status block_positions(const int32_t* blocks, const int32_t* counts, int64_t Q, int32_t n_kv, int32_t W,
                           const int32_t* query_pos, int64_t L, int32_t block_size, int32_t* out, int32_t out_width,
                           int32_t* out_count, void* stream);

/* ------------------------------------------------------ block_select_static
 * block_select for callers that cannot allocate device memory: code that runs
 * inside a host framework which owns every device allocation (and offers no
 * allocator handle to plug-ins), or on a latency-critical path where a
 * cudaMalloc could stall on the driver or fail under memory pressure.  No
 * source page has a counterpart of this entry point; it is a deployment
 * convenience with the same result as block_select.
 *
 * Identical arguments and output to block_select, minus (stats, ws,
 * ws_bytes); every block score is computed in the page's order.  The
 * per-(query, head, block) scratch lives in a fixed device array inside the
 * library, 2^23 words (32 MiB), which every GPU that loads the library holds
 * until the process exits.  Calls with Q * n_kv * ceil(L / block_size) above
 * 2^23 are refused with IDX_ERR_WORKSPACE_TOO_SMALL before anything runs.
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  Nothing is allocated: no cudaMalloc, cudaFree or allocating
 * library routine is called.  All calls share the one array and it keeps the
 * previous call's contents (every entry a call reads it has written first, so
 * nothing needs clearing); calls that overlap on the GPU race on it, so
 * serialise them (one stream, or events). */
idx_status block_select_static(const float* index_q, const float* index_k, const int32_t* query_pos, int64_t Q,
                               int32_t n_kv, int32_t D, int64_t L, const block_sparse_config* cfg, int32_t* out,
                               int32_t out_width, int32_t* out_count, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* IDX_H_ */
