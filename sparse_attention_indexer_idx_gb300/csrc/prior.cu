// DSA decode top-K with recent selections as a prior ("DoSA：用安全上界减少 Indexer
// 的完整打分": the decode path keeps full FP8 scoring; the keys of recent
// selections set a threshold, so the score write-back and the top-K input shrink).
//
// For row m, let I be the prior ids (recent selections: the previous steps'
// top-K, any number of them) that are still visible and distinct, n = min(K,
// L_m), and tau_m the n-th largest current score over I.  If |I| >= n, at
// least n keys score >= tau_m, so the current top-K (score desc, id asc) lies
// within {k : s(k) >= tau_m}; the wider the prior, the tighter tau_m:
//  1. prior_check_kernel: the distinct visible prior ids of each row (a
//     per-row bitmap in shared memory) and whether the row can use them;
//  2. their exact scores (the gathered-key score kernel: the same MMA shape and
//     epilogue chain as the dense scores, so the same bits) and tau_m (radix
//     select of the n-th largest);
//  3. every visible key scored once more in full (kFilter: the dense score
//     kernel whose epilogue keeps only s >= tau_m as (id, score));
//  4. top-K over those candidates (ids mapped, so ties break by key id);
//  5. rows without a usable prior, or whose candidates overflowed the list,
//     take the dense path (all scores, top-K), masked to those rows.
// The output is bit-identical to idx_topk on the same inputs.
#include "internal.h"

namespace idx {

cudaError_t launch_score_filter(const idx_problem& p, const float* tau, int32_t* cand, float* cand_sc,
                                int32_t* cand_cnt, int64_t cap, int32_t* status, const int32_t* row_mask,
                                cudaStream_t st);

constexpr int kPrThreads = 256;
constexpr int64_t kPrMaxBitmapKeys = (int64_t)1 << 20;   // 128 KB of shared bitmap

struct PriorWs {
  int32_t* plist;     // [M, P] distinct visible prior ids
  int32_t* pcnt;      // [M]
  float* psc;         // [M, P] their scores
  float* tau;         // [M]
  int32_t* mask;      // [M] 1: the row has a usable prior
  int32_t* okmask;    // [M] 1: the row's top-K comes from its candidates
  int32_t* fbmask;    // [M] 1: the row takes the dense path
  int32_t* cand;      // [M, cap]
  float* cand_sc;     // [M, cap]
  int32_t* cand_cnt;  // [M]
  int32_t* cand_n;    // [M] candidates used (0 on dense rows)
  int32_t* status;    // [M] bit 1: candidate overflow
  float* fb_scores;   // [M, ldmax]
  char* tk_ws;
};

static PriorWs prior_carve(void* base, const idx_problem& p, int K, int P, int64_t cap, size_t* used) {
  WsCarver c(base);
  const int64_t M = p.M, ld = p.max_key_len > 0 ? p.max_key_len : 1;
  PriorWs w;
  w.plist = c.take<int32_t>((size_t)(M * P));
  w.pcnt = c.take<int32_t>((size_t)M);
  w.psc = c.take<float>((size_t)(M * P));
  w.tau = c.take<float>((size_t)M);
  w.mask = c.take<int32_t>((size_t)M);
  w.okmask = c.take<int32_t>((size_t)M);
  w.fbmask = c.take<int32_t>((size_t)M);
  w.cand = c.take<int32_t>((size_t)(M * cap));
  w.cand_sc = c.take<float>((size_t)(M * cap));
  w.cand_cnt = c.take<int32_t>((size_t)M);
  w.cand_n = c.take<int32_t>((size_t)M);
  w.status = c.take<int32_t>((size_t)M);
  w.fb_scores = c.take<float>((size_t)(M * ld));
  const size_t a = topk_dense_ws(M, (int)cap, K), b = topk_dense_ws(M, p.max_key_len, K);
  w.tk_ws = c.take<char>(a > b ? a : b);
  if (used) *used = c.used + 256;
  return w;
}

size_t topk_prior_ws(const idx_problem& p, int K, int P, int64_t cap) {
  size_t used = 0;
  prior_carve(nullptr, p, K, P, cap, &used);
  return used;
}

// One CTA per row: the distinct visible prior ids (any order), and whether they
// bound the row's top-K from below.  Rows longer than the bitmap take the
// dense path.  Resets the row's candidate counter and status.
__global__ void __launch_bounds__(kPrThreads) prior_check_kernel(idx_problem p, const int32_t* __restrict__ prior,
                                                                 int P, int K, PriorWs w, int use_bitmap) {
  extern __shared__ uint32_t bits[];
  __shared__ int n_s;
  const int64_t m = blockIdx.x;
  int64_t off;
  int len;
  row_extent(p, m, &off, &len);
  const int nwords = (int)((p.max_key_len + 31) / 32);
  if (threadIdx.x == 0) n_s = 0;
  if (use_bitmap)
    for (int i = threadIdx.x; i < nwords; i += kPrThreads) bits[i] = 0u;
  __syncthreads();
  if (use_bitmap) {
    for (int j = threadIdx.x; j < P; j += kPrThreads) {
      const int32_t id = prior[m * P + j];
      if (id < 0 || id >= len) continue;
      const uint32_t bit = 1u << (id & 31);
      const uint32_t old = atomicOr(&bits[id >> 5], bit);
      if (old & bit) continue;   // a repeat
      w.plist[m * P + atomicAdd(&n_s, 1)] = id;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int n = n_s;
    const int need = K < len ? K : len;
    w.pcnt[m] = n;
    w.mask[m] = (use_bitmap && len > 0 && n >= need) ? 1 : 0;
    w.cand_cnt[m] = 0;
    w.status[m] = 0;
  }
}

// One CTA per row: tau = the n-th largest score of the row's prior ids, n =
// min(K, L_m): four 8-bit radix passes over the order-preserving keys.
__global__ void __launch_bounds__(kPrThreads) prior_tau_kernel(idx_problem p, int P, int K, PriorWs w) {
  __shared__ int hist[256];
  __shared__ int s_digit, s_above;
  const int64_t m = blockIdx.x;
  if (!w.mask[m]) return;
  int64_t off;
  int len;
  row_extent(p, m, &off, &len);
  const int n = w.pcnt[m];
  int need = K < len ? K : len;   // 1 <= need <= n (the mask says so)
  const float* sc = w.psc + m * (int64_t)P;
  uint32_t prefix = 0, pmask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kPrThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kPrThreads) {
      const uint32_t k = score_key(sc[i]);
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l holds digits 255 - 8l - j (descending); the first digit whose
      // running count from the top reaches `need`
      const int lane = threadIdx.x;
      int c[8], csum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        csum += c[j];
      }
      int incl = csum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
      const int fl = hit ? __ffs(hit) - 1 : 31;
      if (lane == fl) {
        int run = incl - csum, d = 255 - 8 * lane - 7;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= need) {
            d = 255 - 8 * lane - j;
            break;
          }
          run += c[j];
        }
        s_digit = d;
        s_above = run;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)s_digit << shift;
    pmask |= 255u << shift;
    need -= s_above;
    __syncthreads();
  }
  if (threadIdx.x == 0) w.tau[m] = key_score(prefix);
}

// Per row: candidates or the dense path, and the candidate count the top-K reads.
__global__ void prior_route_kernel(int64_t M, int64_t cap, PriorWs w) {
  const int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const bool ok = w.mask[m] && !(w.status[m] & 2);
  w.okmask[m] = ok ? 1 : 0;
  w.fbmask[m] = ok ? 0 : 1;
  const int32_t c = w.cand_cnt[m];
  w.cand_n[m] = ok ? (c < cap ? c : (int32_t)cap) : 0;
}

// row_status (0 candidates, 1 no usable prior, 2 candidate overflow) and the counters.
__global__ void prior_stats_kernel(int64_t M, PriorWs w, int32_t* row_status, topk_prior_stats* stats) {
  const int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const int st = w.okmask[m] ? 0 : (w.mask[m] ? 2 : 1);
  if (row_status) row_status[m] = st;
  if (stats) {
    if (st == 0) {
      atomicAdd(&stats->rows_filtered, 1ull);
      atomicAdd(&stats->candidates, (unsigned long long)w.cand_n[m]);
    } else {
      atomicAdd(&stats->dense_rows, 1ull);
    }
  }
}

cudaError_t launch_topk_prior(const idx_problem& p, int K, const int32_t* prior, int P, int64_t cap,
                              int32_t* out_ids, float* out_scores, int32_t* row_status, topk_prior_stats* stats,
                              void* ws, cudaStream_t st, const cudaEvent_t* ev) {
  const int64_t M = p.M;
  if (M <= 0) return cudaSuccess;
  PriorWs w = prior_carve(ws, p, K, P, cap, nullptr);
  const int64_t ld = p.max_key_len > 0 ? p.max_key_len : 1;
  cudaError_t e;
  // ev (optional, 6 events): before the prior check, after it, after tau, after the
  // filtered scoring, after the candidate top-K, after the unpruned rows and the counters
  auto mark = [&](int i) { return ev && ev[i] ? cudaEventRecord(ev[i], st) : cudaSuccess; };
  if ((e = mark(0)) != cudaSuccess) return e;
  // the filter runs on the tensor-core score kernel; other shapes take the dense path for every row
  const int use_bitmap = score_uses_tensor_cores(p) && p.max_key_len <= kPrMaxBitmapKeys ? 1 : 0;
  const size_t bsm = use_bitmap ? (size_t)((p.max_key_len + 31) / 32) * 4 : 0;
  if (bsm > 48 * 1024 &&
      (e = cudaFuncSetAttribute(prior_check_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bsm)) !=
          cudaSuccess)
    return e;
  prior_check_kernel<<<(unsigned)M, kPrThreads, bsm, st>>>(p, prior, P, K, w, use_bitmap);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = mark(1)) != cudaSuccess) return e;
  if (use_bitmap) {
    if ((e = launch_score_gather(p, w.plist, w.pcnt, P, w.psc, P, w.mask, st)) != cudaSuccess) return e;
    prior_tau_kernel<<<(unsigned)M, kPrThreads, 0, st>>>(p, P, K, w);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = mark(2)) != cudaSuccess) return e;
  if (use_bitmap &&
      (e = launch_score_filter(p, w.tau, w.cand, w.cand_sc, w.cand_cnt, cap, w.status, w.mask, st)) != cudaSuccess)
    return e;
  if ((e = mark(3)) != cudaSuccess) return e;
  prior_route_kernel<<<(unsigned)((M + 255) / 256), 256, 0, st>>>(M, cap, w);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (use_bitmap &&
      (e = launch_topk_dense(w.cand_sc, cap, w.cand_n, nullptr, M, (int)cap, K, out_ids, out_scores, w.tk_ws, st,
                             w.cand, cap, w.okmask)) != cudaSuccess)
    return e;
  if ((e = mark(4)) != cudaSuccess) return e;
  // the dense path, only for the rows that need it
  if ((e = launch_score(p, w.fb_scores, ld, st, w.fbmask)) != cudaSuccess) return e;
  if ((e = launch_topk_dense(w.fb_scores, ld, nullptr, &p, M, p.max_key_len, K, out_ids, out_scores, w.tk_ws, st,
                             nullptr, 0, w.fbmask)) != cudaSuccess)
    return e;
  prior_stats_kernel<<<(unsigned)((M + 255) / 256), 256, 0, st>>>(M, w, row_status, stats);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return mark(5);
}

}  // namespace idx
