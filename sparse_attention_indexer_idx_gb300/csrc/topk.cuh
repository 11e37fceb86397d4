// Exact top-K of one row per thread block, under the total order
// (key desc, id asc) -- the final selection of the indexer
// ("DoSA：用安全上界减少 Indexer 的完整打分", section 1 and the note after
// section 2: the original scorer decides, one consistent total order for ties).
//
// A row is read through an accessor (n(), key(i), id(i)); keys are ordered
// uint32 values (see score_key), ids distinct non-negative int32.  Method:
//   1. radix select on the key, 11+11+10 bits, finds the K-th largest key T
//      and how many elements equal to T are needed (need);
//   2. when more than `need` elements tie at T, a second radix select on the
//      id picks the `need` smallest ids among them;
//   3. the K winners are gathered into shared memory as 64-bit composites
//      (key << 32 | ~id) and bitonic-sorted descending (or by id ascending).
// Every element is read once per radix pass straight from global memory (L2
// for rows produced just before).
#pragma once

#include "common.cuh"

namespace idx {

constexpr int kTopkBins = 2048;

template <int NT>
struct TopkShared {
  uint32_t hist[kTopkBins];
  uint32_t warp_sums[NT / 32];
  uint32_t found_bin;
  uint32_t found_above;
  uint32_t count;
};

// Suffix search over hist (bins ordered high to low): finds the bin b such that
// (#elements in bins > b) < remaining <= (#elements in bins >= b).
template <int NT>
__device__ __forceinline__ void topk_find_bin(TopkShared<NT>& sh, uint32_t nbins, uint32_t remaining) {
  constexpr int PER = kTopkBins / NT;
  const int t = threadIdx.x;
  uint32_t local[PER];
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    int rank = t * PER + j;                 // rank 0 = highest bin
    int bin = (int)nbins - 1 - rank;
    local[j] = (bin >= 0) ? sh.hist[bin] : 0u;
    sum += local[j];
  }
  // exclusive scan of `sum` over threads in order
  uint32_t incl = sum;
  const int lane = t & 31, wid = t >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sh.warp_sums[wid] = incl;
  __syncthreads();
  uint32_t warp_off = 0;
  for (int w = 0; w < wid; ++w) warp_off += sh.warp_sums[w];
  uint32_t run = warp_off + incl - sum;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    int rank = t * PER + j;
    int bin = (int)nbins - 1 - rank;
    if (bin >= 0 && run < remaining && run + local[j] >= remaining) {
      sh.found_bin = (uint32_t)bin;
      sh.found_above = run;
    }
    run += local[j];
  }
  __syncthreads();
}

// Radix select of the `want`-th largest value of f(i) over the elements that
// pass `filter`; returns the value and sets *above = number strictly greater.
template <int NT, class Row, class KeyFn, class Filter>
__device__ uint32_t topk_radix_select(TopkShared<NT>& sh, const Row& row, int n, uint32_t want, KeyFn f,
                                      Filter filter, uint32_t* above_out, uint32_t* eq_out) {
  uint32_t prefix = 0, mask = 0, remaining = want, eq = 0;
  const int shifts[3] = {21, 10, 0};
  const uint32_t widths[3] = {11, 11, 10};
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const uint32_t dmask = (1u << widths[pass]) - 1u;
    for (int b = threadIdx.x; b < kTopkBins; b += NT) sh.hist[b] = 0;
    __syncthreads();
    // eight elements per thread and iteration, their loads in flight together
    for (int i0 = threadIdx.x; i0 < n; i0 += 8 * NT) {
      uint32_t kk[8];
      bool on[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * NT;
        on[u] = i < n && filter(i);
        kk[u] = on[u] ? f(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (on[u] && (kk[u] & mask) == prefix) atomicAdd(&sh.hist[(kk[u] >> shift) & dmask], 1u);
    }
    __syncthreads();
    topk_find_bin<NT>(sh, dmask + 1u, remaining);
    const uint32_t bin = sh.found_bin;
    remaining -= sh.found_above;
    eq = sh.hist[bin];
    prefix |= bin << shift;
    mask |= dmask << shift;
    __syncthreads();
  }
  *above_out = want - remaining;
  *eq_out = eq;
  return prefix;
}

// Sort `n` (power of two) 64-bit values in shared memory, descending.
template <int NT>
__device__ void bitonic_sort_desc(uint64_t* v, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < (n >> 1); t += NT) {
        int lo = 2 * t - (t & (stride - 1));
        int hi = lo + stride;
        bool desc = ((lo & size) == 0);
        uint64_t a = v[lo], b = v[hi];
        if ((a < b) == desc) {
          v[lo] = b;
          v[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

// Top-K of one row.  sel: shared scratch of at least next_pow2(K) uint64.
// Writes out_ids[0..K) (and out_scores if non-null, via key_score), padded
// with -1 / -inf.  by_id: order the output by id ascending instead of by
// (key desc, id asc).  Returns the number of real entries.
template <int NT, class Row>
__device__ int block_topk(TopkShared<NT>& sh, uint64_t* sel, const Row& row, int K, int32_t* out_ids,
                          float* out_scores, bool by_id) {
  const int n = row.n();
  auto key_of = [&](int i) { return row.key(i); };
  auto all = [&](int) { return true; };
  uint32_t T = 0, need = 0, I = 0;
  bool take_all = (n <= K);
  bool all_ties = true;
  if (!take_all) {
    uint32_t above, eq;
    T = topk_radix_select<NT>(sh, row, n, (uint32_t)K, key_of, all, &above, &eq);
    need = (uint32_t)K - above;
    if (eq != need) {
      all_ties = false;
      uint32_t above2, eq2;
      auto idk = [&](int i) { return id_key(row.id(i)); };
      auto is_tie = [&](int i) { return row.key(i) == T; };
      I = topk_radix_select<NT>(sh, row, n, need, idk, is_tie, &above2, &eq2);
    }
  }
  if (threadIdx.x == 0) sh.count = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += NT) {
    uint32_t k = row.key(i);
    bool take = take_all || k > T || (k == T && (all_ties || id_key(row.id(i)) >= I));
    if (take) {
      uint32_t pos = atomicAdd(&sh.count, 1u);
      if (pos < (uint32_t)K) {
        uint32_t lo = by_id ? (0xffffffffu - (uint32_t)row.id(i)) : id_key(row.id(i));
        uint32_t hi = by_id ? 0u : k;
        // by_id: sort on ~id descending == id ascending; keep key in a side slot
        sel[pos] = by_id ? (((uint64_t)lo << 32) | k) : (((uint64_t)hi << 32) | lo);
      }
    }
  }
  __syncthreads();
  const int cnt = (int)min(sh.count, (uint32_t)K);
  int P = 1;
  while (P < cnt) P <<= 1;
  for (int i = cnt + threadIdx.x; i < P; i += NT) sel[i] = 0ull;
  __syncthreads();
  if (P > 1) bitonic_sort_desc<NT>(sel, P);
  for (int j = threadIdx.x; j < K; j += NT) {
    int32_t id = -1;
    float s = -__int_as_float(0x7f800000);
    if (j < cnt) {
      uint64_t c = sel[j];
      if (by_id) {
        id = (int32_t)(0xffffffffu - (uint32_t)(c >> 32));
        s = key_score((uint32_t)c);
      } else {
        id = key_id((uint32_t)c);
        s = key_score((uint32_t)(c >> 32));
      }
    }
    out_ids[j] = id;
    if (out_scores) out_scores[j] = s;
  }
  __syncthreads();
  return cnt;
}

// ----------------------------------------------------------- row accessors --
struct DenseScoreRow {
  const float* s;
  int len;
  __device__ int n() const { return len; }
  __device__ uint32_t key(int i) const { return score_key(__ldg(s + i)); }
  __device__ int32_t id(int i) const { return i; }
};

struct PairRow {  // explicit (score, id) list
  const float* s;
  const int32_t* ids;
  int len;
  __device__ int n() const { return len; }
  __device__ uint32_t key(int i) const { return score_key(s[i]); }
  __device__ int32_t id(int i) const { return ids[i]; }
};

}  // namespace idx
