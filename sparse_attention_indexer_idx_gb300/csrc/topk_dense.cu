// Exact top-K of dense score rows, under (score desc, key id asc)
// ("DoSA：用安全上界减少 Indexer 的完整打分", section 1 and the note after
// section 2: selection by the original scorer with one total order for ties).
//
// Two passes over a row's scores, which are read once from memory:
//   filter  one thread block per (row, 16384 scores) takes a row threshold T
//           from 1024 evenly spaced samples of the row (the same in every block
//           of the row) and writes the keys >= T, as 64-bit composites
//           key << 32 | ~id whose descending order is exactly (score desc, id
//           asc), and their count to the chunk's own slots;
//   finish  one thread block per row bucket-sorts the ~1.5-2.5 K candidates at
//           once and writes the first K.  A bucket with heavy ties sends the
//           candidates through two radix selects (key, then id among ties) that
//           cut them to exactly K and a register bitonic sort; a threshold that
//           missed (too few or too many candidates) sends the row through an
//           exact radix select over its scores.
#include "internal.h"
#include "topk.cuh"

namespace idx {

constexpr int TK_NT = 1024;
constexpr int TK_CH = 32768;
constexpr int TK_CAP = 8192;

// Shared memory of the finish pass: candidates, and a scratch area whose lower
// half takes sorted / selected composites and upper half the bucket arrays.
struct TkShared {
  uint32_t keys[TK_CH];       // scratch (128 KB)
  uint64_t cand[TK_CAP];
  uint32_t hist[kTopkBins];
  uint32_t red[TK_NT / 32];
  uint32_t found_bin;
  uint32_t found_above;
  uint32_t kmin, kmax, bmax, kend;
};

__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, uint32_t* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  uint32_t t = 0;
#pragma unroll
  for (int w = 0; w < TK_NT / 32; ++w) t += red[w];
  return t;
}

// Adds one to hist[bin] for every lane with `active` set, one shared-memory
// atomic per distinct bin of the warp (lanes with equal bins are grouped by
// match.any): rows with thousands of equal scores would otherwise serialise
// their atomics on one address.  Every lane of the warp must call it.
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, uint32_t bin, bool active) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const unsigned peers = __match_any_sync(act, bin);
  if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

// Exclusive prefix sum over the block (thread order); *total = block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* red, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();
  if (lane == 31) red[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    uint32_t x = red[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += u;
    }
    red[lane] = x;
  }
  __syncthreads();
  *total = red[31];
  return (wid ? red[wid - 1] : 0u) + incl - v;
}

template <class T>
__device__ void bitonic_desc(T* v, int n, int nt) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < (n >> 1); t += nt) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const T a = v[lo], b = v[hi];
        if ((a < b) == desc) {
          v[lo] = b;
          v[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

// ---- register-resident bitonic sort --------------------------------------
// S = TK_NT * EPT values, thread t holding elements t*EPT .. t*EPT+EPT-1.
// Strides below EPT are swaps inside a thread, strides below 32*EPT are warp
// shuffles, only the larger ones go through shared memory (with barriers).
template <class T>
__device__ __forceinline__ T shfl_xor_t(T v, int m) {
  if constexpr (sizeof(T) == 8) {
    uint32_t lo = (uint32_t)v, hi = (uint32_t)(v >> 32);
    lo = __shfl_xor_sync(0xffffffffu, lo, m);
    hi = __shfl_xor_sync(0xffffffffu, hi, m);
    return ((T)hi << 32) | lo;
  } else {
    return (T)__shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  }
}

template <class T>
__device__ __forceinline__ T cmpx(T a, T o, int e, int stride, int size) {
  // keep the larger value when (lower half) == (descending block)
  const bool keep_max = (((e & stride) == 0) == ((e & size) == 0));
  return ((a < o) == keep_max) ? o : a;
}

template <int EPT, int STRIDE, class T>
__device__ __forceinline__ void thread_stage(T (&v)[EPT], int size) {
  T n[EPT];
#pragma unroll
  for (int r = 0; r < EPT; ++r) n[r] = cmpx(v[r], v[r ^ STRIDE], threadIdx.x * EPT + r, STRIDE, size);
#pragma unroll
  for (int r = 0; r < EPT; ++r) v[r] = n[r];
}

template <int EPT, class T>
__device__ void reg_bitonic_desc(T (&v)[EPT], T* xchg) {
  constexpr int S = TK_NT * EPT;
  const int tid = threadIdx.x;
#pragma unroll 1
  for (int size = 2; size <= S; size <<= 1) {
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32 * EPT) {
#pragma unroll
        for (int r = 0; r < EPT; ++r) xchg[tid * EPT + r] = v[r];
        __syncthreads();
#pragma unroll
        for (int r = 0; r < EPT; ++r) {
          const int e = tid * EPT + r;
          v[r] = cmpx(v[r], xchg[e ^ stride], e, stride, size);
        }
        __syncthreads();
      } else if (stride >= EPT) {
        const int lx = stride / EPT;
#pragma unroll
        for (int r = 0; r < EPT; ++r) v[r] = cmpx(v[r], shfl_xor_t(v[r], lx), tid * EPT + r, stride, size);
      } else {
        if constexpr (EPT > 8) { if (stride == 8) thread_stage<EPT, 8>(v, size); }
        if constexpr (EPT > 4) { if (stride == 4) thread_stage<EPT, 4>(v, size); }
        if constexpr (EPT > 2) { if (stride == 2) thread_stage<EPT, 2>(v, size); }
        if constexpr (EPT > 1) { if (stride == 1) thread_stage<EPT, 1>(v, size); }
      }
    }
  }
}

// Sorts buf[0..S) descending (S a power of two, >= TK_NT) through registers.
template <int EPT>
__device__ void sort_smem_via_regs(uint64_t* buf) {
  uint64_t v[EPT];
#pragma unroll
  for (int r = 0; r < EPT; ++r) v[r] = buf[threadIdx.x * EPT + r];
  __syncthreads();
  reg_bitonic_desc<EPT>(v, buf);
  __syncthreads();
#pragma unroll
  for (int r = 0; r < EPT; ++r) buf[threadIdx.x * EPT + r] = v[r];
  __syncthreads();
}

__device__ void sort_candidates(uint64_t* buf, int S) {
  switch (S / TK_NT) {
    case 0: bitonic_desc<uint64_t>(buf, S, TK_NT); break;
    case 1: sort_smem_via_regs<1>(buf); break;
    case 2: sort_smem_via_regs<2>(buf); break;
    case 4: sort_smem_via_regs<4>(buf); break;
    default: sort_smem_via_regs<8>(buf); break;
  }
}

__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* red, uint32_t* total);

// Sorts the n nonzero, distinct composites src[0..n) descending: one bucket
// pass into dst -- 8192 buckets spread evenly over [min key, max key] (a
// monotone map; bucket 0 holds the largest keys) -- then every element finds
// its place inside its bucket by counting the larger ones there and is written
// back to src.  The bucket arrays live in the upper half of the key area,
// which every caller leaves free (src and dst hold at most 8192 composites
// each and sit elsewhere).  have_range: sh.kmin / sh.kmax already hold the
// keys' minimum and maximum.  Only the first `limit` places are needed:
// buckets that start at or after it are left out of the scatter and the
// placement.  Returns false, with src untouched, when a bucket would hold more
// than kBucketMax entries (heavy ties): the caller then uses the bitonic
// network.
constexpr uint32_t kBucketMax = 256;
constexpr int kSortBuckets = 8192;
__device__ bool bucket_sort_desc(TkShared& sh, uint64_t* src, int n, uint64_t* dst, bool have_range = false,
                                 int limit = 0x7fffffff) {
  const int tid = threadIdx.x;
  uint32_t* bh = sh.keys + TK_CH / 2;          // count, then cursor / end, per bucket
  uint32_t* bs = bh + kSortBuckets;           // first slot per bucket
  static_assert(TK_CH / 2 + 2 * kSortBuckets <= TK_CH, "bucket arrays");
  constexpr int PER = kSortBuckets / TK_NT;   // buckets per thread (contiguous)
  static_assert(PER == 8, "two 16-byte vectors per thread");
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  reinterpret_cast<uint4*>(bh)[2 * tid] = z;
  reinterpret_cast<uint4*>(bh)[2 * tid + 1] = z;
  if (!have_range) {
    if (tid == 0) {
      sh.kmin = 0xffffffffu;
      sh.kmax = 0u;
    }
    __syncthreads();
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (int i = tid; i < n; i += TK_NT) {
      const uint32_t k = (uint32_t)(src[i] >> 32);
      mn = min(mn, k);
      mx = max(mx, k);
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if ((tid & 31) == 0) {
      atomicMin(&sh.kmin, mn);
      atomicMax(&sh.kmax, mx);
    }
  }
  if (tid == 0) {
    sh.bmax = 0u;
    sh.kend = (uint32_t)n;
  }
  __syncthreads();
  const uint32_t kmin = sh.kmin;
  const float scale = (float)kSortBuckets / ((float)(sh.kmax - kmin) + 1.0f);
  auto bucket = [&](uint64_t v) {
    uint32_t b = (uint32_t)((float)((uint32_t)(v >> 32) - kmin) * scale);
    b = b < (uint32_t)kSortBuckets ? b : (uint32_t)kSortBuckets - 1u;
    return (uint32_t)kSortBuckets - 1u - b;   // largest keys first
  };
  for (int i = tid; i < n; i += TK_NT) atomicAdd(&bh[bucket(src[i])], 1u);
  __syncthreads();
  // exclusive scan over the buckets in order; the largest per-thread range
  const uint4 c0 = reinterpret_cast<const uint4*>(bh)[2 * tid];
  const uint4 c1 = reinterpret_cast<const uint4*>(bh)[2 * tid + 1];
  const uint32_t cnt8[PER] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  uint32_t sum = 0, big = 0;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    sum += cnt8[q];
    big = max(big, cnt8[q]);
  }
  uint32_t total;
  uint32_t run = block_excl_scan(sum, sh.red, &total);
  big = __reduce_max_sync(0xffffffffu, big);
  if ((tid & 31) == 0) atomicMax(&sh.bmax, big);
  const uint32_t lim = (uint32_t)(limit < n ? limit : n);
  uint32_t st8[PER], kend = 0xffffffffu;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    st8[q] = run;
    if (run >= lim && cnt8[q]) kend = min(kend, run);   // first bucket left out
    run += cnt8[q];
  }
  kend = __reduce_min_sync(0xffffffffu, kend);
  if ((tid & 31) == 0 && kend != 0xffffffffu) atomicMin(&sh.kend, kend);
  reinterpret_cast<uint4*>(bs)[2 * tid] = make_uint4(st8[0], st8[1], st8[2], st8[3]);
  reinterpret_cast<uint4*>(bs)[2 * tid + 1] = make_uint4(st8[4], st8[5], st8[6], st8[7]);
  reinterpret_cast<uint4*>(bh)[2 * tid] = make_uint4(st8[0], st8[1], st8[2], st8[3]);   // scatter cursors
  reinterpret_cast<uint4*>(bh)[2 * tid + 1] = make_uint4(st8[4], st8[5], st8[6], st8[7]);
  __syncthreads();
  if (sh.bmax > kBucketMax) return false;
  for (int i = tid; i < n; i += TK_NT) {
    const uint64_t v = src[i];
    const uint32_t b = bucket(v);
    if (bs[b] >= lim) continue;
    const uint32_t pos = atomicAdd(&bh[b], 1u);
    dst[pos] = v;
  }
  __syncthreads();
  // place: bucket start + the number of larger elements in the bucket; the
  // scattered elements fill dst[0, kend)
  const int used = (int)sh.kend;
  for (int i = tid; i < used; i += TK_NT) {
    const uint64_t v = dst[i];
    const uint32_t b = bucket(v);
    const int b0 = (int)bs[b], b1 = (int)bh[b];
    int r = b0;
    for (int q = b0; q < b1; ++q) r += dst[q] > v ? 1 : 0;
    src[r] = v;
  }
  __syncthreads();
  return true;
}

// Descending order of src[0..cnt) (nonzero, distinct), in place (dst is
// scratch): the bucket pass, or, when the buckets are too uneven, the bitonic
// network over src zero-padded to P.
__device__ const uint64_t* order_desc(TkShared& sh, uint64_t* src, int cnt, int P, uint64_t* dst) {
  if (cnt <= 1) return src;
  if (bucket_sort_desc(sh, src, cnt, dst)) return src;
  for (int i = cnt + threadIdx.x; i < P; i += TK_NT) src[i] = 0ull;
  __syncthreads();
  sort_candidates(src, P);
  return src;
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int32_t id) {
  return ((uint64_t)key << 32) | id_key(id);
}

template <class F, class Flag>
__device__ uint32_t smem_radix_select(TkShared& sh, int cn, uint32_t want, F f, Flag flag, uint32_t* above_out,
                                      uint32_t* eq_out);
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* red, uint32_t* total);

// Keeps exactly the K largest of the n nonzero composites src[0..n) (n >= K),
// appending them to dst (unsorted).  Two radix selects: the K-th key, then,
// among the keys equal to it, the ids.
__device__ void select_exact_k(TkShared& sh, const uint64_t* src, int n, int K, uint64_t* dst) {
  uint32_t above, eq;
  auto hi = [&](int i) { return (uint32_t)(src[i] >> 32); };
  auto real = [&](int i) { return src[i] != 0ull; };
  const uint32_t KT = smem_radix_select(sh, n, (uint32_t)K, hi, real, &above, &eq);
  const uint32_t need = (uint32_t)K - above;
  uint32_t IT = 0;   // with no surplus ties every element at KT is taken
  if (eq != need) {
    auto lo = [&](int i) { return (uint32_t)src[i]; };
    auto tie = [&](int i) { return src[i] != 0ull && (uint32_t)(src[i] >> 32) == KT; };
    uint32_t above2, eq2;
    IT = smem_radix_select(sh, n, need, lo, tie, &above2, &eq2);
  }
  auto take = [&](int i) {
    const uint64_t v = src[i];
    const uint32_t k = (uint32_t)(v >> 32);
    return v != 0ull && (k > KT || (k == KT && (uint32_t)v >= IT));
  };
  uint32_t local = 0;
  for (int i = threadIdx.x; i < n; i += TK_NT) local += take(i) ? 1u : 0u;
  uint32_t total;
  uint32_t off = block_excl_scan(local, sh.red, &total);
  for (int i = threadIdx.x; i < n; i += TK_NT)
    if (take(i)) dst[off++] = src[i];
  __syncthreads();
}

// Suffix search over sh.hist[0..nb) (bins high to low): the bin b with
// (#in bins > b) < remaining <= (#in bins >= b) -> sh.found_bin/found_above.
template <class SH>
__device__ __forceinline__ void hist_suffix_find(SH& sh, int nb, uint32_t remaining) {
  constexpr int PER = kTopkBins / TK_NT;
  uint32_t loc[PER], sum = 0;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int bin = nb - 1 - (threadIdx.x * PER + q);
    loc[q] = bin >= 0 ? sh.hist[bin] : 0u;
    sum += loc[q];
  }
  uint32_t total;
  uint32_t run = block_excl_scan(sum, sh.red, &total);
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int bin = nb - 1 - (threadIdx.x * PER + q);
    if (bin >= 0 && run < remaining && run + loc[q] >= remaining) {
      sh.found_bin = (uint32_t)bin;
      sh.found_above = run;
    }
    run += loc[q];
  }
  __syncthreads();
}

// Exact radix select over n elements in shared memory: the `want`-th largest
// value of f(i) (11+11+10-bit digits) among the flagged elements; *eq_out =
// how many flagged elements equal it.
template <class F, class Flag>
__device__ uint32_t smem_radix_select(TkShared& sh, int cn, uint32_t want, F f, Flag flag, uint32_t* above_out,
                                      uint32_t* eq_out) {
  uint32_t prefix = 0, mask = 0, remaining = want, eq = 0;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3ffu : 0x7ffu;
    for (int b = threadIdx.x; b < kTopkBins; b += TK_NT) sh.hist[b] = 0;
    __syncthreads();
    // eight elements per thread and iteration (their loads in flight together),
    // warp-uniform trip counts for the aggregated adds
    for (int i0 = (int)(threadIdx.x & ~31u); i0 < cn; i0 += 8 * TK_NT) {
      uint32_t kk[8];
      bool on[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * TK_NT + (int)(threadIdx.x & 31);
        on[u] = i < cn && flag(i);
        kk[u] = on[u] ? f(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) hist_add_warp(sh.hist, (kk[u] >> shift) & dmask, on[u] && (kk[u] & mask) == prefix);
    }
    __syncthreads();
    hist_suffix_find(sh, (int)dmask + 1, remaining);
    remaining -= sh.found_above;
    eq = sh.hist[sh.found_bin];
    prefix |= sh.found_bin << shift;
    mask |= dmask << shift;
    __syncthreads();
  }
  *above_out = want - remaining;
  *eq_out = eq;
  return prefix;
}

// ------------------------------------------------------------ the filter --
// Pass 1, one thread block per (row, chunk of TF_CH scores): the keys >= a row
// threshold T go to the chunk's slots (at most TF_CAPC; the count is written
// whole).  Every block of a row takes T from the same 1024 evenly spaced
// samples of the row with the same code, so all of them use the same T: the
// sample rank that should leave ~1.15 K + 3.5 sigma keys above it (a two-level
// histogram of the samples, top 11 bits then the next 11), rounded down to its
// 10-bit prefix.
constexpr int TF_NT = 1024;
constexpr int TF_PER = 16;
constexpr int TF_CH = TF_NT * TF_PER;
constexpr int TF_CAPC = TF_CH / 4;          // candidate slots per chunk
constexpr int TK_ROWCAP = TK_CAP;           // candidates a row may sort

struct TfShared {
  uint32_t hist[kTopkBins];
  uint32_t red[TF_NT / 32];
  uint32_t found_bin;
  uint32_t found_above;
};

__device__ __forceinline__ int row_length(const int32_t* lens, const idx_problem& p, int use_p, int max_len,
                                          int64_t m) {
  int n;
  if (use_p) {
    int64_t off;
    row_extent(p, m, &off, &n);
  } else {
    n = lens[m];
    n = n < 0 ? 0 : (n > max_len ? max_len : n);
  }
  return n;
}

// The row threshold (n > K): see above.  Uniform across the block.
__device__ uint32_t row_threshold(TfShared& sh, const float* row, int n, int K) {
  const int tid = threadIdx.x;
  constexpr int NS = TF_NT;
  const uint32_t sv = score_key(__ldg(row + (int)(((int64_t)tid * n) / NS)));
  const float expect = (float)NS * (float)K / (float)n;
  int r = (int)ceilf(1.15f * expect + 3.5f * sqrtf(expect)) + 1;
  r = r < 1 ? 1 : (r > NS ? NS : r);
  for (int b = tid; b < kTopkBins; b += TF_NT) sh.hist[b] = 0;
  __syncthreads();
  atomicAdd(&sh.hist[sv >> 21], 1u);
  __syncthreads();
  hist_suffix_find(sh, kTopkBins, (uint32_t)r);
  const uint32_t b1 = sh.found_bin, a1 = sh.found_above;
  __syncthreads();
  for (int b = tid; b < kTopkBins; b += TF_NT) sh.hist[b] = 0;
  __syncthreads();
  if ((sv >> 21) == b1) atomicAdd(&sh.hist[(sv >> 10) & 0x7ffu], 1u);
  __syncthreads();
  hist_suffix_find(sh, kTopkBins, (uint32_t)r - a1);
  const uint32_t T = (b1 << 21) | (sh.found_bin << 10);
  __syncthreads();
  return T ? T : 1u;
}

__global__ void __launch_bounds__(TF_NT, 2)
    topk_filter_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ lens, idx_problem p,
                       int use_p, int max_len, int K, const int32_t* __restrict__ id_map, int64_t id_ld,
                       const int32_t* __restrict__ row_mask, uint64_t* __restrict__ cand,
                       uint32_t* __restrict__ cnt) {
  // cand / cnt: slots of chunk (row, blockIdx.y) at index m * gridDim.y + blockIdx.y
  __shared__ TfShared sh;
  const int64_t m = blockIdx.x;
  const int64_t base = (int64_t)blockIdx.y * TF_CH;
  if (row_mask && !row_mask[m]) return;
  const int n = row_length(lens, p, use_p, max_len, m);
  if (base >= n) return;
  const int tid = threadIdx.x;
  const float* row = scores + m * ld;
  // every visible key when the row has at most K of them (ordered keys are >= 1)
  const uint32_t T = n <= K ? 1u : row_threshold(sh, row, n, K);
  uint32_t kv[TF_PER];
#pragma unroll
  for (int u = 0; u < TF_PER; ++u) {
    const int64_t i = base + u * TF_NT + tid;
    kv[u] = i < n ? score_key(__ldg(row + i)) : 0u;
  }
  uint32_t local = 0;
#pragma unroll
  for (int u = 0; u < TF_PER; ++u) local += kv[u] >= T ? 1u : 0u;
  uint32_t total;
  uint32_t pos = block_excl_scan(local, sh.red, &total);
  const int64_t slot = m * (int64_t)gridDim.y + blockIdx.y;
  if (tid == 0) cnt[slot] = total;
  const int32_t* idm = id_map ? id_map + m * id_ld : nullptr;
  uint64_t* out = cand + slot * TF_CAPC;
#pragma unroll
  for (int u = 0; u < TF_PER; ++u) {
    if (kv[u] >= T) {
      const int64_t i = base + u * TF_NT + tid;
      if (pos < (uint32_t)TF_CAPC) out[pos] = composite(kv[u], idm ? idm[i] : (int32_t)i);
      ++pos;
    }
  }
}

// ------------------------------------------------------------ the finish --
// Pass 2, one thread block per row: the candidates of the row's chunks are
// gathered, bucket-sorted at once and the first min(K, n) written.  When they
// are short of that or a chunk (or the row) overflowed (the threshold
// missed), the row is selected exactly from the scores themselves: radix
// select of the K-th key, then of the ids among its ties, compaction of
// exactly K, sort.
__global__ void __launch_bounds__(TK_NT, 1)
    topk_finish_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ lens, idx_problem p,
                       int use_p, int max_len, int K, int P, const int32_t* __restrict__ id_map, int64_t id_ld,
                       const int32_t* __restrict__ row_mask, const uint64_t* __restrict__ cand,
                       const uint32_t* __restrict__ cnt, int n_chunks, int32_t* __restrict__ out_ids,
                       float* __restrict__ out_scores) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  TkShared& sh = *reinterpret_cast<TkShared*>(tk_smem);
  const int64_t m = blockIdx.x;
  if (row_mask && !row_mask[m]) return;
  const int n = row_length(lens, p, use_p, max_len, m);
  const int tid = threadIdx.x;
  const int want = n < K ? n : K;
  uint64_t* best = reinterpret_cast<uint64_t*>(sh.keys);   // scratch, lower half of the key area
  auto emit = [&](const uint64_t* sorted, int have) {
    for (int j = tid; j < K; j += TK_NT) {
      const uint64_t v = j < have ? sorted[j] : 0ull;
      out_ids[m * K + j] = v ? key_id((uint32_t)v) : -1;
      if (out_scores) out_scores[m * K + j] = v ? key_score((uint32_t)(v >> 32)) : -__int_as_float(0x7f800000);
    }
  };
  if (want <= 0) {
    emit(nullptr, 0);
    return;
  }
  // the row's chunks: their counts (an overflowed chunk forces the exact path)
  const int rc = (int)((n + (int64_t)TF_CH - 1) / TF_CH);
  uint32_t total = 0;
  bool over = false;
  for (int c = 0; c < rc; ++c) {
    const uint32_t k = cnt[m * (int64_t)n_chunks + c];
    over |= k > (uint32_t)TF_CAPC;
    total += k;
  }
  if (!over && total >= (uint32_t)want && total <= (uint32_t)TK_ROWCAP) {
    uint32_t pre = 0;
    for (int c = 0; c < rc; ++c) {
      const int64_t slot = m * (int64_t)n_chunks + c;
      const int k = (int)cnt[slot];
      const uint64_t* src = cand + slot * TF_CAPC;
      for (int j = tid; j < k; j += TK_NT) sh.cand[pre + j] = src[j];
      pre += (uint32_t)k;
    }
    __syncthreads();
    if (total > 1 && bucket_sort_desc(sh, sh.cand, (int)total, best, false, want)) {
      emit(sh.cand, want);
      return;
    }
    int c2 = (int)total;
    if (c2 > want) {
      select_exact_k(sh, sh.cand, c2, want, best);
      c2 = want;
    } else {
      for (int j = tid; j < c2; j += TK_NT) best[j] = sh.cand[j];
      __syncthreads();
    }
    emit(order_desc(sh, best, c2, P, sh.cand), c2);
    return;
  }
  // exact, from the scores (pathological rows only)
  const float* row = scores + m * ld;
  const int32_t* idm = id_map ? id_map + m * id_ld : nullptr;
  auto idof = [&](int i) { return idm ? idm[i] : (int32_t)i; };
  auto key_f = [&](int i) { return score_key(__ldg(row + i)); };
  auto all = [&](int) { return true; };
  uint32_t above, eq;
  const uint32_t KT = smem_radix_select(sh, n, (uint32_t)want, key_f, all, &above, &eq);
  const uint32_t need = (uint32_t)want - above;
  uint32_t IT = 0;
  if (eq != need) {
    auto tie = [&](int i) { return key_f(i) == KT; };
    auto idk = [&](int i) { return id_key(idof(i)); };
    uint32_t above2, eq2;
    IT = smem_radix_select(sh, n, need, idk, tie, &above2, &eq2);
  }
  auto take = [&](int i) {
    const uint32_t kk = key_f(i);
    return kk > KT || (kk == KT && id_key(idof(i)) >= IT);
  };
  uint32_t local = 0;
  for (int i = tid; i < n; i += TK_NT) local += take(i) ? 1u : 0u;
  uint32_t tot2;
  uint32_t off = block_excl_scan(local, sh.red, &tot2);
  for (int i = tid; i < n; i += TK_NT)
    if (take(i)) sh.cand[off++] = composite(key_f(i), idof(i));
  __syncthreads();
  emit(order_desc(sh, sh.cand, want, P, best), want);
}

// ------------------------------------------------- many long rows, fused --
// When there are at least two rows per SM and the rows are long (the causal
// prefill: 4096 rows of up to 65536 scores; DoSA's seed and merge rows), one
// thread block of 512 threads per row does both passes, two blocks per SM so
// that one block's scan overlaps the other's sort: the row threshold once
// (the filter's rule, from 1024 evenly spaced samples), one coalesced stream
// over the row that collects the keys >= T in shared memory (a per-warp
// reservation, no global slots), then the same bucket sort and rank placement
// as the finish pass over those candidates, and the first min(K, n) written.
// Heavy ties take the two radix selects and a bitonic sort; a threshold that
// missed (fewer than min(K, n) candidates, or more than the candidate space)
// takes the exact radix select over the row's scores.  The output is the
// same as the two-pass path's (the exact top-K under (score desc, id asc)).
constexpr int TR_NT = 512;
constexpr int TR_NW = TR_NT / 32;
constexpr int TR_CAP = 7168;                // candidates a row may collect
constexpr int TR_KMAX = 2048;               // largest K this kernel takes
constexpr uint32_t kTrBucketMax = 256;      // a larger bucket: heavy ties
constexpr int TR_DST = TR_KMAX + 256;       // scatter space: the first K places plus one bucket
constexpr int TR_NB = 4096;                 // buckets of the sort
constexpr int TR_V = 4;                     // 4-score vectors per thread, round and register buffer
constexpr int TR_PD = 2;                    // rounds prefetched into L2 ahead of the loads
constexpr int TR_NS = 1024;                 // threshold samples

struct TrShared {
  uint64_t cand[TR_CAP];
  uint64_t dst[TR_DST];
  union {
    struct {
      uint32_t cur[TR_NB];                  // count, then scatter cursor, per bucket
      uint32_t start[TR_NB];                // first slot per bucket
    } b;
    uint32_t hist[kTopkBins];               // radix histograms (never live with the buckets)
  } u;
  uint32_t red[TR_NW];
  uint32_t found_bin, found_above;
  uint32_t kmin, kmax, bmax, kend, ncand;
};

// Exclusive prefix sum over the block in thread order; *total = block sum.
__device__ __forceinline__ uint32_t tr_excl_scan(uint32_t v, uint32_t* red, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();
  if (lane == 31) red[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    uint32_t x = lane < TR_NW ? red[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += u;
    }
    if (lane < TR_NW) red[lane] = x;
  }
  __syncthreads();
  *total = red[TR_NW - 1];
  return (wid ? red[wid - 1] : 0u) + incl - v;
}

// Suffix search over u.hist[0..nb) (bins high to low): the bin b with
// (#in bins > b) < remaining <= (#in bins >= b) -> found_bin / found_above.
__device__ __forceinline__ void tr_suffix_find(TrShared& sh, int nb, uint32_t remaining) {
  constexpr int PER = kTopkBins / TR_NT;
  uint32_t loc[PER], sum = 0;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int bin = nb - 1 - (threadIdx.x * PER + q);
    loc[q] = bin >= 0 ? sh.u.hist[bin] : 0u;
    sum += loc[q];
  }
  uint32_t total;
  uint32_t run = tr_excl_scan(sum, sh.red, &total);
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int bin = nb - 1 - (threadIdx.x * PER + q);
    if (bin >= 0 && run < remaining && run + loc[q] >= remaining) {
      sh.found_bin = (uint32_t)bin;
      sh.found_above = run;
    }
    run += loc[q];
  }
  __syncthreads();
}

// Row thresholds, one warp per row, before the fused kernel: from 1024 samples
// (32 per lane, in runs of 8 evenly spread), v = the key of the sample ranked r (the filter's
// rank: ~1.15 K + 3.5 sigma keys expected above it), found exactly by a search
// over its 32 bits (the largest key with at least r samples at or above it).
// thr[m] = v rounded down to its 22-bit prefix, as in the filter -- unless v
// is a heavily repeated value (8 or more samples equal to it: a plateau of
// equal scores, e.g. the exact zeros of rows whose heads all clip), then
// thr[m] = v + 1 and piv[m] = v: the plateau is left out of the candidates and
// the fused kernel takes from it only what the top-K needs.  Rows with at most
// K visible keys get thr = 1 (everything).
constexpr int TT_WARPS = 8;

__global__ void __launch_bounds__(32 * TT_WARPS, 1)
    topk_thresh_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ lens, idx_problem p,
                       int use_p, int max_len, int K, const int32_t* __restrict__ row_mask, int64_t M,
                       uint32_t* __restrict__ thr, uint32_t* __restrict__ piv) {
  const int64_t m = (int64_t)blockIdx.x * TT_WARPS + (threadIdx.x >> 5);
  if (m >= M) return;
  const int lane = threadIdx.x & 31;
  if (row_mask && !row_mask[m]) return;
  const int n = row_length(lens, p, use_p, max_len, m);
  if (n <= K) {
    if (lane == 0) {
      thr[m] = 1u;
      piv[m] = 0u;
    }
    return;
  }
  // samples in 128 runs of 8 consecutive scores (one 32-byte sector each) spread
  // evenly over the row: sample s sits at run_start(s / 8) + s % 8.  A lone
  // 4-byte sample costs a whole 128-byte line of DRAM traffic, so runs cut
  // the threshold's traffic about eightfold.
  const float* row = scores + m * ld;
  uint32_t kv[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int smp = lane + 32 * j;
    int pos = (int)(((int64_t)(smp >> 3) * n) / (TR_NS / 8)) + (smp & 7);
    pos = pos < n ? pos : n - 1;
    kv[j] = score_key(__ldg(row + pos));
  }
  const float expect = (float)TR_NS * (float)K / (float)n;
  int r = (int)ceilf(1.15f * expect + 3.5f * sqrtf(expect)) + 1;
  r = r < 1 ? 1 : (r > TR_NS ? TR_NS : r);
  uint32_t v = 0;
#pragma unroll 1
  for (int b = 31; b >= 0; --b) {
    const uint32_t trial = v | (1u << b);
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) c += kv[j] >= trial ? 1u : 0u;
    if (__reduce_add_sync(0xffffffffu, c) >= (uint32_t)r) v = trial;
  }
  uint32_t eq = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) eq += kv[j] == v ? 1u : 0u;
  eq = __reduce_add_sync(0xffffffffu, eq);
  uint32_t T = v & ~0x3ffu, pv = 0u;
  if (eq >= 8u && v < 0xffffffffu) {
    T = v + 1u;
    pv = v;
  }
  if (lane == 0) {
    thr[m] = T ? T : 1u;
    piv[m] = pv;
  }
}

// Exact radix select over cn elements: the want-th largest f(i) among the
// flagged ones (11 + 11 + 10 bits); *eq_out = how many flagged equal it.
template <class F, class Flag>
__device__ uint32_t tr_radix_select(TrShared& sh, int cn, uint32_t want, F f, Flag flag, uint32_t* above_out,
                                    uint32_t* eq_out) {
  uint32_t prefix = 0, mask = 0, remaining = want, eq = 0;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3ffu : 0x7ffu;
    for (int b = threadIdx.x; b < kTopkBins; b += TR_NT) sh.u.hist[b] = 0;
    __syncthreads();
    // eight elements per thread and iteration (their loads in flight together),
    // warp-uniform trip counts for the aggregated adds
    for (int i0 = (int)(threadIdx.x & ~31u); i0 < cn; i0 += 8 * TR_NT) {
      uint32_t kk[8];
      bool on[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * TR_NT + (int)(threadIdx.x & 31);
        on[u] = i < cn && flag(i);
        kk[u] = on[u] ? f(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) hist_add_warp(sh.u.hist, (kk[u] >> shift) & dmask, on[u] && (kk[u] & mask) == prefix);
    }
    __syncthreads();
    tr_suffix_find(sh, (int)dmask + 1, remaining);
    remaining -= sh.found_above;
    eq = sh.u.hist[sh.found_bin];
    prefix |= sh.found_bin << shift;
    mask |= dmask << shift;
    __syncthreads();
  }
  *above_out = want - remaining;
  *eq_out = eq;
  return prefix;
}

// Sorts the first `limit` places of the n nonzero, distinct composites src
// descending (the finish pass's bucket sort, 4096 buckets): src[0, limit) ends
// up in order.  dst takes the scattered elements (at most limit + 255).
// Returns false, src untouched, when a bucket holds more than kTrBucketMax.
__device__ bool tr_bucket_sort(TrShared& sh, uint64_t* src, int n, uint64_t* dst, int limit) {
  const int tid = threadIdx.x;
  uint32_t* bh = sh.u.b.cur;
  uint32_t* bs = sh.u.b.start;
  constexpr int PER = TR_NB / TR_NT;
  static_assert(PER == 8, "two 16-byte vectors per thread");
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  reinterpret_cast<uint4*>(bh)[2 * tid] = z;
  reinterpret_cast<uint4*>(bh)[2 * tid + 1] = z;
  if (tid == 0) {
    sh.kmin = 0xffffffffu;
    sh.kmax = 0u;
    sh.bmax = 0u;
    sh.kend = (uint32_t)n;
  }
  __syncthreads();
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int i = tid; i < n; i += TR_NT) {
    const uint32_t k = (uint32_t)(src[i] >> 32);
    mn = min(mn, k);
    mx = max(mx, k);
  }
  mn = __reduce_min_sync(0xffffffffu, mn);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if ((tid & 31) == 0) {
    atomicMin(&sh.kmin, mn);
    atomicMax(&sh.kmax, mx);
  }
  __syncthreads();
  const uint32_t kmin = sh.kmin;
  const float scale = (float)TR_NB / ((float)(sh.kmax - kmin) + 1.0f);
  auto bucket = [&](uint64_t v) {
    uint32_t b = (uint32_t)((float)((uint32_t)(v >> 32) - kmin) * scale);
    b = b < (uint32_t)TR_NB ? b : (uint32_t)TR_NB - 1u;
    return (uint32_t)TR_NB - 1u - b;   // largest keys first
  };
  for (int i = tid; i < n; i += TR_NT) atomicAdd(&bh[bucket(src[i])], 1u);
  __syncthreads();
  const uint4 c0 = reinterpret_cast<const uint4*>(bh)[2 * tid];
  const uint4 c1 = reinterpret_cast<const uint4*>(bh)[2 * tid + 1];
  const uint32_t cnt8[PER] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  uint32_t sum = 0, big = 0;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    sum += cnt8[q];
    big = max(big, cnt8[q]);
  }
  uint32_t total;
  uint32_t run = tr_excl_scan(sum, sh.red, &total);
  big = __reduce_max_sync(0xffffffffu, big);
  if ((tid & 31) == 0) atomicMax(&sh.bmax, big);
  const uint32_t lim = (uint32_t)(limit < n ? limit : n);
  uint32_t st8[PER], kend = 0xffffffffu;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    st8[q] = run;
    if (run >= lim && cnt8[q]) kend = min(kend, run);   // first bucket left out
    run += cnt8[q];
  }
  kend = __reduce_min_sync(0xffffffffu, kend);
  if ((tid & 31) == 0 && kend != 0xffffffffu) atomicMin(&sh.kend, kend);
  reinterpret_cast<uint4*>(bs)[2 * tid] = make_uint4(st8[0], st8[1], st8[2], st8[3]);
  reinterpret_cast<uint4*>(bs)[2 * tid + 1] = make_uint4(st8[4], st8[5], st8[6], st8[7]);
  reinterpret_cast<uint4*>(bh)[2 * tid] = make_uint4(st8[0], st8[1], st8[2], st8[3]);   // scatter cursors
  reinterpret_cast<uint4*>(bh)[2 * tid + 1] = make_uint4(st8[4], st8[5], st8[6], st8[7]);
  __syncthreads();
  if (sh.bmax > kTrBucketMax) return false;
  for (int i = tid; i < n; i += TR_NT) {
    const uint64_t v = src[i];
    const uint32_t b = bucket(v);
    if (bs[b] >= lim) continue;
    const uint32_t pos = atomicAdd(&bh[b], 1u);
    dst[pos] = v;
  }
  __syncthreads();
  const int used = (int)sh.kend;
  for (int i = tid; i < used; i += TR_NT) {
    const uint64_t v = dst[i];
    const uint32_t b = bucket(v);
    const int b0 = (int)bs[b], b1 = (int)bh[b];
    int r = b0;
    for (int q = b0; q < b1; ++q) r += dst[q] > v ? 1 : 0;
    src[r] = v;
  }
  __syncthreads();
  return true;
}

// Bitonic sort of buf[0..S) descending (S a power of two).
__device__ void tr_bitonic_desc(uint64_t* v, int S) {
  for (int size = 2; size <= S; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < (S >> 1); t += TR_NT) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const uint64_t a = v[lo], b = v[hi];
        if ((a < b) == desc) {
          v[lo] = b;
          v[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

// The `want` largest of the n composites src[0..n) (want <= n), sorted, in
// src[0..want) or dst[0..want): returns where.  Bucket sort, else (heavy ties)
// two radix selects cut exactly `want` into dst and a bitonic sort orders them.
__device__ const uint64_t* tr_order_top(TrShared& sh, uint64_t* src, int n, int want, int P, uint64_t* dst) {
  if (n <= 1) return src;
  if (tr_bucket_sort(sh, src, n, dst, want)) return src;
  int c = n;
  if (n > want) {
    uint32_t above, eq;
    auto hi = [&](int i) { return (uint32_t)(src[i] >> 32); };
    auto real = [&](int i) { return src[i] != 0ull; };
    const uint32_t KT = tr_radix_select(sh, n, (uint32_t)want, hi, real, &above, &eq);
    const uint32_t need = (uint32_t)want - above;
    uint32_t IT = 0;
    if (eq != need) {
      auto lo = [&](int i) { return (uint32_t)src[i]; };
      auto tie = [&](int i) { return src[i] != 0ull && (uint32_t)(src[i] >> 32) == KT; };
      uint32_t above2, eq2;
      IT = tr_radix_select(sh, n, need, lo, tie, &above2, &eq2);
    }
    auto take = [&](int i) {
      const uint64_t v = src[i];
      const uint32_t k = (uint32_t)(v >> 32);
      return v != 0ull && (k > KT || (k == KT && (uint32_t)v >= IT));
    };
    uint32_t local = 0;
    for (int i = threadIdx.x; i < n; i += TR_NT) local += take(i) ? 1u : 0u;
    uint32_t total;
    uint32_t off = tr_excl_scan(local, sh.red, &total);
    for (int i = threadIdx.x; i < n; i += TR_NT)
      if (take(i)) dst[off++] = src[i];
    c = want;
  } else {
    for (int i = threadIdx.x; i < n; i += TR_NT) dst[i] = src[i];
  }
  for (int i = c + threadIdx.x; i < P; i += TR_NT) dst[i] = 0ull;
  __syncthreads();
  tr_bitonic_desc(dst, P);
  return dst;
}

__global__ void __launch_bounds__(TR_NT, 2)
    topk_rows_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ lens, idx_problem p,
                     int use_p, int max_len, int K, int P, const int32_t* __restrict__ id_map, int64_t id_ld,
                     const int32_t* __restrict__ row_mask, int32_t* __restrict__ out_ids,
                     float* __restrict__ out_scores, int vec4, const uint32_t* __restrict__ thr,
                     const uint32_t* __restrict__ piv) {
  extern __shared__ __align__(16) uint8_t tr_smem[];
  TrShared& sh = *reinterpret_cast<TrShared*>(tr_smem);
  const int64_t m = blockIdx.x;
  if (row_mask && !row_mask[m]) return;
  const int n = row_length(lens, p, use_p, max_len, m);
  const int tid = threadIdx.x, lane = tid & 31;
  const int want = n < K ? n : K;
  auto emit = [&](const uint64_t* sorted, int have) {
    for (int j = tid; j < K; j += TR_NT) {
      const uint64_t v = j < have ? sorted[j] : 0ull;
      out_ids[m * K + j] = v ? key_id((uint32_t)v) : -1;
      if (out_scores) out_scores[m * K + j] = v ? key_score((uint32_t)(v >> 32)) : -__int_as_float(0x7f800000);
    }
  };
  if (want <= 0) {
    emit(nullptr, 0);
    return;
  }
  const float* row = scores + m * ld;
  const int32_t* idm = id_map ? id_map + m * id_ld : nullptr;
  auto idof = [&](int i) { return idm ? idm[i] : (int32_t)i; };
  // keys >= T (T = 1: every visible key), compared as floats: x >= key_score(T)
  // is key(x) >= T for every finite x (a T below every finite key maps to a NaN
  // float, and then everything is kept)
  const uint32_t T = thr[m], pv = piv[m];
  const float Tf = key_score(T);
  const bool keep_all = T <= 1u || !(Tf == Tf);
  if (tid == 0) sh.ncand = 0;
  __syncthreads();
  // one stream over the row: keys >= T into the candidate space.  Rounds of
  // 4 x TR_NT x TR_V scores, thread tid reading the four at c0 + 4 (v TR_NT +
  // tid) .. + 3 (one 16-byte load when the rows allow it: ld a multiple of 4
  // and an aligned base, checked by the host); two register buffers, so that
  // one round's loads are in flight while the previous round is processed; one
  // shared-memory reservation per warp and round.
  auto load_round = [&](float4 (&buf)[TR_V], int c0) {
#pragma unroll
    for (int v = 0; v < TR_V; ++v) {
      const int i0 = c0 + 4 * (v * TR_NT + tid);
      float4 f = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (i0 < n) {
        if (vec4) {
          // i0 < n <= ld and ld % 4 == 0, so the vector lies inside the row's storage
          f = __ldg(reinterpret_cast<const float4*>(row + i0));
        } else {
          f.x = __ldg(row + i0);
          if (i0 + 1 < n) f.y = __ldg(row + i0 + 1);
          if (i0 + 2 < n) f.z = __ldg(row + i0 + 2);
          if (i0 + 3 < n) f.w = __ldg(row + i0 + 3);
        }
      }
      buf[v] = f;
    }
  };
  constexpr int kStep = 4 * TR_NT * TR_V;
  auto process_round = [&](const float4 (&buf)[TR_V], int c0) {
    uint32_t kmask = 0;                        // bit 4 v + e: score e of vector v is kept
    if (c0 + kStep <= n && !keep_all) {
      // a whole round of visible scores (all rounds but a row's last): one
      // compare per score
#pragma unroll
      for (int v = 0; v < TR_V; ++v) {
        const float x[4] = {buf[v].x, buf[v].y, buf[v].z, buf[v].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) kmask |= (x[e] >= Tf ? 1u : 0u) << (4 * v + e);
      }
    } else {
#pragma unroll
      for (int v = 0; v < TR_V; ++v) {
        const int i0 = c0 + 4 * (v * TR_NT + tid);
        const float x[4] = {buf[v].x, buf[v].y, buf[v].z, buf[v].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i0 + e < n && (keep_all || x[e] >= Tf)) kmask |= 1u << (4 * v + e);
      }
    }
    const uint32_t c = (uint32_t)__popc(kmask);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t base = 0;
    if (wtot) {
      if (lane == 31) base = atomicAdd(&sh.ncand, wtot);
      base = __shfl_sync(0xffffffffu, base, 31);
    }
    uint32_t pos = base + incl - c;
#pragma unroll
    for (int v = 0; v < TR_V; ++v) {
      uint32_t m4 = (kmask >> (4 * v)) & 0xfu;
      while (m4) {
        const int e = __ffs(m4) - 1;
        m4 &= m4 - 1u;
        const float4 f = buf[v];
        const float xv = e == 0 ? f.x : (e == 1 ? f.y : (e == 2 ? f.z : f.w));
        if (pos < (uint32_t)TR_CAP) sh.cand[pos] = composite(score_key(xv), idof(c0 + 4 * (v * TR_NT + tid) + e));
        ++pos;
      }
    }
  };
  // The register buffers hold two rounds (64 KB a block); an L2 prefetch of the
  // rounds TR_PD ahead (one bulk request by thread 0 per round, aligned rows
  // only) lets those loads find their data in L2.  Each request covers the
  // round's scores rounded up to 16 bytes, inside the row's storage (ld is a
  // multiple of 4 when vec4).
  auto prefetch_round = [&](int c0p) {
    if (vec4 && tid == 0 && c0p < n) {
      const int cnt = n - c0p < kStep ? n - c0p : kStep;
      l2_prefetch_bulk(row + c0p, (uint32_t)(((cnt + 3) & ~3) * 4));
    }
  };
#pragma unroll
  for (int r = 1; r <= TR_PD; ++r) prefetch_round(r * kStep);
  float4 ba[TR_V], bb[TR_V];
  load_round(ba, 0);
#pragma unroll 1
  for (int c0 = 0; c0 < n; c0 += 2 * kStep) {
    prefetch_round(c0 + (TR_PD + 1) * kStep);
    load_round(bb, c0 + kStep);
    process_round(ba, c0);
    prefetch_round(c0 + (TR_PD + 2) * kStep);
    load_round(ba, c0 + 2 * kStep);
    process_round(bb, c0 + kStep);
  }
  __syncthreads();
  const uint32_t total = sh.ncand;
  if (total >= (uint32_t)want && total <= (uint32_t)TR_CAP) {
    emit(tr_order_top(sh, sh.cand, (int)total, want, P, sh.dst), want);
    return;
  }
  if (pv && !idm && total < (uint32_t)want) {
    // The plateau at pv was left out and the keys above it are fewer than
    // min(K, n): if the row has enough keys equal to pv, the K-th key is pv and
    // the rest of the top-K are the keys equal to pv with the smallest ids --
    // the first ones in row order (ids are positions here).  One ordered scan:
    // thread t takes four consecutive positions of each 2048-position chunk.
    const uint32_t need = (uint32_t)want - total;
    uint32_t found = 0;
#pragma unroll 1
    for (int c0 = 0; c0 < n && found < need; c0 += 4 * TR_NT) {
      const int i0 = c0 + 4 * tid;
      uint32_t ek[4];
      uint32_t c = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ek[e] = i0 + e < n ? score_key(__ldg(row + i0 + e)) : 0u;
        c += ek[e] == pv ? 1u : 0u;
      }
      uint32_t chunk;
      uint32_t rank = found + tr_excl_scan(c, sh.red, &chunk);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (ek[e] == pv) {
          if (rank < need) sh.cand[total + rank] = composite(pv, i0 + e);
          ++rank;
        }
      }
      found += chunk;
    }
    __syncthreads();
    if (found >= need) {
      emit(tr_order_top(sh, sh.cand, want, want, P, sh.dst), want);
      return;
    }
  }
  // the threshold missed: exact radix select over the row's scores
  auto key_f = [&](int i) { return score_key(__ldg(row + i)); };
  auto all = [&](int) { return true; };
  uint32_t above, eq;
  const uint32_t KT = tr_radix_select(sh, n, (uint32_t)want, key_f, all, &above, &eq);
  const uint32_t need = (uint32_t)want - above;
  uint32_t IT = 0;
  if (eq != need) {
    auto tie = [&](int i) { return key_f(i) == KT; };
    auto idk = [&](int i) { return id_key(idof(i)); };
    uint32_t above2, eq2;
    IT = tr_radix_select(sh, n, need, idk, tie, &above2, &eq2);
  }
  auto take = [&](int i) {
    const uint32_t kk = key_f(i);
    return kk > KT || (kk == KT && id_key(idof(i)) >= IT);
  };
  uint32_t local = 0;
  for (int i = tid; i < n; i += TR_NT) local += take(i) ? 1u : 0u;
  uint32_t tot2;
  uint32_t off = tr_excl_scan(local, sh.red, &tot2);
  for (int i = tid; i < n; i += TR_NT)
    if (take(i)) sh.cand[off++] = composite(key_f(i), idof(i));
  __syncthreads();
  emit(tr_order_top(sh, sh.cand, want, want, P, sh.dst), want);
}

// The fused kernel takes a launch when the rows are long, there are at least
// two per SM and K fits its sort space.
static bool topk_rows_applies(int64_t M, int max_len, int K) {
  return K <= TR_KMAX && max_len > 4096 && M >= 2 * (int64_t)sm_count();
}

static int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

static int filter_chunks(int max_len) { return max_len > 0 ? (max_len + TF_CH - 1) / TF_CH : 1; }

// Workspace: a candidate count per (row, chunk), then TF_CAPC candidate slots per (row, chunk).
size_t topk_dense_ws(int64_t M, int max_len, int K) {
  (void)K;
  if (M <= 0) return 0;
  const size_t slots = (size_t)M * (size_t)filter_chunks(max_len);
  WsCarver c(nullptr);
  c.take<uint32_t>(slots);
  c.take<uint64_t>(slots * TF_CAPC);
  return c.used;
}

cudaError_t launch_topk_dense(const float* scores, int64_t ld, const int32_t* lens, const idx_problem* p_or_null,
                              int64_t M, int max_len, int K, int32_t* out_ids, float* out_scores, void* ws,
                              cudaStream_t st, const int32_t* id_map, int64_t id_ld, const int32_t* row_mask) {
  if (M <= 0) return cudaSuccess;
  const int P = pow2_at_least(K);
  if (topk_rows_applies(M, max_len, K)) {
    if (M > 0x7fffffff) return cudaErrorInvalidValue;
    idx_problem p{};
    if (p_or_null) p = *p_or_null;
    const size_t smem = sizeof(TrShared);
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int vec4 = (ld % 4 == 0 && (reinterpret_cast<uintptr_t>(scores) & 15) == 0) ? 1 : 0;
    WsCarver c(ws);
    uint32_t* thr = c.take<uint32_t>((size_t)M);
    uint32_t* piv = c.take<uint32_t>((size_t)M);
    topk_thresh_kernel<<<(unsigned)((M + TT_WARPS - 1) / TT_WARPS), 32 * TT_WARPS, 0, st>>>(
        scores, ld, lens, p, p_or_null ? 1 : 0, max_len, K, row_mask, M, thr, piv);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    topk_rows_kernel<<<(unsigned)M, TR_NT, smem, st>>>(scores, ld, lens, p, p_or_null ? 1 : 0, max_len, K, P, id_map,
                                                       id_ld, row_mask, out_ids, out_scores, vec4, thr, piv);
    return cudaGetLastError();
  }
  const int n_chunks = filter_chunks(max_len);
  if (n_chunks > 65535 || M > 0x7fffffff) return cudaErrorInvalidValue;
  idx_problem p{};
  if (p_or_null) p = *p_or_null;
  WsCarver c(ws);
  const size_t slots = (size_t)M * (size_t)n_chunks;
  uint32_t* cnt = c.take<uint32_t>(slots);
  uint64_t* cand = c.take<uint64_t>(slots * TF_CAPC);
  cudaError_t e;
  topk_filter_kernel<<<dim3((unsigned)M, (unsigned)n_chunks), TF_NT, 0, st>>>(
      scores, ld, lens, p, p_or_null ? 1 : 0, max_len, K, id_map, id_ld, row_mask, cand, cnt);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(TkShared);
  e = cudaFuncSetAttribute(topk_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_finish_kernel<<<(unsigned)M, TK_NT, smem, st>>>(scores, ld, lens, p, p_or_null ? 1 : 0, max_len, K, P, id_map,
                                                       id_ld, row_mask, cand, cnt, n_chunks, out_ids, out_scores);
  return cudaGetLastError();
}

}  // namespace idx
