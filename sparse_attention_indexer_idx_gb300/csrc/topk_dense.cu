// Exact top-K of dense score rows, under (score desc, key id asc)
// ("DoSA：用安全上界减少 Indexer 的完整打分", section 1 and the note after
// section 2: selection by the original scorer with one total order for ties).
//
// A row is cut into chunks of TK_CH = 32768 scores; one thread block owns a
// chunk and keeps it in registers (64 ordered keys per thread), so the row is
// read from memory exactly once.  Selection inside a chunk:
//   1. 1024 keys sampled from the chunk are bitonic-sorted; the sample rank
//      that should leave ~1.2 K + 3 sigma keys above it gives a threshold T;
//   2. one pass counts the keys >= T (block reduction, no atomics); if the
//      count is at least K and fits the candidate buffer, a second pass
//      compacts them (warp ballot + one atomic per warp) as 64-bit composites
//      key << 32 | ~id, whose descending order is exactly (score desc, id asc);
//      otherwise T is lowered (or, failing that, an exact radix select on the
//      registers takes over);
//   3. the K winners are bitonic-sorted (in-thread and warp-shuffle stages,
//      shared memory only for strides that cross warps).
// The candidates are cut to exactly K by two radix selects (key, then id among
// ties) and only then sorted, in registers.  A row of one chunk writes its
// result directly; longer rows write every chunk's (unsorted) top-K set to the
// workspace, and a merge kernel folds the sets into a running best-K and sorts
// once.
#include "internal.h"
#include "topk.cuh"

namespace idx {

constexpr int TK_NT = 1024;
constexpr int TK_CH = 32768;
constexpr int TK_NS = 1024;
constexpr int TK_CAP = 8192;

struct TkShared {
  uint32_t keys[TK_CH];       // the chunk's ordered keys
  uint64_t cand[TK_CAP];
  uint32_t samp[TK_NS];
  uint32_t hist[kTopkBins];
  uint32_t bstart[kTopkBins];
  uint32_t red[TK_NT / 32];
  uint32_t cnt;
  uint32_t found_bin;
  uint32_t found_above;
  uint32_t kmin, kmax, bmax;
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
// keys' minimum and maximum.  Returns false, with src untouched, when a bucket
// would hold more than kBucketMax entries (heavy ties): the caller then uses
// the bitonic network.
constexpr uint32_t kBucketMax = 32;
constexpr int kSortBuckets = 8192;
__device__ bool bucket_sort_desc(TkShared& sh, uint64_t* src, int n, uint64_t* dst, bool have_range = false) {
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
  if (tid == 0) sh.bmax = 0u;
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
  uint32_t st8[PER];
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    st8[q] = run;
    run += cnt8[q];
  }
  reinterpret_cast<uint4*>(bs)[2 * tid] = make_uint4(st8[0], st8[1], st8[2], st8[3]);
  reinterpret_cast<uint4*>(bs)[2 * tid + 1] = make_uint4(st8[4], st8[5], st8[6], st8[7]);
  reinterpret_cast<uint4*>(bh)[2 * tid] = make_uint4(st8[0], st8[1], st8[2], st8[3]);   // scatter cursors
  reinterpret_cast<uint4*>(bh)[2 * tid + 1] = make_uint4(st8[4], st8[5], st8[6], st8[7]);
  __syncthreads();
  if (sh.bmax > kBucketMax) return false;
  for (int i = tid; i < n; i += TK_NT) {
    const uint64_t v = src[i];
    const uint32_t pos = atomicAdd(&bh[bucket(v)], 1u);
    dst[pos] = v;
  }
  __syncthreads();
  // place: bucket start + the number of larger elements in the bucket
  for (int i = tid; i < n; i += TK_NT) {
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
__device__ __forceinline__ void hist_suffix_find(TkShared& sh, int nb, uint32_t remaining) {
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
    for (int i = threadIdx.x; i < cn; i += TK_NT) {
      if (flag(i)) {
        const uint32_t k = f(i);
        if ((k & mask) == prefix) atomicAdd(&sh.hist[(k >> shift) & dmask], 1u);
      }
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

// One chunk of one row.  Writes the final top-K when the row is one chunk,
// else the chunk's sorted top-K list (P = next_pow2(K) composites, 0-padded).
__global__ void __launch_bounds__(TK_NT, 1)
    topk_chunk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ lens,
                      idx_problem p, int use_p, int max_len, int K, int P, int32_t* __restrict__ out_ids,
                      float* __restrict__ out_scores, uint64_t* __restrict__ lists, int n_chunks,
                      const int32_t* __restrict__ id_map, int64_t id_ld, const int32_t* __restrict__ row_mask) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  TkShared& sh = *reinterpret_cast<TkShared*>(tk_smem);
  const int64_t m = blockIdx.x;
  const int c = blockIdx.y;
  if (row_mask && !row_mask[m]) return;
  int n;
  if (use_p) {
    int64_t off;
    row_extent(p, m, &off, &n);
  } else {
    n = lens[m];
    n = n < 0 ? 0 : (n > max_len ? max_len : n);
  }
  const int64_t base = (int64_t)c * TK_CH;
  if (c > 0 && base >= n) return;
  const bool single = n <= TK_CH;
  const int cn = (int)min((int64_t)TK_CH, (int64_t)n - base > 0 ? (int64_t)n - base : 0);
  const float* row = scores + m * ld + base;
  const int tid = threadIdx.x;
  const int32_t* idm = id_map ? id_map + m * id_ld + base : nullptr;
  auto idof = [&](int i) { return idm ? idm[i] : (int32_t)(base + i); };

  // stage the chunk as ordered keys in shared memory (8 loads in flight per thread)
  uint32_t* K_ = sh.keys;
  for (int i0 = 0; i0 < cn; i0 += 8 * TK_NT) {
    float f[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * TK_NT + tid;
      f[u] = i < cn ? __ldg(row + i) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * TK_NT + tid;
      if (i < cn) K_[i] = score_key(f[u]);
    }
  }
  __syncthreads();

  // Candidates: every key >= T (or, exact_ids, the exact top set), written
  // through a block prefix sum (no atomics); their smallest and largest key go
  // to sh.kmin / sh.kmax.  `counted`: this thread's count of them when the
  // caller already has it.
  auto compact = [&](uint32_t T, uint32_t KT, uint32_t IT, bool exact_ids, int counted) {
    auto take = [&](int i) {
      const uint32_t kk = K_[i];
      return exact_ids ? (kk > KT || (kk == KT && id_key(idof(i)) >= IT)) : kk >= T;
    };
    uint32_t local = 0;
    if (counted >= 0) {
      local = (uint32_t)counted;
    } else {
      for (int i = tid; i < cn; i += TK_NT) local += take(i) ? 1u : 0u;
    }
    if (tid == 0) {
      sh.kmin = 0xffffffffu;
      sh.kmax = 0u;
    }
    uint32_t total;
    uint32_t off = block_excl_scan(local, sh.red, &total);
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (int i = tid; i < cn; i += TK_NT) {
      if (take(i)) {
        const uint32_t kk = K_[i];
        mn = min(mn, kk);
        mx = max(mx, kk);
        if (off < (uint32_t)TK_CAP) sh.cand[off] = composite(kk, idof(i));
        ++off;
      }
    }
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if ((tid & 31) == 0) {
      atomicMin(&sh.kmin, mn);
      atomicMax(&sh.kmax, mx);
    }
    if (tid == 0) sh.cnt = total;
    __syncthreads();
  };

  if (cn <= K) {
    compact(0u, 0u, 0u, false, -1);      // every key (keys are >= 1)
  } else {
    // 1. threshold from 1024 evenly spaced sample keys: the sample rank r that
    //    should leave ~1.15 K + 3 sigma keys above, located by a two-level
    //    histogram of the samples (top 11 bits, then the next 11)
    const int step = cn / TK_NS > 0 ? cn / TK_NS : 1;
    const int si = tid * step;
    const uint32_t sv = si < cn ? K_[si] : 0u;
    const int nvalid = min(TK_NS, cn);
    const float expect = (float)nvalid * (float)K / (float)cn;
    int r = (int)ceilf(1.15f * expect + 3.0f * sqrtf(expect)) + 1;
    r = r < 1 ? 1 : (r > nvalid ? nvalid : r);
    uint32_t T = 0, count = 0, mine = 0;
    bool ok = false;
#pragma unroll 1
    for (int attempt = 0; attempt < 3; ++attempt) {
      for (int b2 = tid; b2 < kTopkBins; b2 += TK_NT) sh.hist[b2] = 0;
      __syncthreads();
      if (sv) atomicAdd(&sh.hist[sv >> 21], 1u);
      __syncthreads();
      hist_suffix_find(sh, kTopkBins, (uint32_t)r);
      const uint32_t b1 = sh.found_bin, a1 = sh.found_above;
      __syncthreads();
      for (int b2 = tid; b2 < kTopkBins; b2 += TK_NT) sh.hist[b2] = 0;
      __syncthreads();
      if (sv && (sv >> 21) == b1) atomicAdd(&sh.hist[(sv >> 10) & 0x7ffu], 1u);
      __syncthreads();
      hist_suffix_find(sh, kTopkBins, (uint32_t)r - a1);
      T = (b1 << 21) | (sh.found_bin << 10);
      if (T == 0u) T = 1u;
      __syncthreads();
      uint32_t local = 0;
      for (int i = tid; i < cn; i += TK_NT) local += (K_[i] >= T) ? 1u : 0u;
      mine = local;
      count = block_sum_u32(local, sh.red);
      if (count > (uint32_t)TK_CAP) break;
      if (count >= (uint32_t)K) {
        ok = true;
        break;
      }
      if (r == nvalid) break;
      r = min(nvalid, 2 * r);
    }
    if (ok) {
      compact(T, 0u, 0u, false, (int)mine);
    } else {
      // exact: radix select of the K-th key, then of the ids among its ties
      uint32_t above, eq;
      auto key_f = [&](int i) { return K_[i]; };
      auto all = [&](int) { return true; };
      const uint32_t KT = smem_radix_select(sh, cn, (uint32_t)K, key_f, all, &above, &eq);
      const uint32_t need = (uint32_t)K - above;
      uint32_t IT = 0;
      if (eq != need) {
        auto tie = [&](int i) { return K_[i] == KT; };
        auto idk = [&](int i) { return id_key(idof(i)); };
        uint32_t above2, eq2;
        IT = smem_radix_select(sh, cn, need, idk, tie, &above2, &eq2);
      }
      compact(0u, KT, IT, true, -1);
    }
  }
  __syncthreads();
  int cnt = (int)min(sh.cnt, (uint32_t)TK_CAP);
  uint64_t* best = reinterpret_cast<uint64_t*>(sh.keys);   // the (now free) key area
  if (single && cnt > K) {
    // the candidates are distinct composites: when their buckets are even, one
    // bucket sort of all of them orders the row and its first K are the answer
    if (sh.cnt <= (uint32_t)TK_CAP && bucket_sort_desc(sh, sh.cand, cnt, best, true)) {
      for (int j = tid; j < K; j += TK_NT) {
        const uint64_t v = sh.cand[j];
        out_ids[m * K + j] = key_id((uint32_t)v);
        if (out_scores) out_scores[m * K + j] = key_score((uint32_t)(v >> 32));
      }
      return;
    }
  }
  // exactly min(K, cn) composites
  if (cnt > K) {
    select_exact_k(sh, sh.cand, cnt, K, best);
    cnt = K;
  } else {
    for (int i = tid; i < cnt; i += TK_NT) best[i] = sh.cand[i];
    __syncthreads();
  }
  if (!single) {
    uint64_t* dst = lists + ((int64_t)m * n_chunks + c) * P;
    for (int j = tid; j < P; j += TK_NT) dst[j] = j < cnt ? best[j] : 0ull;
    return;
  }
  const uint64_t* sorted = order_desc(sh, best, cnt, P, sh.cand);
  for (int j = tid; j < K; j += TK_NT) {
    const uint64_t v = j < cnt ? sorted[j] : 0ull;
    out_ids[m * K + j] = v ? key_id((uint32_t)v) : -1;
    if (out_scores) out_scores[m * K + j] = v ? key_score((uint32_t)(v >> 32)) : -__int_as_float(0x7f800000);
  }
}

// Folds the chunk candidate sets of every multi-chunk row into its top-K:
// a running best-K set meets each chunk's set, an exact selection keeps the K
// largest, and one sort orders the result.
__global__ void __launch_bounds__(TK_NT, 1)
    topk_merge_kernel(const int32_t* __restrict__ lens, idx_problem p, int use_p, int max_len, int K, int P,
                      const uint64_t* __restrict__ lists, int n_chunks, int32_t* __restrict__ out_ids,
                      float* __restrict__ out_scores, const int32_t* __restrict__ row_mask) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  TkShared& sh = *reinterpret_cast<TkShared*>(tk_smem);
  uint64_t* pair = reinterpret_cast<uint64_t*>(sh.keys);   // [best P | chunk P]
  uint64_t* best = sh.cand;
  const int64_t m = blockIdx.x;
  if (row_mask && !row_mask[m]) return;
  int n;
  if (use_p) {
    int64_t off;
    row_extent(p, m, &off, &n);
  } else {
    n = lens[m];
    n = n < 0 ? 0 : (n > max_len ? max_len : n);
  }
  if (n <= TK_CH) return;   // written by the chunk kernel
  const int chunks = (int)((n + TK_CH - 1) / TK_CH);
  const uint64_t* src = lists + (int64_t)m * n_chunks * P;
  for (int i = threadIdx.x; i < P; i += TK_NT) pair[i] = src[i];
  for (int c = 1; c < chunks; ++c) {
    const uint64_t* s2 = src + (int64_t)c * P;
    for (int i = threadIdx.x; i < P; i += TK_NT) pair[P + i] = s2[i];
    __syncthreads();
    select_exact_k(sh, pair, 2 * P, K, best);     // at least K real entries: chunk 0 alone has K
    for (int i = threadIdx.x; i < P; i += TK_NT) pair[i] = i < K ? best[i] : 0ull;
    __syncthreads();
  }
  // the running set holds exactly K real entries (chunk 0 alone has K)
  const uint64_t* sorted = order_desc(sh, pair, K, P, best);
  for (int j = threadIdx.x; j < K; j += TK_NT) {
    const uint64_t v = sorted[j];
    out_ids[m * K + j] = v ? key_id((uint32_t)v) : -1;
    if (out_scores) out_scores[m * K + j] = v ? key_score((uint32_t)(v >> 32)) : -__int_as_float(0x7f800000);
  }
}

static int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

size_t topk_dense_ws(int64_t M, int max_len, int K) {
  if (max_len <= TK_CH || M <= 0) return 0;
  const int n_chunks = (max_len + TK_CH - 1) / TK_CH;
  return (size_t)M * n_chunks * pow2_at_least(K) * sizeof(uint64_t);
}

cudaError_t launch_topk_dense(const float* scores, int64_t ld, const int32_t* lens, const idx_problem* p_or_null,
                              int64_t M, int max_len, int K, int32_t* out_ids, float* out_scores, void* ws,
                              cudaStream_t st, const int32_t* id_map, int64_t id_ld, const int32_t* row_mask) {
  if (M <= 0) return cudaSuccess;
  const int P = pow2_at_least(K);
  const int n_chunks = max_len > 0 ? (max_len + TK_CH - 1) / TK_CH : 1;
  idx_problem p{};
  if (p_or_null) p = *p_or_null;
  const size_t smem = sizeof(TkShared);
  cudaError_t e = cudaFuncSetAttribute(topk_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (n_chunks > 65535) return cudaErrorInvalidValue;
  dim3 grid((unsigned)M, (unsigned)n_chunks);
  topk_chunk_kernel<<<grid, TK_NT, smem, st>>>(scores, ld, lens, p, p_or_null ? 1 : 0, max_len, K, P, out_ids,
                                               out_scores, (uint64_t*)ws, n_chunks, id_map, id_ld, row_mask);
  e = cudaGetLastError();
  if (e != cudaSuccess || n_chunks == 1) return e;
  e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_merge_kernel<<<(unsigned)M, TK_NT, smem, st>>>(lens, p, p_or_null ? 1 : 0, max_len, K, P, (const uint64_t*)ws,
                                                      n_chunks, out_ids, out_scores, row_mask);
  return cudaGetLastError();
}

}  // namespace idx
