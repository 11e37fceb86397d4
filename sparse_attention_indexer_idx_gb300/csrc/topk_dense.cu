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
//   3. the candidates are bitonic-sorted and the first K are the chunk's top-K.
// A row of one chunk writes its result directly.  Longer rows write every
// chunk's sorted top-K list to the workspace, and a merge kernel folds the
// lists pairwise with bitonic merges, keeping the best K each time.
#include "internal.h"
#include "topk.cuh"

namespace idx {

constexpr int TK_NT = 512;
constexpr int TK_E = 64;
constexpr int TK_CH = TK_NT * TK_E;
constexpr int TK_NS = 1024;
constexpr int TK_CAP = 8192;

struct TkShared {
  uint64_t cand[TK_CAP];
  uint32_t samp[TK_NS];
  uint32_t hist[kTopkBins];
  uint32_t red[TK_NT / 32];
  uint32_t cnt;
  uint32_t found_bin;
  uint32_t found_above;
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

// Bitonic merge of a bitonic sequence of n (power of two) values, descending.
__device__ void bitonic_merge_desc(uint64_t* v, int n) {
  for (int stride = n >> 1; stride > 0; stride >>= 1) {
    for (int t = threadIdx.x; t < (n >> 1); t += TK_NT) {
      const int lo = 2 * t - (t & (stride - 1));
      const int hi = lo + stride;
      const uint64_t a = v[lo], b = v[hi];
      if (a < b) {
        v[lo] = b;
        v[hi] = a;
      }
    }
    __syncthreads();
  }
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int32_t id) {
  return ((uint64_t)key << 32) | id_key(id);
}

// Warp-aggregated append of the flagged composite to sh.cand.
__device__ __forceinline__ void append(TkShared& sh, bool take, uint64_t v) {
  const unsigned mask = __ballot_sync(0xffffffffu, take);
  if (!mask) return;
  const int lane = threadIdx.x & 31;
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(&sh.cnt, (uint32_t)__popc(mask));
  base = __shfl_sync(0xffffffffu, base, 0);
  if (take) {
    const uint32_t pos = base + __popc(mask & ((1u << lane) - 1u));
    if (pos < TK_CAP) sh.cand[pos] = v;
  }
}

// Exact radix select over the register-resident keys: the `want`-th largest
// value of f (11+11+10-bit digits) among the flagged elements.
template <class F, class Flag>
__device__ uint32_t reg_radix_select(TkShared& sh, uint32_t want, F f, Flag flag, uint32_t* above_out) {
  uint32_t prefix = 0, mask = 0, remaining = want;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3ffu : 0x7ffu;
    for (int b = threadIdx.x; b < kTopkBins; b += TK_NT) sh.hist[b] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < TK_E; ++j) {
      if (flag(j)) {
        const uint32_t k = f(j);
        if ((k & mask) == prefix) atomicAdd(&sh.hist[(k >> shift) & dmask], 1u);
      }
    }
    __syncthreads();
    // suffix search over the bins, high to low (4 bins per thread)
    const int nb = (int)dmask + 1;
    uint32_t loc[4], sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int bin = nb - 1 - (threadIdx.x * 4 + q);
      loc[q] = bin >= 0 ? sh.hist[bin] : 0u;
      sum += loc[q];
    }
    uint32_t incl = sum;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sh.red[wid] = incl;
    __syncthreads();
    uint32_t run = incl - sum;
    for (int w = 0; w < wid; ++w) run += sh.red[w];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int bin = nb - 1 - (threadIdx.x * 4 + q);
      if (bin >= 0 && run < remaining && run + loc[q] >= remaining) {
        sh.found_bin = (uint32_t)bin;
        sh.found_above = run;
      }
      run += loc[q];
    }
    __syncthreads();
    remaining -= sh.found_above;
    prefix |= sh.found_bin << shift;
    mask |= dmask << shift;
    __syncthreads();
  }
  *above_out = want - remaining;
  return prefix;
}

// One chunk of one row.  Writes the final top-K when the row is one chunk,
// else the chunk's sorted top-K list (P = next_pow2(K) composites, 0-padded).
__global__ void __launch_bounds__(TK_NT, 1)
    topk_chunk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ lens,
                      idx_problem p, int use_p, int max_len, int K, int P, int32_t* __restrict__ out_ids,
                      float* __restrict__ out_scores, uint64_t* __restrict__ lists, int n_chunks) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  TkShared& sh = *reinterpret_cast<TkShared*>(tk_smem);
  const int64_t m = blockIdx.x;
  const int c = blockIdx.y;
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

  uint32_t k[TK_E];
#pragma unroll
  for (int j = 0; j < TK_E; ++j) {
    const int i = tid + j * TK_NT;
    k[j] = i < cn ? score_key(__ldg(row + i)) : 0u;   // 0 sorts below every finite score
  }
  if (tid == 0) sh.cnt = 0;
  __syncthreads();

  if (cn <= K) {
#pragma unroll
    for (int j = 0; j < TK_E; ++j) {
      const int i = tid + j * TK_NT;
      append(sh, i < cn, composite(k[j], (int32_t)(base + i)));
    }
  } else {
    // 1. sample threshold
    sh.samp[tid] = k[0];
    sh.samp[tid + TK_NT] = k[TK_E / 2];
    __syncthreads();
    bitonic_desc<uint32_t>(sh.samp, TK_NS, TK_NT);
    const int nvalid = min(TK_NT, cn) + max(0, min(TK_NT, cn - (TK_E / 2) * TK_NT));
    const float expect = (float)nvalid * (float)K / (float)cn;
    int r = (int)ceilf(1.2f * expect + 3.0f * sqrtf(expect)) + 1;
    r = r < 1 ? 1 : (r > nvalid ? nvalid : r);
    uint32_t T = 0;
    bool ok = false;
#pragma unroll 1
    for (int attempt = 0; attempt < 4; ++attempt) {
      T = sh.samp[r - 1];
      uint32_t local = 0;
#pragma unroll
      for (int j = 0; j < TK_E; ++j) local += (k[j] >= T && k[j] != 0u) ? 1u : 0u;
      const uint32_t count = block_sum_u32(local, sh.red);
      if (count > (uint32_t)TK_CAP) break;
      if (count >= (uint32_t)K) {
        ok = true;
        break;
      }
      if (r == nvalid) break;
      r = min(nvalid, 2 * r);
    }
    if (ok) {
#pragma unroll
      for (int j = 0; j < TK_E; ++j) {
        const int i = tid + j * TK_NT;
        append(sh, k[j] >= T && k[j] != 0u, composite(k[j], (int32_t)(base + i)));
      }
    } else {
      // 2'. exact: radix select of the K-th key, then of the ids among its ties
      uint32_t above;
      auto key_f = [&](int j) { return k[j]; };
      auto valid = [&](int j) { return tid + j * TK_NT < cn; };
      const uint32_t KT = reg_radix_select(sh, (uint32_t)K, key_f, valid, &above);
      const uint32_t need = (uint32_t)K - above;
      auto tie = [&](int j) { return tid + j * TK_NT < cn && k[j] == KT; };
      auto idk = [&](int j) { return id_key((int32_t)(base + tid + j * TK_NT)); };
      uint32_t above2;
      const uint32_t IT = reg_radix_select(sh, need, idk, tie, &above2);
#pragma unroll
      for (int j = 0; j < TK_E; ++j) {
        const int i = tid + j * TK_NT;
        const bool take = i < cn && (k[j] > KT || (k[j] == KT && id_key((int32_t)(base + i)) >= IT));
        append(sh, take, composite(k[j], (int32_t)(base + i)));
      }
    }
  }
  __syncthreads();
  const int cnt = (int)min(sh.cnt, (uint32_t)TK_CAP);
  int S = 1;
  while (S < cnt) S <<= 1;
  for (int i = cnt + tid; i < S; i += TK_NT) sh.cand[i] = 0ull;
  __syncthreads();
  if (S > 1) bitonic_desc<uint64_t>(sh.cand, S, TK_NT);
  if (single) {
    for (int j = tid; j < K; j += TK_NT) {
      const uint64_t v = j < cnt ? sh.cand[j] : 0ull;
      out_ids[m * K + j] = v ? key_id((uint32_t)v) : -1;
      if (out_scores) out_scores[m * K + j] = v ? key_score((uint32_t)(v >> 32)) : -__int_as_float(0x7f800000);
    }
  } else {
    uint64_t* dst = lists + ((int64_t)m * n_chunks + c) * P;
    for (int j = tid; j < P; j += TK_NT) dst[j] = (j < K && j < cnt) ? sh.cand[j] : 0ull;
  }
}

// Folds the sorted chunk lists of every multi-chunk row into its top-K.
__global__ void __launch_bounds__(TK_NT, 1)
    topk_merge_kernel(const int32_t* __restrict__ lens, idx_problem p, int use_p, int max_len, int K, int P,
                      const uint64_t* __restrict__ lists, int n_chunks, int32_t* __restrict__ out_ids,
                      float* __restrict__ out_scores) {
  extern __shared__ __align__(16) uint8_t tk_smem[];
  uint64_t* buf = reinterpret_cast<uint64_t*>(tk_smem);   // 2P
  const int64_t m = blockIdx.x;
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
  for (int i = threadIdx.x; i < P; i += TK_NT) buf[i] = src[i];
  for (int c = 1; c < chunks; ++c) {
    const uint64_t* s2 = src + (int64_t)c * P;
    for (int i = threadIdx.x; i < P; i += TK_NT) buf[P + i] = s2[P - 1 - i];   // reversed: bitonic
    __syncthreads();
    bitonic_merge_desc(buf, 2 * P);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < K; j += TK_NT) {
    const uint64_t v = buf[j];
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
                              cudaStream_t st) {
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
                                               out_scores, (uint64_t*)ws, n_chunks);
  e = cudaGetLastError();
  if (e != cudaSuccess || n_chunks == 1) return e;
  const size_t msmem = 2 * (size_t)P * sizeof(uint64_t);
  e = cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msmem);
  if (e != cudaSuccess) return e;
  topk_merge_kernel<<<(unsigned)M, TK_NT, msmem, st>>>(lens, p, p_or_null ? 1 : 0, max_len, K, P, (const uint64_t*)ws,
                                                       n_chunks, out_ids, out_scores);
  return cudaGetLastError();
}

}  // namespace idx
