// DoSA safe-upper-bound pruning of the indexer top-K
// ("DoSA：用安全上界减少 Indexer 的完整打分", sections 2, 3.1, 3.2, 4).
//
// Pipeline (one stream, no host synchronisation):
//   seeds      per row a set of distinct visible seed keys, as a bitmap and an
//              ascending list: the caller's lists, the cold rule of section 4
//              for one shared key sequence (four evenly spaced representative
//              queries fully scored; keys ranked by how many representative
//              top-K lists hold them, then their best representative score,
//              then id), or floor(i L / n) for per-row keys;
//   seed top-K the seeds scored with every head by the same tensor-core score
//              kernel as the unpruned path, then the exact top-K; tau = the
//              K-th seed score (section 2 step 1);
//   planner    per query: R retained heads (largest |w_h| ||q_h||), an anchor
//              q_j, beta = max(0, q_h.q_j/||q_j||^2) and ||q_h - beta q_j|| for
//              every omitted positive head (section 3.1), folded weights
//              w'_j = w_j + sum beta_h w_h, c = sum w_h ||d_h||, the omitted
//              negative heads active (q_h.k > 0) on at least act_freq_min of the
//              seed samples and their |w|-weighted aggregate a_A (section 3.2),
//              a_A rounded to bf16 with the rounding distance added to the
//              margin, plus gamma * (sum_h |w_h| ||q_h|| + ||a_A||);
//   bound scan the tensor-core kernel in bound mode: U >= tau sets the key's
//              bit in the row's candidate bitmap; compaction turns the bitmap
//              into an ascending id list (a row over its capacity falls back);
//   rescoring  the candidates scored exactly (gathered tiles, same MMA shape
//              per pair); survivors have s >= tau (section 2 step 3).  With the
//              shared stream (section 4, one key sequence): queries in groups
//              of four; a candidate that at least two rows of the group kept
//              and that all of them can see is scored once for the four (one
//              MMA tile, N = 4H), the rest on their own rows' lists; a row
//              keeps the group records that it can see, that are not its seeds
//              and whose s >= tau;
//   merge      exact top-K of the seed top-K plus the survivors;
//   fallback   rows with too few seeds or an overflowing candidate list are
//              recomputed on the unpruned path.
// The output equals idx_topk bit for bit: every exact score comes from the
// same kernel family, the bound exceeds the computed score (margin), ties at
// tau are kept, and the final selection uses the same total order.
#include <cstring>

#include "internal.h"
#include "topk.cuh"

namespace idx {

constexpr int kVec = 32;          // prepared vectors per query: R retained + aggregate at row 31
constexpr int kPlanThreads = 256;

__global__ void fill_i32_kernel(int32_t* p, int64_t n, int32_t v) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) p[i] = v;
}

static cudaError_t fill_i32(void* p, int64_t n, int32_t v, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fill_i32_kernel<<<(unsigned)blocks, 256, 0, st>>>((int32_t*)p, n, v);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ seeds --

__global__ void min_len_kernel(idx_problem p, int32_t* out) {
  __shared__ int32_t red[32];
  int32_t mn = 0x7fffffff;
  for (int64_t m = threadIdx.x; m < p.M; m += blockDim.x) {
    int64_t off;
    int len;
    row_extent(p, m, &off, &len);
    mn = len < mn ? len : mn;
  }
  for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mn;
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t v = 0x7fffffff;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) v = min(v, red[w]);
    *out = p.M > 0 ? v : 0;
  }
}

struct Reps {
  int64_t m[4];
  int n;
};

__global__ void gather_reps_kernel(idx_problem p, Reps r, const int32_t* common_len, uint16_t* q_out, float* w_out,
                                   int32_t* len_out) {
  const int i = blockIdx.x;
  const int64_t m = r.m[i];
  const int64_t hd = (int64_t)p.H * p.D;
  const uint16_t* q = (const uint16_t*)p.q + m * hd;
  for (int64_t e = threadIdx.x; e < hd; e += blockDim.x) q_out[i * hd + e] = q[e];
  for (int h = threadIdx.x; h < p.H; h += blockDim.x) w_out[i * p.H + h] = p.w[m * p.H + h];
  if (threadIdx.x == 0) len_out[i] = *common_len;
}

__global__ void rep_count_kernel(const int32_t* rep_ids, int nrep, int K, uint32_t* count) {
  const int64_t n = (int64_t)nrep * K;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t id = rep_ids[i];
    if (id >= 0) atomicAdd(&count[id], 1u);
  }
}

// The best representative score of every key of [0, Lc), as an ordered key.
__global__ void rep_best_kernel(const float* rep_sc, int64_t ld, int nrep, const int32_t* common_len,
                                uint32_t* best) {
  const int Lc = *common_len;
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < Lc; k += gridDim.x * blockDim.x) {
    float b = rep_sc[k];
    for (int r = 1; r < nrep; ++r) b = fmaxf(b, rep_sc[r * ld + k]);
    best[k] = score_key(b);
  }
}

// Cold rule: the n_seed best keys of [0, Lc) by (count desc, best rep score
// desc, id asc) are marked in the shared seed bitmap.
constexpr int kColdThreads = 1024;
struct DummyRow {};

__global__ void __launch_bounds__(kColdThreads) cold_select_kernel(const uint32_t* count, const uint32_t* best,
                                                                   const int32_t* common_len, int n_seed,
                                                                   uint32_t* seedbits) {
  __shared__ TopkShared<kColdThreads> sh;
  __shared__ uint32_t cnt_hist[8];
  const int Lc = *common_len;
  auto best_key = [&](int k) { return best[k]; };
  if (Lc <= n_seed) {
    for (int k = threadIdx.x; k < Lc; k += kColdThreads) atomicOr(&seedbits[k >> 5], 1u << (k & 31));
    return;
  }
  if (threadIdx.x < 8) cnt_hist[threadIdx.x] = 0;
  __syncthreads();
  for (int k = threadIdx.x; k < Lc; k += kColdThreads) atomicAdd(&cnt_hist[min(count[k], 7u)], 1u);
  __syncthreads();
  // c*: the count level where the cumulative number of keys (from the top) reaches n_seed
  int cstar = 0;
  uint32_t above = 0;
  {
    uint32_t cum = 0;
    for (int c = 7; c >= 0; --c) {
      if (cum + cnt_hist[c] >= (uint32_t)n_seed) {
        cstar = c;
        above = cum;
        break;
      }
      cum += cnt_hist[c];
    }
  }
  const uint32_t need = (uint32_t)n_seed - above;
  DummyRow dr;
  auto at_c = [&](int k) { return (int)min(count[k], 7u) == cstar; };
  uint32_t above_b, eq_b;
  const uint32_t T = topk_radix_select<kColdThreads>(sh, dr, Lc, need, best_key, at_c, &above_b, &eq_b);
  const uint32_t need_t = need - above_b;
  uint32_t I = 0;
  if (eq_b != need_t) {
    auto idk = [&](int k) { return id_key(k); };
    auto tie = [&](int k) { return at_c(k) && best_key(k) == T; };
    uint32_t a2, e2;
    I = topk_radix_select<kColdThreads>(sh, dr, Lc, need_t, idk, tie, &a2, &e2);
  }
  for (int k = threadIdx.x; k < Lc; k += kColdThreads) {
    const int c = (int)min(count[k], 7u);
    bool take = c > cstar;
    if (c == cstar) {
      const uint32_t bk = best_key(k);
      take = bk > T || (bk == T && id_key(k) >= I);
    }
    if (take) atomicOr(&seedbits[k >> 5], 1u << (k & 31));
  }
}

__global__ void strided_seeds_kernel(idx_problem p, int n_seed, uint32_t* bits, int64_t W) {
  const int64_t m = blockIdx.x;
  int64_t off;
  int L;
  row_extent(p, m, &off, &L);
  const int n = L < n_seed ? L : n_seed;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t x = ((int64_t)i * L) / n;
    atomicOr(&bits[m * W + (x >> 5)], 1u << (x & 31));
  }
}

__global__ void caller_seeds_kernel(idx_problem p, const int32_t* seed_ids, int seed_ld, uint32_t* bits, int64_t W) {
  const int64_t m = blockIdx.x;
  int64_t off;
  int L;
  row_extent(p, m, &off, &L);
  for (int j = threadIdx.x; j < seed_ld; j += blockDim.x) {
    const int32_t id = seed_ids[m * seed_ld + j];
    if (id >= 0 && id < L) atomicOr(&bits[m * W + (id >> 5)], 1u << (id & 31));
  }
}

// Bitmap row b[0..W) -> ascending id list out[0..cap) (block of kListThreads
// threads, wsum: 32 words of shared memory); returns the number of set bits.
constexpr int kListThreads = 1024;
__device__ int64_t bits_row_to_list(const uint32_t* b, int64_t W, int32_t* out, int64_t cap, uint32_t* wsum) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int64_t run = 0;
  for (int64_t w0 = 0; w0 < W; w0 += kListThreads) {
    const int64_t w = w0 + threadIdx.x;
    const uint32_t word = w < W ? b[w] : 0u;
    const uint32_t pc = __popc(word);
    uint32_t incl = pc;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    uint32_t woff = 0, tot = 0;
    for (int i = 0; i < kListThreads / 32; ++i) {
      if (i < wid) woff += wsum[i];
      tot += wsum[i];
    }
    int64_t pos = run + woff + incl - pc;
    uint32_t v = word;
    while (v) {
      const int bit = __ffs(v) - 1;
      v &= v - 1;
      if (pos < cap) out[pos] = (int32_t)(w * 32 + bit);
      ++pos;
    }
    run += tot;
    __syncthreads();
  }
  return run;
}

// Seed bitmap row -> ascending id list (at most cap entries) and its count.
__global__ void __launch_bounds__(kListThreads) bits_to_list_kernel(const uint32_t* bits, int64_t W, int32_t* list,
                                                                     int64_t cap, int32_t* cnt) {
  __shared__ uint32_t wsum[32];
  const int64_t r = blockIdx.x;
  const int64_t run = bits_row_to_list(bits + r * W, W, list + r * cap, cap, wsum);
  if (threadIdx.x == 0) cnt[r] = (int32_t)(run < cap ? run : cap);
}

// Candidate bitmap row m (the words below its visible length) -> ascending id
// list; cand_cnt = all candidates, cand_n = those to rescore (0 for a row on
// the unpruned path; a row over cap joins it with status bit 2).
__global__ void __launch_bounds__(kListThreads) cand_compact_kernel(idx_problem p, const uint32_t* bits, int64_t W,
                                                                     int32_t* status, int32_t* cand, int64_t cap,
                                                                     int32_t* cand_cnt, int32_t* cand_n) {
  __shared__ uint32_t wsum[32];
  const int64_t m = blockIdx.x;
  if (status[m] != 0) {
    if (threadIdx.x == 0) {
      cand_cnt[m] = 0;
      cand_n[m] = 0;
    }
    return;
  }
  int64_t off;
  int len;
  row_extent(p, m, &off, &len);
  int64_t nw = ((int64_t)len + 31) / 32;
  nw = nw < W ? nw : W;
  const int64_t run = bits_row_to_list(bits + m * W, nw, cand + m * cap, cap, wsum);
  if (threadIdx.x == 0) {
    cand_cnt[m] = (int32_t)run;
    if (run > cap) status[m] |= 2;
    cand_n[m] = run > cap ? 0 : (int32_t)run;
  }
}

// Copies the shared seed keys (and scales) into a contiguous buffer.
__global__ void gather_keys_kernel(idx_problem p, const int32_t* list, const int32_t* cnt, void* out_keys,
                                   float* out_scale) {
  const int n = *cnt;
  const int row_bytes = p.k_dtype == IDX_FP8_E4M3 ? 128 : 256;
  const int words = row_bytes / 16;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < (int64_t)n * words;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / words, c = t % words;
    const int64_t id = list[i];
    const uint4* src = (const uint4*)((const char*)p.keys + id * row_bytes);
    ((uint4*)((char*)out_keys + i * row_bytes))[c] = src[c];
    if (c == 0 && out_scale) out_scale[i] = p.key_scale[id];
  }
}

__global__ void broadcast_i32_kernel(const int32_t* src, int32_t* dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = *src;
}

// tau, status and the active-row mask after the seed top-K.
__global__ void seed_status_kernel(int64_t M, int K, const int32_t* seed_cnt, int shared, const float* stop_sc,
                                   float* tau, int32_t* status, int32_t* active) {
  for (int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; m < M; m += (int64_t)gridDim.x * blockDim.x) {
    const int32_t c = seed_cnt[shared ? 0 : m];
    const bool ok = c >= K;
    tau[m] = ok ? stop_sc[m * K + K - 1] : 0.0f;
    status[m] = ok ? 0 : 1;
    active[m] = ok ? 1 : 0;
  }
}

// ---------------------------------------------------------------- planner --

struct PlanArgs {
  idx_problem p;
  int R;
  int n_sample;
  float act_min;
  float gamma;
  const int32_t* seed_list;   // [rows, list_ld]
  int64_t list_ld;
  const int32_t* seed_cnt;
  int shared_seeds;
  int32_t* active;            // cleared for a row predicted to overflow
  int32_t* status;            // bit 4 set for such a row
  const float* tau;           // [M]
  int64_t cap;                // candidate capacity per row
  uint16_t* qprep;            // [M, 32, D] bf16, or the bound's group layout (glayout)
  int glayout;
  float* wfold;               // [M, 32]
  float* coef;                // [M]
  // per (row, head) record of the plan: the head's role (position r >= 0 among
  // the retained heads; 1024 + j for an omitted positive head anchored on head
  // j; -2 for an omitted negative head in A; -1 otherwise), beta and ||d_h||
  int32_t* plan_head;         // [M, H]
  float* plan_beta;           // [M, H]
  float* plan_dn;             // [M, H]
};

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f_to_bf16_rn(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ float e4m3_to_f(uint8_t b) {
  const int s = b >> 7, e = (b >> 3) & 0xf, m = b & 7;
  float v = e == 0 ? (float)m * 0.001953125f : ldexpf(1.0f + (float)m * 0.125f, e - 7);
  return s ? -v : v;
}

// The planner's tiles: rows of D = 128 bf16 values, kPS elements apart (the
// 8 extra elements put the 8 rows x 4 words of an mma fragment load in 32
// different banks).
constexpr int kPS = 136;

// Rows row_of(i), i < n, of `base` (128 values each: bf16, or e4m3 codes --
// which bf16 holds exactly) into dst[i * kPS + d] as bf16; rows n..n_pad-1 are
// zero.  By the whole block: every thread issues up to four 16-byte loads
// before it stores any, so the rows arrive in about one memory latency.
template <class RowOf>
__device__ void block_load_rows_bf16(const void* base, int dtype, int n, int n_pad, uint16_t* dst, RowOf row_of) {
  const int esz = dtype == IDX_FP8_E4M3 ? 1 : 2;
  const int per = 16 / esz;                 // values per 16-byte chunk
  const int cpr = 128 / per;                // chunks per row
  const int total = n_pad * cpr;
  for (int c0 = 0; c0 < total; c0 += 4 * kPlanThreads) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * kPlanThreads + threadIdx.x;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (c < total && c / cpr < n) {
        const int64_t row = row_of(c / cpr);
        v[u] = *reinterpret_cast<const uint4*>(static_cast<const char*>(base) + (row * 128 + (c % cpr) * per) * esz);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * kPlanThreads + threadIdx.x;
      if (c >= total) continue;
      uint16_t* o = dst + (c / cpr) * kPS + (c % cpr) * per;
      if (dtype == IDX_FP8_E4M3) {
        const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t ow[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t lo = f_to_bf16_rn(e4m3_to_f((uint8_t)(w4[(2 * e) >> 2] >> (8 * ((2 * e) & 3)))));
          const uint32_t hi = f_to_bf16_rn(e4m3_to_f((uint8_t)(w4[(2 * e + 1) >> 2] >> (8 * ((2 * e + 1) & 3)))));
          ow[e] = lo | (hi << 16);
        }
        reinterpret_cast<uint4*>(o)[0] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        reinterpret_cast<uint4*>(o)[1] = make_uint4(ow[4], ow[5], ow[6], ow[7]);
      } else {
        *reinterpret_cast<uint4*>(o) = v[u];
      }
    }
  }
}

// Two bf16 (elements col, col + 1 of a tile row; col even) as one word.
__device__ __forceinline__ uint32_t tile_word(const uint16_t* t, int row, int col) {
  return *reinterpret_cast<const uint32_t*>(t + row * kPS + col);
}

// d += A (16 x 16, rows of `a` from row a0) times B (16 x 8, B[k][n] = row
// n of `b`, entry k; b_ok false: that column is zero), over D = 128 in eight
// K steps, on the warp's tensor core (bf16 products are exact in the fp32
// accumulator).  Fragment positions: lane = 4 g + t holds d[0], d[1] at row
// g, columns 2t, 2t + 1 and d[2], d[3] at row g + 8.
__device__ __forceinline__ void warp_mma_rows(float (&d)[4], const uint16_t* a, int a0, const uint16_t* brow,
                                              bool b_ok) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int k0 = 0; k0 < 128; k0 += 16) {
    const uint32_t x0 = tile_word(a, a0 + g, k0 + 2 * t), x1 = tile_word(a, a0 + g + 8, k0 + 2 * t);
    const uint32_t x2 = tile_word(a, a0 + g, k0 + 2 * t + 8), x3 = tile_word(a, a0 + g + 8, k0 + 2 * t + 8);
    const uint32_t y0 = b_ok ? *reinterpret_cast<const uint32_t*>(brow + k0 + 2 * t) : 0u;
    const uint32_t y1 = b_ok ? *reinterpret_cast<const uint32_t*>(brow + k0 + 2 * t + 8) : 0u;
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(x0), "r"(x1), "r"(x2), "r"(x3), "r"(y0), "r"(y1));
  }
}

// Shared memory of the planner for H heads and n_sample samples.
__host__ __device__ constexpr size_t plan_smem_bytes(int H, int n_sample) {
  return (size_t)2 * kPS * ((size_t)H + (size_t)((n_sample + 15) / 16 * 16) + 32) +
         (size_t)4 * ((size_t)H * 33 + 5 * (size_t)H + 128 + 32 + (size_t)((n_sample + 15) / 16 * 16) +
                      4 * (size_t)H + 33 + 24);
}

// One thread block per query (8 warps).  The three small contractions of the
// plan -- q_h . q_j for every head and retained head, q_h . k over the seed
// samples, and the prepared vectors against the estimate keys -- run as warp
// tensor-core tiles (mma.sync m16n8k16, bf16 in, fp32 out) over bf16 tiles in
// shared memory; the rest is per head or per key.
__global__ void __launch_bounds__(kPlanThreads) dosa_plan_kernel(PlanArgs a) {
  extern __shared__ __align__(16) uint8_t pl_raw[];
  const idx_problem& p = a.p;
  const int64_t m = blockIdx.x;
  const int H = p.H, R = a.R;
  constexpr int D = 128;
  const int NSP = (a.n_sample + 15) / 16 * 16;   // sample rows (padded to whole tiles)
  uint16_t* qs = reinterpret_cast<uint16_t*>(pl_raw);   // H rows: q_h
  uint16_t* ks = qs + H * kPS;                   // NSP rows: seed samples, later the estimate keys
  uint16_t* vs = ks + NSP * kPS;                 // 32 rows: the prepared vectors (retained, zero, a_A at 31)
  float* gram = reinterpret_cast<float*>(vs + 32 * kPS);   // [H][33]: q_h . q_{rlist[r]}
  float* qn2 = gram + H * 33;                    // H: ||q_h||^2
  float* mag = qn2 + H;                          // H: |w_h| ||q_h||
  float* beta = mag + H;                         // H
  float* dn = beta + H;                          // H: ||d_h||
  float* wq = dn + H;                            // H: w_h
  float* aggv = wq + H;                          // D: a_A
  float* wfs = aggv + D;                         // 32: folded weights
  float* kn2 = wfs + 32;                         // NSP: ||k||^2 of the estimate keys
  int* anchor = reinterpret_cast<int*>(kn2 + NSP);   // H
  int* ret_pos = anchor + H;                     // H: position among retained, -1 if omitted
  int* act = ret_pos + H;                        // H: activation counts
  int* rlist = act + H;                          // 32: retained heads ascending
  int* a_list = rlist + 32;                      // H + 1: A's heads ascending, then their count
  float* red = reinterpret_cast<float*>(a_list + H + 1);   // 2 x 8 partial sums, coef, pass count
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  constexpr int nw = kPlanThreads / 32;

  float* wout = a.wfold + m * kVec;
  // prepared row r of this query (r < 31: vector r, 31: the aggregate; the group
  // layout keeps 16 vectors per query and the group's aggregates in one block,
  // with one zero row per query behind them)
  const int nvec = a.glayout ? 16 : kVec - 1;
  auto qrow = [&](int r) -> uint16_t* {
    if (!a.glayout) return a.qprep + (m * kVec + r) * D;
    const int64_t gg = m >> 3, qi = m & 7;
    return a.qprep + (gg * 144 + (r == 31 ? 128 + qi : (r == 32 ? 136 + qi : qi * 16 + r))) * D;
  };
  if (!a.active[m]) {
    for (int i = tid; i < (nvec + 2) * D; i += kPlanThreads) {
      const int r = i / D;
      if (r < nvec) qrow(r)[i % D] = 0;
      else if (r == nvec) qrow(31)[i % D] = 0;
      else if (a.glayout) qrow(32)[i % D] = 0;
    }
    for (int i = tid; i < kVec; i += kPlanThreads) wout[i] = 0.0f;
    if (tid == 0) a.coef[m] = 0.0f;
    return;
  }
  for (int h = tid; h < H; h += kPlanThreads) {
    wq[h] = p.w[m * H + h];
    act[h] = 0;
  }
  block_load_rows_bf16(p.q, IDX_BF16, H, H, qs, [&](int h) { return (int64_t)(m * H + h); });
  // sample keys: seed[floor(i n / ns)], i < ns = min(n_sample, n)
  const int32_t* sl = a.seed_list + (a.shared_seeds ? 0 : m * a.list_ld);
  const int n = a.seed_cnt[a.shared_seeds ? 0 : m];
  const int ns = n < a.n_sample ? n : a.n_sample;
  const int64_t kbase = p.key_off ? p.key_off[m] : 0;
  block_load_rows_bf16(p.keys, p.k_dtype, ns, NSP, ks, [&](int si) {
    return kbase + (int64_t)sl[n <= a.n_sample ? si : (int)(((int64_t)si * n) / a.n_sample)];
  });
  __syncthreads();
  // ||q_h||^2 and |w_h| ||q_h||, one warp per head (lane: elements 4 lane .. 4 lane + 3)
  for (int h = wid; h < H; h += nw) {
    const uint32_t w0 = tile_word(qs, h, 4 * lane), w1 = tile_word(qs, h, 4 * lane + 2);
    const float x[4] = {bf16_to_f((uint16_t)w0), bf16_to_f((uint16_t)(w0 >> 16)), bf16_to_f((uint16_t)w1),
                        bf16_to_f((uint16_t)(w1 >> 16))};
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) s = __fmaf_rn(x[e], x[e], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      qn2[h] = s;
      mag[h] = fabsf(wq[h]) * sqrtf(s);
    }
  }
  __syncthreads();
  // retained heads: the R largest |w_h| ||q_h||, ties to the lower head (the
  // rank of head h counted by one warp, its lanes over the other heads)
  for (int h = wid; h < H; h += nw) {
    const float mh = mag[h];
    unsigned rank = 0;
    for (int q = lane; q < H; q += 32) {
      const float mq = mag[q];
      rank += (mq > mh || (mq == mh && q < h)) ? 1u : 0u;
    }
    rank = __reduce_add_sync(0xffffffffu, rank);
    if (lane == 0) ret_pos[h] = (int)rank < R ? 1 : -1;
  }
  __syncthreads();
  if (wid == 0) {
    // their list, ascending: one ballot per 32 heads places them
    int c = 0;
    for (int h0 = 0; h0 < H; h0 += 32) {
      const int h = h0 + lane;
      const bool r = h < H && ret_pos[h] > 0;
      const unsigned bal = __ballot_sync(0xffffffffu, r);
      if (r) {
        const int at = c + __popc(bal & ((1u << lane) - 1u));
        rlist[at] = h;
        ret_pos[h] = at;
      }
      c += __popc(bal);
    }
  }
  __syncthreads();
  // q_h . q_j for every head h and retained head j (section 3.1's beta needs them)
  {
    const int mt = H / 16, nt = (R + 7) / 8;
    for (int tile = wid; tile < mt * nt; tile += nw) {
      const int r0 = (tile / nt) * 16, c0 = (tile % nt) * 8;
      const bool ok = c0 + g < R;
      float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      warp_mma_rows(d, qs, r0, qs + (ok ? rlist[c0 + g] : 0) * kPS, ok);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = c0 + 2 * t + j;
        if (col < R) {
          gram[(r0 + g) * 33 + col] = d[j];
          gram[(r0 + g + 8) * 33 + col] = d[2 + j];
        }
      }
    }
  }
  // activation counts of every head on the samples (section 3.2: "active" is
  // q_h . k > 0; only the omitted negative heads' counts are used)
  {
    const int mt = H / 16, nt = NSP / 8;
    for (int tile = wid; tile < mt * nt; tile += nw) {
      const int r0 = (tile / nt) * 16, c0 = (tile % nt) * 8;
      float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      warp_mma_rows(d, qs, r0, ks + (c0 + g) * kPS, true);
      int lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (c0 + 2 * t + j < ns) {
          lo += d[j] > 0.0f ? 1 : 0;
          hi += d[2 + j] > 0.0f ? 1 : 0;
        }
      }
      lo += __shfl_xor_sync(0xffffffffu, lo, 1);
      lo += __shfl_xor_sync(0xffffffffu, lo, 2);
      hi += __shfl_xor_sync(0xffffffffu, hi, 1);
      hi += __shfl_xor_sync(0xffffffffu, hi, 2);
      if (t == 0) {
        if (lo) atomicAdd(&act[r0 + g], lo);
        if (hi) atomicAdd(&act[r0 + g + 8], hi);
      }
    }
  }
  __syncthreads();
  // anchors of the omitted positive heads: the retained j with the smallest
  // ||q_h - beta q_j||^2 = ||q_h||^2 - 2 beta q_h.q_j + beta^2 ||q_j||^2, ties to
  // the lower j; four threads per head (retained positions r = sub (mod 4)),
  // their bests combined in order of (r2, j)
  for (int hb = 0; hb < H; hb += kPlanThreads / 4) {
    const int h = hb + (tid >> 2), sub = tid & 3;
    int bj = -1;
    float bb = 0.0f, best = 0.0f;
    if (h < H && ret_pos[h] < 0 && wq[h] > 0.0f) {
      for (int r = sub; r < R; r += 4) {
        const int j = rlist[r];
        const float dot = gram[h * 33 + r];
        const float b = qn2[j] > 0.0f ? fmaxf(0.0f, dot / qn2[j]) : 0.0f;
        const float r2 = qn2[h] - 2.0f * b * dot + b * b * qn2[j];
        if (bj < 0 || r2 < best) {
          best = r2;
          bj = j;
          bb = b;
        }
      }
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
      const float ob = __shfl_xor_sync(0xffffffffu, bb, o), obest = __shfl_xor_sync(0xffffffffu, best, o);
      if (oj >= 0 && (bj < 0 || obest < best || (obest == best && oj < bj))) {
        bj = oj;
        bb = ob;
        best = obest;
      }
    }
    if (h < H && sub == 0) {
      anchor[h] = bj;
      beta[h] = bb;
    }
  }
  __syncthreads();
  // residual norm of the chosen decomposition, computed directly and rounded up
  for (int h = wid; h < H; h += nw) {
    float dnh = 0.0f;
    const int j = anchor[h];
    if (j >= 0) {
      const float bb = beta[h];
      float sres = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const uint32_t wh = tile_word(qs, h, 4 * lane + e), wj = tile_word(qs, j, 4 * lane + e);
        const float x0 = __fmaf_rn(-bb, bf16_to_f((uint16_t)wj), bf16_to_f((uint16_t)wh));
        const float x1 = __fmaf_rn(-bb, bf16_to_f((uint16_t)(wj >> 16)), bf16_to_f((uint16_t)(wh >> 16)));
        sres = __fmaf_rn(x0, x0, sres);
        sres = __fmaf_rn(x1, x1, sres);
      }
      for (int o = 16; o > 0; o >>= 1) sres += __shfl_xor_sync(0xffffffffu, sres, o);
      dnh = __fsqrt_ru(sres) * (1.0f + 1.0e-6f);
    }
    if (lane == 0) dn[h] = dnh;
  }
  // aggregate a_A = sum_{h in A} |w_h| q_h (heads in order), prepared rows; A's
  // heads listed first (ascending, one ballot per 32 heads)
  const float need_act = a.act_min * (float)ns;
  if (wid == 0) {
    int c = 0;
    for (int h0 = 0; h0 < H; h0 += 32) {
      const int h = h0 + lane;
      const bool inA = h < H && ret_pos[h] < 0 && wq[h] < 0.0f && ns > 0 && (float)act[h] >= need_act;
      const unsigned bal = __ballot_sync(0xffffffffu, inA);
      if (inA) a_list[c + __popc(bal & ((1u << lane) - 1u))] = h;
      c += __popc(bal);
    }
    if (lane == 0) a_list[H] = c;
  }
  __syncthreads();
  const int nA = a_list[H];
  for (int d = tid; d < D; d += kPlanThreads) {
    float sa = 0.0f;
    for (int i = 0; i < nA; ++i) {
      const int h = a_list[i];
      sa = __fmaf_rn(-wq[h], bf16_to_f(qs[h * kPS + d]), sa);
    }
    aggv[d] = sa;
    const uint16_t ab = f_to_bf16_rn(sa);
    qrow(31)[d] = ab;
    vs[31 * kPS + d] = ab;
    if (a.glayout) qrow(32)[d] = 0;
  }
  for (int i = tid; i < nvec * D; i += kPlanThreads) {
    const int r = i / D, d = i % D;
    qrow(r)[d] = r < R ? qs[rlist[r] * kPS + d] : (uint16_t)0;
  }
  for (int i = tid; i < 31 * D; i += kPlanThreads) {
    const int r = i / D, d = i % D;
    vs[r * kPS + d] = r < R ? qs[rlist[r] * kPS + d] : (uint16_t)0;
  }
  __syncthreads();   // dn complete
  for (int h = tid; h < H; h += kPlanThreads) {
    const float wh = wq[h];
    int code = -1;
    if (ret_pos[h] >= 0) code = ret_pos[h];
    else if (anchor[h] >= 0) code = 1024 + anchor[h];
    else if (wh < 0.0f && ns > 0 && (float)act[h] >= need_act) code = -2;
    a.plan_head[m * H + h] = code;
    a.plan_beta[m * H + h] = beta[h];
    a.plan_dn[m * H + h] = dn[h];
  }
  // folded weights w'_r = w_j + sum of w_h beta_h over the heads anchored on
  // j = rlist[r]: one warp per position, its lanes over the heads
  for (int r = wid; r < kVec; r += nw) {
    float wf = 0.0f;
    if (r < R) {
      const int j = rlist[r];
      for (int h = lane; h < H; h += 32)
        if (anchor[h] == j) wf = __fmaf_rn(wq[h], beta[h], wf);
      for (int o = 16; o > 0; o >>= 1) wf += __shfl_xor_sync(0xffffffffu, wf, o);
      wf += wq[j];
    }
    if (lane == 0) {
      wout[r] = wf;
      wfs[r] = wf;
    }
  }
  // margin: bf16 rounding distance of a_A, plus gamma * (sum |w_h| ||q_h|| + ||a_A||)
  float e2 = 0.0f, a2 = 0.0f;
  for (int d = tid; d < D; d += kPlanThreads) {
    const float ad = bf16_to_f(f_to_bf16_rn(aggv[d])) - aggv[d];
    e2 = __fmaf_rn(ad, ad, e2);
    a2 = __fmaf_rn(aggv[d], aggv[d], a2);
  }
  for (int o = 16; o > 0; o >>= 1) {
    e2 += __shfl_xor_sync(0xffffffffu, e2, o);
    a2 += __shfl_xor_sync(0xffffffffu, a2, o);
  }
  if (lane == 0) {
    red[wid] = e2;
    red[nw + wid] = a2;
  }
  __syncthreads();
  if (wid == 0) {
    // c = sum w_h ||d_h|| over the anchored heads and W = sum |w_h| ||q_h||, lanes
    // over the heads
    float c = 0.0f, W = 0.0f;
    for (int h = lane; h < H; h += 32) {
      const float wh = wq[h];
      if (anchor[h] >= 0) c = __fmaf_rn(wh, dn[h], c);
      W = __fmaf_rn(fabsf(wh), sqrtf(qn2[h]), W);
    }
    for (int o = 16; o > 0; o >>= 1) {
      c += __shfl_xor_sync(0xffffffffu, c, o);
      W += __shfl_xor_sync(0xffffffffu, W, o);
    }
    float E2 = 0.0f, A2 = 0.0f;
    for (int w = 0; w < nw; ++w) {
      E2 += red[w];
      A2 += red[nw + w];
    }
    float margin = __fsqrt_ru(E2) * (1.0f + 0.0009765625f) + a.gamma * (W + sqrtf(A2) * 1.01f);
    if (p.k_dtype == IDX_FP8_E4M3) {
      // FP8 keys: the tensor cores see every query-side vector v as sigma (hi + lo),
      // two e4m3 vectors with a power-of-two sigma <= max|v| / 128 over the query's
      // vectors; each element is off by at most 2^-10 sigma, so a vector by at most
      // sqrt(D) 2^-17 max_i ||v_i||.  Both the exact scores (H query heads) and the
      // bound (R retained vectors, folded weights, the aggregate) carry that error.
      float qmax = 0.0f, sw = 0.0f, swf = 1.0f;
      for (int h = 0; h < H; ++h) {
        qmax = fmaxf(qmax, sqrtf(qn2[h]));
        sw += fabsf(wq[h]);
      }
      for (int r = 0; r < kVec; ++r) swf += fabsf(wfs[r]);
      const float vmax = fmaxf(qmax, sqrtf(A2) * 1.01f + sqrtf(E2) * 1.01f);
      margin += 2.0f * sqrtf((float)D) * 7.62939453125e-6f * (sw * qmax + swf * vmax);
    }
    if (lane == 0) {
      a.coef[m] = (c + margin) * (1.0f + 1.0e-6f);
      red[2 * nw] = (c + margin) * (1.0f + 1.0e-6f);   // coef, for the estimate below
      reinterpret_cast<int*>(red)[2 * nw + 1] = 0;     // the estimate's pass count
    }
  }
  // Overflow estimate: the bound U of n_sample evenly spaced visible keys of the
  // row against tau, from the same bf16 vectors the bound scan multiplies.  A
  // row whose candidates would clearly exceed the capacity skips the bound scan
  // and is computed on the unpruned path (as an overflowing row would be); the
  // output is the same either way.
  __syncthreads();
  const float coef = red[2 * nw];
  int64_t off;
  int len;
  row_extent(p, m, &off, &len);
  const int ne = len < a.n_sample ? len : a.n_sample;   // the sample area holds n_sample keys
  if (ne <= 0) return;
  const int NEP = (ne + 15) / 16 * 16;
  block_load_rows_bf16(p.keys, p.k_dtype, ne, NEP, ks, [&](int si) { return off + ((int64_t)si * len) / ne; });
  __syncthreads();
  // ||k||^2 of the estimate keys: two threads per key (halves of the row, the
  // partner's sum added by a shuffle)
  for (int k0 = 0; k0 < ne; k0 += kPlanThreads / 2) {
    const int k = k0 + (tid >> 1), half = tid & 1;
    float s2 = 0.0f;
    if (k < ne) {
      for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 2) {
        const uint32_t w = tile_word(ks, k, c);
        const float x0 = bf16_to_f((uint16_t)w), x1 = bf16_to_f((uint16_t)(w >> 16));
        s2 = __fmaf_rn(x0, x0, s2);
        s2 = __fmaf_rn(x1, x1, s2);
      }
    }
    s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
    if (k < ne && half == 0) kn2[k] = s2;
  }
  __syncthreads();
  const float tau = a.tau[m];
  int pass = 0;
  if (wid * 16 < NEP) {
    // this warp's 16 keys against the 32 prepared vectors (four n-tiles)
    float acc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[nt][j] = 0.0f;
      warp_mma_rows(acc[nt], ks, wid * 16, vs + (nt * 8 + g) * kPS, true);
    }
    float plo = 0.0f, phi = 0.0f, alo = 0.0f, ahi = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = nt * 8 + 2 * t + j;
        if (col < R) {
          plo = __fmaf_rn(wfs[col], fmaxf(acc[nt][j], 0.0f), plo);
          phi = __fmaf_rn(wfs[col], fmaxf(acc[nt][2 + j], 0.0f), phi);
        }
        if (col == 31) {
          alo = acc[nt][j];
          ahi = acc[nt][2 + j];
        }
      }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      plo += __shfl_xor_sync(0xffffffffu, plo, o);
      phi += __shfl_xor_sync(0xffffffffu, phi, o);
      alo += __shfl_xor_sync(0xffffffffu, alo, o);
      ahi += __shfl_xor_sync(0xffffffffu, ahi, o);
    }
    if (t == 0) {
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int k = wid * 16 + g + 8 * hlf;
        if (k < ne) {
          float u = (hlf ? phi : plo) - fmaxf(hlf ? ahi : alo, 0.0f);
          u = __fmaf_rn(coef, sqrtf(kn2[k]), u);
          if (p.k_dtype == IDX_FP8_E4M3) u *= p.key_scale[off + ((int64_t)k * len) / ne];
          pass += u >= tau ? 1 : 0;
        }
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) pass += __shfl_xor_sync(0xffffffffu, pass, o);
  if (lane == 0 && pass) atomicAdd(reinterpret_cast<int*>(red) + 2 * nw + 1, pass);
  __syncthreads();
  if (tid == 0) {
    const int total = reinterpret_cast<int*>(red)[2 * nw + 1];
    const float nonseed = (float)(len - (n < len ? n : len));
    if ((float)total / (float)ne * nonseed > 1.25f * (float)a.cap) {
      a.active[m] = 0;
      a.status[m] |= 4;
    }
  }
}

// --------------------------------------------------------------- merging --

// The shared stream's output for the merge: group g's list and the scores of
// its four rows by list position.
struct GroupRecs {
  const int32_t* glist;      // [G, capg] ascending ids (nullptr: no shared stream)
  const int32_t* gcnt;       // [G]
  const float* gsc;          // [M, capg]
  int64_t capg;
  const uint32_t* seedbits;  // seed bitmap, row stride seed_stride words (0: one for all rows)
  int64_t seed_stride;
  idx_problem p;
};

// Row m of the merge input: the seed top-K then the rescored candidates (those
// below tau become -inf); also the fallback mask and the survivor count.  With
// the shared stream the row's own candidates are already in place at K.., and
// the group records that the row can see, that are not its seeds and whose
// score reaches tau follow them (in list order).  One warp per row (eight rows
// a block): the records are compacted 32 at a time by a ballot, in list order,
// with eight such steps' loads in flight per lane -- no block-wide scans.
constexpr int kMergeThreads = 256;
constexpr int kMergeRows = kMergeThreads / 32;
__global__ void __launch_bounds__(kMergeThreads) merge_rows_kernel(
    int64_t M, int K, int64_t cap, const int32_t* stop_ids, const float* stop_sc, const int32_t* cand,
    const int32_t* cand_n, const float* cand_sc, const float* tau, const int32_t* status, GroupRecs gr, float* mrg_sc,
    int32_t* mrg_id, int32_t* mrg_len, int32_t* fbmask, unsigned long long* survivors) {
  const int lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * kMergeRows + (threadIdx.x >> 5);
  if (m >= M) return;
  const int64_t ld = K + cap;
  const bool ok = status[m] == 0;
  if (lane == 0) fbmask[m] = ok ? 0 : 1;
  if (!ok) {
    if (lane == 0) mrg_len[m] = 0;
    return;
  }
  float* osc = mrg_sc + m * ld;
  int32_t* oid = mrg_id + m * ld;
  if ((K & 3) == 0 && (ld & 3) == 0) {
    // 16-byte copies (rows of K and of ld elements start 16-byte aligned)
    const float4* ss = reinterpret_cast<const float4*>(stop_sc + m * K);
    const int4* si = reinterpret_cast<const int4*>(stop_ids + m * K);
    for (int j = lane; j < K / 4; j += 32) {
      reinterpret_cast<float4*>(osc)[j] = ss[j];
      reinterpret_cast<int4*>(oid)[j] = si[j];
    }
  } else {
    for (int j = lane; j < K; j += 32) {
      osc[j] = stop_sc[m * K + j];
      oid[j] = stop_ids[m * K + j];
    }
  }
  const float t = tau[m];
  const int n = cand_n[m];
  uint32_t surv = 0;
  for (int i = lane; i < n; i += 32) {
    const float sv = cand_sc[m * cap + i];
    const bool keep = sv >= t;
    surv += keep ? 1u : 0u;
    osc[K + i] = keep ? sv : -__int_as_float(0x7f800000);
    if (!gr.glist) oid[K + i] = cand[m * cap + i];
  }
  int64_t fill = n;
  if (gr.glist) {
    // the group's records, compacted in list order behind the row's own candidates
    const int64_t g = m >> 2;
    const int gn = gr.gcnt[g];
    int64_t off;
    int len;
    row_extent(gr.p, m, &off, &len);
    const uint32_t* sbits = gr.seedbits + (gr.seed_stride ? m * gr.seed_stride : 0);
    const int32_t* gl = gr.glist + g * gr.capg;
    const float* gs = gr.gsc + m * gr.capg;
    const uint32_t lt = (1u << lane) - 1u;
    constexpr int ST = 8;   // ballot steps per round
    for (int i0 = 0; i0 < gn; i0 += 32 * ST) {
      int32_t id[ST];
      float sv[ST];
#pragma unroll
      for (int u = 0; u < ST; ++u) {
        const int i = i0 + 32 * u + lane;
        id[u] = i < gn ? gl[i] : 0x7fffffff;
        sv[u] = i < gn ? gs[i] : 0.0f;
      }
      uint32_t word[ST];
#pragma unroll
      for (int u = 0; u < ST; ++u) word[u] = id[u] < len ? sbits[id[u] >> 5] : 0xffffffffu;
#pragma unroll
      for (int u = 0; u < ST; ++u) {
        const bool keep = id[u] < len && sv[u] >= t && !((word[u] >> (id[u] & 31)) & 1u);
        const uint32_t bal = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          const int64_t pos = fill + __popc(bal & lt);
          if (pos < cap) {
            oid[K + pos] = id[u];
            osc[K + pos] = sv[u];
          }
        }
        fill += __popc(bal);
      }
    }
    if (lane == 0) surv += (uint32_t)(fill - n);
  }
  if (lane == 0) {
    // more records than places can only come from a bound that failed: the row then takes the unpruned path
    const bool over = fill > cap;
    mrg_len[m] = over ? 0 : (int32_t)(K + fill);
    if (over) fbmask[m] = 1;
  }
  for (int o = 16; o > 0; o >>= 1) surv += __shfl_xor_sync(0xffffffffu, surv, o);
  if (lane == 0 && surv) atomicAdd(survivors, (unsigned long long)surv);
}

// ||k|| of every key of one shared key sequence (e4m3 codes for FP8 keys),
// squares summed by fmaf in d order, square root rounded up: the bound's
// c ||k|| term, computed once instead of in every epilogue warp.
__global__ void key_norm_kernel(idx_problem p, float* knorm) {
  const int D = p.D;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < p.n_keys;
       k += (int64_t)gridDim.x * blockDim.x) {
    float ss = 0.0f;
    if (p.k_dtype == IDX_FP8_E4M3) {
      const uint8_t* row = (const uint8_t*)p.keys + k * D;
      for (int d = 0; d < D; d += 16) {
        const uint4 c = *reinterpret_cast<const uint4*>(row + d);
        const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
        for (int e = 0; e < 16; ++e) {
          const float x = e4m3_to_f((uint8_t)(w4[e >> 2] >> (8 * (e & 3))));
          ss = __fmaf_rn(x, x, ss);
        }
      }
    } else {
      const uint16_t* row = (const uint16_t*)p.keys + k * D;
      for (int d = 0; d < D; d += 8) {
        const uint4 c = *reinterpret_cast<const uint4*>(row + d);
        const uint32_t w4[4] = {c.x, c.y, c.z, c.w};
        for (int e = 0; e < 4; ++e) {
          const float lo = bf16_to_f((uint16_t)(w4[e] & 0xffffu)), hi = bf16_to_f((uint16_t)(w4[e] >> 16));
          ss = __fmaf_rn(lo, lo, ss);
          ss = __fmaf_rn(hi, hi, ss);
        }
      }
    }
    knorm[k] = __fsqrt_ru(ss);
  }
}

// ---------------------------------------------------------- shared stream --

constexpr int kGrpThreads = 1024;
constexpr int kGrpChunk = 64 * kGrpThreads;     // keys per pass (two bitmap words per thread)

// One block per group g (rows 4g..4g+3) over the rows' candidate bitmaps (row
// stride W words, the words below each row's visible length).  A row on the
// unpruned path (status != 0) takes no part; a row with more than cap
// candidates joins that path (status bit 2).  Then, in passes of kGrpChunk
// ids: a key kept by at least two of the remaining rows and below all of their
// visible lengths goes to the group list (glist, ascending), each row's other
// candidates to its own list (solo, ascending).  cand_cnt[m] = the row's
// candidates, solo_n[m] = its own-list length.
__global__ void __launch_bounds__(kGrpThreads) group_split_kernel(
    idx_problem p, int64_t cap, const uint32_t* bits, int64_t W, int32_t* status, int32_t* cand_cnt, int32_t* solo,
    int64_t solo_ld, int32_t* solo_n, int32_t* glist, int32_t* gcnt, int64_t capg, unsigned long long* st_group,
    unsigned long long* st_solo) {
  __shared__ int32_t s_warp[32][5];
  __shared__ int32_t s_tot[5], s_base[5];
  __shared__ int32_t s_len[4], s_nw[4], s_cnt[4];
  __shared__ int32_t s_common, s_maxlen;
  const int64_t g = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid < 4) {
    const int64_t m = 4 * g + tid;
    int len = 0, nw = 0;
    if (m < p.M && status[m] == 0) {
      int64_t off;
      row_extent(p, m, &off, &len);
      const int64_t w = ((int64_t)len + 31) / 32;
      nw = (int)(w < W ? w : W);
    }
    s_len[tid] = len;
    s_nw[tid] = nw;
    s_cnt[tid] = 0;
  }
  if (tid < 5) s_base[tid] = 0;
  __syncthreads();
  // each row's candidate count
  {
    int c[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      for (int w = tid; w < s_nw[i]; w += kGrpThreads) c[i] += __popc(bits[(4 * g + i) * W + w]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c[i] += __shfl_xor_sync(0xffffffffu, c[i], o);
      if (lane == 0 && c[i]) atomicAdd(&s_cnt[i], c[i]);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int common = 0x7fffffff, mx = 0;
    for (int i = 0; i < 4; ++i) {
      const int64_t m = 4 * g + i;
      if (m >= p.M) break;
      cand_cnt[m] = s_cnt[i];
      if (s_nw[i] == 0 && s_len[i] == 0) continue;   // not taking part (or nothing visible)
      if (s_cnt[i] > cap) {
        status[m] |= 2;
        s_nw[i] = 0;
        s_len[i] = 0;
        continue;
      }
      common = s_len[i] < common ? s_len[i] : common;
      mx = s_len[i] > mx ? s_len[i] : mx;
    }
    s_common = common == 0x7fffffff ? 0 : common;
    s_maxlen = mx;
  }
  __syncthreads();
  const int common = s_common, maxlen = s_maxlen;
  for (int c0 = 0; c0 < maxlen; c0 += kGrpChunk) {
    uint32_t sh[2], so[4][2];
    int cnt[5] = {0, 0, 0, 0, 0};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int w = c0 / 32 + 2 * tid + e;
      uint32_t b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] = w < s_nw[i] ? bits[(4 * g + i) * W + w] : 0u;
      const uint32_t two = (b[0] & b[1]) | (b[0] & b[2]) | (b[0] & b[3]) | (b[1] & b[2]) | (b[1] & b[3]) | (b[2] & b[3]);
      const int nv = common - 32 * w;          // keys of this word below the common length
      const uint32_t vis = nv >= 32 ? 0xffffffffu : (nv <= 0 ? 0u : ((1u << nv) - 1u));
      sh[e] = two & vis;
      cnt[0] += __popc(sh[e]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        so[i][e] = b[i] & ~sh[e];
        cnt[1 + i] += __popc(so[i][e]);
      }
    }
    // block exclusive scan of the five counts (warp scans, then a scan of the warp totals)
    int incl[5];
#pragma unroll
    for (int v = 0; v < 5; ++v) {
      int x = cnt[v];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      incl[v] = x;
      if (lane == 31) s_warp[wid][v] = x;
    }
    __syncthreads();
    if (wid == 0) {
#pragma unroll
      for (int v = 0; v < 5; ++v) {
        const int t = s_warp[lane][v];
        int x = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        s_warp[lane][v] = x - t;
        if (lane == 31) s_tot[v] = x;
      }
    }
    __syncthreads();
    int pos[5];
#pragma unroll
    for (int v = 0; v < 5; ++v) pos[v] = s_base[v] + s_warp[wid][v] + incl[v] - cnt[v];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int k0 = c0 + 32 * (2 * tid + e);
      for (uint32_t b = sh[e]; b; b &= b - 1) {
        if (pos[0] < capg) glist[g * capg + pos[0]] = k0 + __ffs(b) - 1;
        ++pos[0];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t m = 4 * g + i;
        for (uint32_t b = so[i][e]; b; b &= b - 1) solo[m * solo_ld + pos[1 + i]++] = k0 + __ffs(b) - 1;
      }
    }
    __syncthreads();
    if (tid == 0)
      for (int v = 0; v < 5; ++v) s_base[v] += s_tot[v];
    __syncthreads();
  }
  if (tid == 0) {
    const int ng = s_base[0] < capg ? s_base[0] : (int)capg;
    gcnt[g] = ng;
    unsigned long long ns = 0;
    for (int i = 0; i < 4; ++i) {
      const int64_t m = 4 * g + i;
      if (m >= p.M) break;
      solo_n[m] = s_base[1 + i];
      ns += (unsigned long long)s_base[1 + i];
    }
    if (st_group) atomicAdd(st_group, (unsigned long long)ng);
    if (st_solo) atomicAdd(st_solo, ns);
  }
}

__global__ void stats_kernel(idx_problem p, const int32_t* seed_cnt, int shared_seeds, const int32_t* cand_cnt,
                             const int32_t* status, const int32_t* active, dosa_stats* st, int32_t* row_status) {
  unsigned long long pairs = 0, seeds = 0, cands = 0, fb = 0, skipped = 0;
  for (int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; m < p.M; m += (int64_t)gridDim.x * blockDim.x) {
    int64_t off;
    int len;
    row_extent(p, m, &off, &len);
    pairs += (unsigned long long)len;
    if (active[m]) {
      seeds += (unsigned long long)seed_cnt[shared_seeds ? 0 : m];
      cands += (unsigned long long)cand_cnt[m];
    }
    const int s = status[m];
    fb += s != 0 ? 1ull : 0ull;
    skipped += (s & 4) ? 1ull : 0ull;
    if (row_status) row_status[m] = (s & 1) ? 1 : ((s & 4) ? 3 : ((s & 2) ? 2 : 0));
  }
  if (!st) return;
  for (int o = 16; o > 0; o >>= 1) {
    pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
    seeds += __shfl_xor_sync(0xffffffffu, seeds, o);
    cands += __shfl_xor_sync(0xffffffffu, cands, o);
    fb += __shfl_xor_sync(0xffffffffu, fb, o);
    skipped += __shfl_xor_sync(0xffffffffu, skipped, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&st->pairs, pairs);
    atomicAdd(&st->seeds, seeds);
    atomicAdd(&st->candidates, cands);
    atomicAdd(&st->fallback_rows, fb);
    atomicAdd(&st->skipped_rows, skipped);
  }
}

// ------------------------------------------------------------- workspace --

struct DosaWs {
  uint32_t* bits;
  int32_t* list;
  int32_t* seed_cnt;
  int32_t* seed_len;       // [M]: per-row seed count (the shared count broadcast)
  int32_t* common;         // [1]
  uint16_t* rep_q;
  float* rep_w;
  int32_t* rep_len;
  float* rep_sc;
  int32_t* rep_ids;
  uint32_t* rep_count;
  uint32_t* rep_best;      // [ldmax] best representative score per key (ordered key)
  void* seed_keys;
  float* seed_scale;
  float* seed_sc;
  int32_t* stop_ids;
  float* stop_sc;
  float* tau;
  int32_t* status;
  int32_t* active;
  uint16_t* qprep;
  float* wfold;
  float* coef;
  int32_t* plan_head;      // [M, H] the planner's record (see PlanArgs)
  float* plan_beta;        // [M, H]
  float* plan_dn;          // [M, H]
  int32_t* cand;
  int32_t* cand_cnt;
  int32_t* cand_n;
  float* cand_sc;
  float* mrg_sc;
  int32_t* mrg_id;
  int32_t* mrg_len;
  int32_t* fbmask;
  unsigned long long* surv;
  float* fb_scores;
  uint32_t* candbits;      // [M, cbW] candidate bitmaps of the bound scan
  float* knorm;            // shared keys: [n_keys] ||k||
  int32_t* glist;          // shared stream: [G, 2 cap] group lists
  int32_t* gcnt;           // [G]
  float* gsc;              // [M, 2 cap] scores of the group lists, by position
  int32_t* solo_n;         // [M] own-list lengths
  char* tk_ws;
  // (surv is the survivor counter used when the caller passes no stats)
  size_t used;
};

struct DosaShape {
  bool shared_keys, shared_seeds;
  bool group;         // shared candidate stream (groups of four rows)
  int64_t G;          // groups
  int64_t W;          // bitmap words per row
  int64_t cbW;        // candidate bitmap words per row (whole 128-key tiles)
  int64_t NS;         // seed list capacity per row
  int64_t cap;        // candidate capacity per row
  int64_t ldmax;      // max_key_len (>= 1)
};

static DosaShape dosa_shape(const idx_problem& p, int K, const dosa_params& dp, int seed_ld) {
  DosaShape s;
  s.shared_keys = p.key_off == nullptr;
  s.shared_seeds = s.shared_keys && seed_ld == 0;
  s.ldmax = p.max_key_len > 0 ? p.max_key_len : 1;
  s.W = (s.ldmax + 31) / 32;
  s.cbW = (s.ldmax + 127) / 128 * 4;
  int64_t ns = seed_ld > 0 ? seed_ld : dp.n_seed;
  if (ns < K) ns = K;
  s.NS = ns < s.ldmax ? ns : s.ldmax;
  if (s.NS < 1) s.NS = 1;
  s.cap = dp.candidate_capacity > 0 ? dp.candidate_capacity : 1;
  s.group = dp.group_stream != 0 && p.M >= 2 && group_stream_supported(p);
  s.G = s.group ? (p.M + 3) / 4 : 0;
  return s;
}

static DosaWs carve(void* base, const idx_problem& p, int K, const dosa_params& dp, int seed_ld) {
  const DosaShape s = dosa_shape(p, K, dp, seed_ld);
  const int64_t M = p.M;
  const int64_t seed_rows = s.shared_seeds ? 1 : M;
  WsCarver c(base);
  DosaWs w;
  w.bits = c.take<uint32_t>(seed_rows * s.W);
  w.list = c.take<int32_t>(seed_rows * s.NS);
  w.seed_cnt = c.take<int32_t>(seed_rows);
  w.seed_len = c.take<int32_t>(M);
  w.common = c.take<int32_t>(1);
  w.rep_q = c.take<uint16_t>((size_t)4 * p.H * p.D);
  w.rep_w = c.take<float>((size_t)4 * p.H);
  w.rep_len = c.take<int32_t>(4);
  w.rep_sc = c.take<float>((size_t)4 * s.ldmax);
  w.rep_ids = c.take<int32_t>((size_t)4 * K);
  w.rep_count = c.take<uint32_t>(s.ldmax);
  w.rep_best = c.take<uint32_t>(s.ldmax);
  const int row_bytes = p.k_dtype == IDX_FP8_E4M3 ? 128 : 256;
  w.seed_keys = c.take<char>(s.shared_seeds ? (size_t)s.NS * row_bytes : 16);
  w.seed_scale = c.take<float>(s.shared_seeds ? (size_t)s.NS : 1);
  w.seed_sc = c.take<float>((size_t)M * s.NS);
  w.stop_ids = c.take<int32_t>((size_t)M * K);
  w.stop_sc = c.take<float>((size_t)M * K);
  w.tau = c.take<float>(M);
  w.status = c.take<int32_t>(M);
  w.active = c.take<int32_t>(M);
  // [M, 32, D], or the bound's group layout: 144 rows per 8 queries
  const size_t qp_rows = (size_t)M * kVec > (size_t)((M + 7) / 8) * 144 ? (size_t)M * kVec : (size_t)((M + 7) / 8) * 144;
  w.qprep = c.take<uint16_t>(qp_rows * p.D);
  w.wfold = c.take<float>((size_t)M * kVec);
  w.coef = c.take<float>(M);
  w.plan_head = c.take<int32_t>((size_t)M * p.H);
  w.plan_beta = c.take<float>((size_t)M * p.H);
  w.plan_dn = c.take<float>((size_t)M * p.H);
  w.cand = c.take<int32_t>((size_t)M * s.cap);
  w.cand_cnt = c.take<int32_t>(M);
  w.cand_n = c.take<int32_t>(M);
  w.cand_sc = c.take<float>((size_t)M * s.cap);
  w.mrg_sc = c.take<float>((size_t)M * (K + s.cap));
  w.mrg_id = c.take<int32_t>((size_t)M * (K + s.cap));
  w.mrg_len = c.take<int32_t>(M);
  w.fbmask = c.take<int32_t>(M);
  w.surv = c.take<unsigned long long>(1);
  w.fb_scores = c.take<float>((size_t)M * s.ldmax);
  w.candbits = c.take<uint32_t>((size_t)M * s.cbW);
  w.knorm = c.take<float>(s.shared_keys ? (size_t)p.n_keys : 1);
  w.glist = c.take<int32_t>(s.group ? (size_t)s.G * 2 * s.cap : 1);
  w.gcnt = c.take<int32_t>(s.group ? (size_t)s.G : 1);
  w.gsc = c.take<float>(s.group ? (size_t)M * 2 * s.cap : 1);
  w.solo_n = c.take<int32_t>(s.group ? (size_t)M : 1);
  size_t tk = topk_dense_ws(M, (int)s.ldmax, K);
  size_t tk2 = topk_dense_ws(M, (int)(K + s.cap), K);
  size_t tk3 = topk_dense_ws(M, (int)s.NS, K);
  tk = tk > tk2 ? tk : tk2;
  tk = tk > tk3 ? tk : tk3;
  w.tk_ws = c.take<char>(tk > 0 ? tk : 16);
  w.used = c.used + 256;
  return w;
}

bool dosa_supported(const idx_problem& p, const dosa_params& dp) {
  return score_uses_tensor_cores(p) && dp.retained_heads < 32 && dp.retained_heads < p.H && dp.n_sample <= 128;
}

size_t dosa_ws(const idx_problem& p, int K, const dosa_params& dp, int seed_ld) {
  if (!dosa_supported(p, dp)) return idx_topk_workspace_size(&p, K);
  return carve(nullptr, p, K, dp, seed_ld).used;
}

bool dosa_layout(const idx_problem& p, int K, const dosa_params& dp, int seed_ld, dosa_ws_layout* out) {
  if (!dosa_supported(p, dp) || p.M <= 0) return false;
  const DosaShape s = dosa_shape(p, K, dp, seed_ld);
  // carved against a nominal 256-aligned base, offsets relative to it
  const uintptr_t base = (uintptr_t)1 << 20;
  const DosaWs w = carve(reinterpret_cast<void*>(base), p, K, dp, seed_ld);
  auto off = [&](const void* x) { return (int64_t)(reinterpret_cast<uintptr_t>(x) - base); };
  out->seed_list = off(w.list);
  out->seed_count = off(w.seed_cnt);
  out->rep_count = off(w.rep_count);
  out->rep_scores = off(w.rep_sc);
  out->tau = off(w.tau);
  out->status = off(w.status);
  out->plan_head = off(w.plan_head);
  out->plan_beta = off(w.plan_beta);
  out->plan_dnorm = off(w.plan_dn);
  out->wfold = off(w.wfold);
  out->coef = off(w.coef);
  out->qprep = off(w.qprep);
  out->seed_ld = s.NS;
  out->rep_ld = s.ldmax;
  out->seed_rows = s.shared_seeds ? 1 : p.M;
  out->group_layout = bound_group_layout(p, dp.retained_heads) ? 1 : 0;
  return true;
}

static int grid_for(int64_t n, int threads) {
  int64_t g = (n + threads - 1) / threads;
  return (int)(g < 1 ? 1 : (g > 4096 ? 4096 : g));
}

#define DOSA_CHECK(x)                   \
  do {                                  \
    cudaError_t e_ = (x);               \
    if (e_ != cudaSuccess) return e_;   \
  } while (0)

cudaError_t launch_dosa(const idx_problem& p, int K, const dosa_params& dp, const int32_t* seed_ids, int seed_ld,
                        int32_t* out_ids, float* out_scores, int32_t* row_status, dosa_stats* stats, void* ws,
                        size_t ws_bytes, cudaStream_t st) {
  const int64_t M = p.M;
  if (!dosa_supported(p, dp)) {
    // exact path (the output contract is the unpruned top-K); every row counts as a fallback row
    const int64_t ld = p.max_key_len > 0 ? p.max_key_len : 1;
    WsCarver c(ws);
    float* scores = c.take<float>((size_t)M * ld);
    char* lists = c.take<char>(topk_dense_ws(M, p.max_key_len, K));
    DOSA_CHECK(launch_score(p, scores, ld, st));
    DOSA_CHECK(launch_topk_dense(scores, ld, nullptr, &p, M, p.max_key_len, K, out_ids, out_scores, lists, st));
    if (row_status) DOSA_CHECK(fill_i32(row_status, M, 1, st));
    return cudaSuccess;
  }
  const DosaShape s = dosa_shape(p, K, dp, seed_ld);
  DosaWs w = carve(ws, p, K, dp, seed_ld);
  if (w.used > ws_bytes) return cudaErrorInvalidValue;
  const int64_t seed_rows = s.shared_seeds ? 1 : M;

  // ---- seeds
  DOSA_CHECK(fill_i32(w.bits, seed_rows * s.W, 0, st));
  if (seed_ids) {
    caller_seeds_kernel<<<(unsigned)M, 256, 0, st>>>(p, seed_ids, seed_ld, w.bits, s.W);
  } else if (!s.shared_seeds) {
    strided_seeds_kernel<<<(unsigned)M, 256, 0, st>>>(p, dp.n_seed, w.bits, s.W);
  } else {
    // cold rule over the common visible prefix
    min_len_kernel<<<1, 1024, 0, st>>>(p, w.common);
    Reps r{};
    for (int i = 0; i < 4; ++i) {
      const int64_t m = M > 1 ? ((int64_t)i * (M - 1)) / 3 : 0;
      bool dup = false;
      for (int j = 0; j < r.n; ++j) dup |= r.m[j] == m;
      if (!dup) r.m[r.n++] = m;
    }
    gather_reps_kernel<<<(unsigned)r.n, 256, 0, st>>>(p, r, w.common, w.rep_q, w.rep_w, w.rep_len);
    idx_problem sub = p;
    sub.q = w.rep_q;
    sub.w = w.rep_w;
    sub.M = r.n;
    sub.key_len = w.rep_len;
    DOSA_CHECK(launch_score(sub, w.rep_sc, s.ldmax, st));
    DOSA_CHECK(launch_topk_dense(w.rep_sc, s.ldmax, w.rep_len, nullptr, r.n, (int)s.ldmax, K, w.rep_ids, nullptr,
                                 w.tk_ws, st));
    DOSA_CHECK(fill_i32(w.rep_count, s.ldmax, 0, st));
    rep_count_kernel<<<grid_for((int64_t)r.n * K, 256), 256, 0, st>>>(w.rep_ids, r.n, K, w.rep_count);
    rep_best_kernel<<<grid_for(s.ldmax, 256), 256, 0, st>>>(w.rep_sc, s.ldmax, r.n, w.common, w.rep_best);
    cold_select_kernel<<<1, kColdThreads, 0, st>>>(w.rep_count, w.rep_best, w.common, dp.n_seed, w.bits);
  }
  DOSA_CHECK(cudaGetLastError());
  bits_to_list_kernel<<<(unsigned)seed_rows, kListThreads, 0, st>>>(w.bits, s.W, w.list, s.NS, w.seed_cnt);
  DOSA_CHECK(cudaGetLastError());

  // ---- seed scores, seed top-K, tau
  if (s.shared_seeds) {
    gather_keys_kernel<<<grid_for(s.NS * 16, 256), 256, 0, st>>>(p, w.list, w.seed_cnt, w.seed_keys,
                                                                  p.key_scale ? w.seed_scale : nullptr);
    broadcast_i32_kernel<<<grid_for(M, 256), 256, 0, st>>>(w.seed_cnt, w.seed_len, M);
    idx_problem sp = p;
    sp.keys = w.seed_keys;
    sp.key_scale = p.key_scale ? w.seed_scale : nullptr;
    sp.n_keys = s.NS;
    sp.key_off = nullptr;
    sp.key_len = w.seed_len;
    sp.max_key_len = (int32_t)s.NS;
    DOSA_CHECK(launch_score(sp, w.seed_sc, s.NS, st));
  } else {
    DOSA_CHECK(cudaMemcpyAsync(w.seed_len, w.seed_cnt, M * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    DOSA_CHECK(launch_score_gather(p, w.list, w.seed_cnt, s.NS, w.seed_sc, s.NS, nullptr, st));
  }
  DOSA_CHECK(launch_topk_dense(w.seed_sc, s.NS, w.seed_len, nullptr, M, (int)s.NS, K, w.stop_ids, w.stop_sc,
                               w.tk_ws, st, w.list, s.shared_seeds ? 0 : s.NS));
  seed_status_kernel<<<grid_for(M, 256), 256, 0, st>>>(M, K, w.seed_cnt, s.shared_seeds ? 1 : 0, w.stop_sc, w.tau,
                                                       w.status, w.active);
  DOSA_CHECK(cudaGetLastError());

  // ---- planner
  PlanArgs pa;
  pa.p = p;
  pa.R = dp.retained_heads;
  pa.n_sample = dp.n_sample;
  pa.act_min = dp.act_freq_min;
  pa.gamma = dp.margin_gamma;
  pa.seed_list = w.list;
  pa.list_ld = s.NS;
  pa.seed_cnt = w.seed_cnt;
  pa.shared_seeds = s.shared_seeds ? 1 : 0;
  pa.active = w.active;
  pa.status = w.status;
  pa.tau = w.tau;
  pa.cap = s.cap;
  pa.qprep = w.qprep;
  pa.glayout = bound_group_layout(p, dp.retained_heads) ? 1 : 0;
  pa.wfold = w.wfold;
  pa.coef = w.coef;
  pa.plan_head = w.plan_head;
  pa.plan_beta = w.plan_beta;
  pa.plan_dn = w.plan_dn;
  const size_t psmem = plan_smem_bytes(p.H, dp.n_sample);
  DOSA_CHECK(cudaFuncSetAttribute(dosa_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem));
  dosa_plan_kernel<<<(unsigned)M, kPlanThreads, psmem, st>>>(pa);
  DOSA_CHECK(cudaGetLastError());

  // ---- bound scan: candidate bitmaps
  idx_problem prep = p;
  prep.q = w.qprep;
  prep.H = kVec;
  if (s.shared_keys) {
    key_norm_kernel<<<grid_for(p.n_keys, 256), 256, 0, st>>>(p, w.knorm);
    DOSA_CHECK(cudaGetLastError());
  }
  DOSA_CHECK(launch_bound(prep, w.wfold, w.coef, w.tau, s.shared_keys ? w.knorm : nullptr, w.bits,
                          s.shared_seeds ? 0 : s.W, w.candbits, s.cbW, dp.retained_heads, w.active, st));

  // ---- exact rescoring of the candidates, merge with the seed top-K
  GroupRecs gr{};
  if (s.group) {
    // shared stream: own lists straight into the merge rows (at K), group lists scored once per group
    const int64_t mld = K + s.cap, capg = 2 * s.cap;
    group_split_kernel<<<(unsigned)s.G, kGrpThreads, 0, st>>>(
        p, s.cap, w.candbits, s.cbW, w.status, w.cand_cnt, w.mrg_id + K, mld, w.solo_n, w.glist, w.gcnt, capg,
        stats ? &stats->group_keys : nullptr, stats ? &stats->solo_keys : nullptr);
    DOSA_CHECK(cudaGetLastError());
    DOSA_CHECK(launch_score_gather(p, w.mrg_id + K, w.solo_n, mld, w.cand_sc, s.cap, w.active, st));
    DOSA_CHECK(launch_score_group(p, w.glist, w.gcnt, capg, w.gsc, capg, st));
    gr = GroupRecs{w.glist, w.gcnt, w.gsc, capg, w.bits, s.shared_seeds ? 0 : s.W, p};
    merge_rows_kernel<<<(unsigned)((M + kMergeRows - 1) / kMergeRows), kMergeThreads, 0, st>>>(
        M, K, s.cap, w.stop_ids, w.stop_sc, nullptr, w.solo_n,
                                                              w.cand_sc, w.tau, w.status, gr, w.mrg_sc, w.mrg_id,
                                                              w.mrg_len, w.fbmask,
                                                              stats ? &stats->survivors : w.surv);
  } else {
    cand_compact_kernel<<<(unsigned)M, kListThreads, 0, st>>>(p, w.candbits, s.cbW, w.status, w.cand, s.cap,
                                                               w.cand_cnt, w.cand_n);
    DOSA_CHECK(cudaGetLastError());
    DOSA_CHECK(launch_score_gather(p, w.cand, w.cand_n, s.cap, w.cand_sc, s.cap, w.active, st));
    merge_rows_kernel<<<(unsigned)((M + kMergeRows - 1) / kMergeRows), kMergeThreads, 0, st>>>(
        M, K, s.cap, w.stop_ids, w.stop_sc, w.cand, w.cand_n,
                                                              w.cand_sc, w.tau, w.status, gr, w.mrg_sc, w.mrg_id,
                                                              w.mrg_len, w.fbmask,
                                                              stats ? &stats->survivors : w.surv);
  }
  DOSA_CHECK(cudaGetLastError());
  DOSA_CHECK(launch_topk_dense(w.mrg_sc, K + s.cap, w.mrg_len, nullptr, M, (int)(K + s.cap), K, out_ids, out_scores,
                               w.tk_ws, st, w.mrg_id, K + s.cap));

  // ---- rows that could not be pruned: the unpruned path, only for them
  DOSA_CHECK(launch_score(p, w.fb_scores, s.ldmax, st, w.fbmask));
  DOSA_CHECK(launch_topk_dense(w.fb_scores, s.ldmax, nullptr, &p, M, (int)s.ldmax, K, out_ids, out_scores, w.tk_ws,
                               st, nullptr, 0, w.fbmask));

  stats_kernel<<<grid_for(M, 256), 256, 0, st>>>(p, w.seed_cnt, s.shared_seeds ? 1 : 0, w.cand_cnt, w.status,
                                                 w.active, stats, row_status);
  return cudaGetLastError();
}

}  // namespace idx
