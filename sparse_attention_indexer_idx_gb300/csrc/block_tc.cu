// MiniMax-M3 block-sparse selection, tensor-core route for 128-token blocks and
// D = 128 ("ferrox_core/block_sparse.rs": block_sparse_select, select_for_head,
// dot).
//
// The page scores a block by the max over its positions of a dot product summed
// in sequence in fp32, and the selected indices depend on those exact values,
// so a tensor-core pass cannot decide the selection by itself.  It can decide
// almost all of it: with A_b the block max computed by the tensor cores and a
// certified bound e_b >= |A_b - E_b| (E_b the page's exact block score), a block
// whose interval [A_b - e_b, A_b + e_b] lies clear of the cut is settled either
// way, and only the few blocks per (query, head) pair whose intervals straddle
// it are scored in the page's order.  The output is the page's selection bit
// for bit.
//
//  1. bt_prep_kernel: queries ordered by their number of visible blocks (a
//     counting sort; a tile of 32 queries then scans about as many blocks as
//     each of its queries needs); every query row and every key block written
//     as fp16 under a power-of-two scale (sigma per row, s_b per block, so
//     that the largest magnitude sits in [2^14, 2^15): 11 significant bits,
//     as many as tf32, at half the bytes and twice the tensor rate); the
//     norm factors of the bound.
//  2. bt_max_kernel: A_b over every visible block of every pair, on
//     tcgen05.mma kind::f16.  A CTA holds 256 (query, head) rows (two M = 128
//     tiles, fetched by TMA gather4 in the sorted order) and streams key
//     blocks (128 keys = N, two 64-element K chunks, one TMA box each) through
//     a ten-stage ring; each key chunk feeds eight MMAs (K = 16, both tiles).
//     A_b = sigma s_b max(acc) (exact power-of-two scaling).  The
//     accumulators (two stages of 2 x 128 TMEM columns) are reduced by eight
//     epilogue warps: a thread owns one (query, head) row, so the block max is
//     a max over its own 128 columns (positions past the query's position or
//     past L masked).  Units are (row tile pair, key block), split into one
//     contiguous range per persistent CTA.
//  3. bt_classify_kernel (one warp per pair): the n_need-th largest lower bound
//     T; candidates are the blocks with upper bound >= T (every other block has
//     n_need blocks certainly above it); a candidate is certainly in when fewer
//     than n_need other candidates could reach its lower bound.  Pairs whose
//     undecided blocks are exactly the places left are done here; the others
//     list their undecided blocks per key block.
//  4. bt_exact_kernel (one CTA per key block): the listed (pair, block) scores
//     in the page's order on the fp32 pipes (packed f32x2 multiply and add,
//     each half rounded as the scalar instructions round).
//  5. bt_resolve_kernel (one warp per open pair): the remaining places from the
//     exact scores by (score desc, block asc); a pair with too many undecided
//     blocks has every non-forced block rescored and takes its whole top list
//     here.
//
// The bound.  The tensor core multiplies exactly q~ = sigma fp16(q / sigma)
// and k~ = s_b fp16(k / s_b) (values this code rounded, so dq = q - q~ and
// dk = k - k~ are known exactly); products of fp16 values are exact in fp32.
// With E_p = q.k_p in the page's order and A_p the tensor-core value,
//   |A_p - E_p| <= |q~.dk| + |dq.k| + (accumulation and page-order sum)
//              <= ||q~|| ||dk_p|| + ||dq|| ||k_p|| + 2^-12 ||q|| ||k_p||,
// the last term a wide allowance (16x) over fp32 accumulation of 128 products
// in 8 MMAs of K = 16 plus the page's sequential sum, plus 2^-118 for products
// below the normal range.  Per block the key factors are their maxima over
// its positions; every factor is rounded up.  The same bound holds for the
// block maxima.  bt_exact_kernel measures |A_b - E_b| / e_b on every block it
// rescores and reports the largest value through block_select_stats.
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "block_select.cuh"

namespace idx {

bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows);

constexpr float kBtGamma = 0.000244140625f;        // 2^-12: accumulation and page-order sum allowance
constexpr float kBtAbs = 3.00926553e-36f;           // 2^-118: products below the normal range
constexpr int kBtRowsT = 256;        // (query, head) rows per CTA tile: two MMA tiles of 128
constexpr int kBtKStages = 10;       // key-chunk ring
constexpr int kBtChunkBytes = 128 * 128;   // 128 rows x 64 fp16 (one 128-byte swizzle span)
constexpr int kBtATile = 2 * kBtChunkBytes;   // 128 rows x 128 fp16
constexpr int kBtNE = 8;             // epilogue warps
// warp 0 TMA producer, warp 1 MMA issue (one thread, every unit, the two
// accumulator stages in turn), warps 2 .. 2 + kBtNE - 1 epilogue
constexpr int kBtThreads = 32 * (2 + kBtNE);
constexpr int kBtTmemCols = 512;     // two stages x two tiles x 128 keys
constexpr int kBtCapC = 256;         // candidates per pair held by the classifier
constexpr int kBtCapU = 64;          // undecided blocks per pair resolved from a list
constexpr int kBtMaxTop = 512;       // top_blocks handled by this route
constexpr int kBtSortBins = 8192;

// Per-pair state written by the classifier.
enum BtStatus { kBtDone = 0, kBtList = 1, kBtFallback = 2 };

struct BtWs {
  int32_t* order;      // [Q] query rank -> query
  int32_t* nbT;        // [nT] blocks scanned by row tile pair T
  __half* q16;         // [Q*n_kv, 128] q / sigma as fp16 (original pair order)
  float* qsig;         // [Q*n_kv] sigma: power-of-two row scale
  float2* qab;         // [Q*n_kv] bound factors (||dq|| + 2^-12 (||q~|| + ||dq||), ||q~||), rounded up
  __half* k16;         // [L, 128] k / s_b as fp16
  float* ksc;          // [nbm] s_b: power-of-two block scale
  float2* kb;          // [nbm] (max ||k_p||, max ||k_p - k~_p||) over the block, rounded up
  float* amax;         // [slots, nbm] A_b (float), overwritten by the exact ordered key when rescored
  int32_t* icnt;       // [nbm] listed pairs per block
  int32_t* ilist;      // [nbm, slots] slots listed per block
  int32_t* ulist;      // [slots, kBtCapU] undecided blocks (ascending)
  int4* sstat;         // [slots] {status, k_in, n_u, m_need}
};

struct BtProblem {
  const float* q;
  const float* k;
  const int32_t* qpos;
  int64_t Q;
  int n_kv;
  int64_t L;
  int64_t slots;   // Q * n_kv
  int64_t nbm;     // ceil(L / 128)
  int64_t nT;      // ceil(slots / 256)
  block_sparse_config c;
};

__host__ __device__ inline int64_t bt_round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

static BtWs bt_carve(void* base, const BtProblem& P) {
  WsCarver w(base);
  BtWs s;
  s.order = w.take<int32_t>((size_t)P.Q);
  s.nbT = w.take<int32_t>((size_t)P.nT);
  s.q16 = w.take<__half>((size_t)P.slots * 128);
  s.qsig = w.take<float>((size_t)P.slots);
  s.qab = w.take<float2>((size_t)P.slots);
  s.k16 = w.take<__half>((size_t)P.L * 128);
  s.ksc = w.take<float>((size_t)P.nbm);
  s.kb = w.take<float2>((size_t)P.nbm);
  s.amax = w.take<float>((size_t)(P.slots * P.nbm));
  s.icnt = w.take<int32_t>((size_t)P.nbm);
  s.ilist = w.take<int32_t>((size_t)(P.nbm * P.slots));
  s.ulist = w.take<int32_t>((size_t)(P.slots * kBtCapU));
  s.sstat = w.take<int4>((size_t)P.slots);
  return s;
}

static size_t bt_ws_bytes(const BtProblem& P) {
  WsCarver w(nullptr);
  w.take<int32_t>((size_t)P.Q);
  w.take<int32_t>((size_t)P.nT);
  w.take<__half>((size_t)P.slots * 128);
  w.take<float>((size_t)P.slots);
  w.take<float2>((size_t)P.slots);
  w.take<__half>((size_t)P.L * 128);
  w.take<float>((size_t)P.nbm);
  w.take<float2>((size_t)P.nbm);
  w.take<float>((size_t)(P.slots * P.nbm));
  w.take<int32_t>((size_t)P.nbm);
  w.take<int32_t>((size_t)(P.nbm * P.slots));
  w.take<int32_t>((size_t)(P.slots * kBtCapU));
  w.take<int4>((size_t)P.slots);
  return w.used + 256;
}

__device__ __forceinline__ int64_t bt_nblocks(int64_t pos, const BtProblem& P) {
  return block_geom(pos, P.L, P.c).n_blocks;
}

// Query of a slot (sorted rank * n_kv + head); slots fit 32 bits on this route.
__device__ __forceinline__ int64_t bt_slot_query(const BtProblem& P, const BtWs& W, int64_t slot) {
  return (int64_t)W.order[(uint32_t)slot / (uint32_t)P.n_kv];
}
// Row of index_q (pair index) of a slot.
__device__ __forceinline__ int64_t bt_slot_pair(const BtProblem& P, const BtWs& W, int64_t slot) {
  const uint32_t sl = (uint32_t)slot, nk = (uint32_t)P.n_kv, rank = sl / nk;
  return (int64_t)W.order[rank] * P.n_kv + (int64_t)(sl - rank * nk);
}

// sqrt of a sum of 128 squares accumulated in fp32 (relative error < 2^-16),
// rounded up with 2^-14 on top: an upper bound of the exact norm.
__device__ __forceinline__ float bt_norm_up(float ss) { return __fmul_ru(__fsqrt_ru(ss), 1.00006103515625f); }

// Sum / max over the 8 lanes of a row group (lanes 8g..8g+7).
__device__ __forceinline__ float bt_sum8(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  return v;
}
__device__ __forceinline__ float bt_max8(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  return v;
}

// Power-of-two scale s of a row or block with largest magnitude amax: amax / s
// in [2^14, 2^15), so x / s is an fp16 value with 11 significant bits for every
// element within a factor 2^14 of amax and never overflows; s >= 2^-100 keeps
// every s * fp16 value an exact fp32 number.
__device__ __forceinline__ float bt_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  int ex;
  frexpf(amax, &ex);   // amax = f 2^ex, f in [0.5, 1)
  return ldexpf(1.0f, ex - 15 > -100 ? ex - 15 : -100);
}

// 16 floats -> 16 fp16 values of x / s (round to nearest even), stored to dst
// (32-byte aligned) when `store`;
// accumulates sum x~^2 and sum (x - x~)^2 with x~ = s * fp16(x / s) (both exact
// in fp32: a power-of-two scaling and a difference of neighbours).
__device__ __forceinline__ void bt_to_f16(const float4 (&v)[4], float s, float inv, __half* dst, bool store,
                                          float& st, float& sd) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float x[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const __half2 h = __floats2half2_rn(x[j] * inv, x[j + 1] * inv);
      const float2 back = __half22float2(h);
      const float t0 = back.x * s, t1 = back.y * s;
      const float d0 = x[j] - t0, d1 = x[j + 1] - t1;
      st = __fmaf_rn(t0, t0, st);
      st = __fmaf_rn(t1, t1, st);
      sd = __fmaf_rn(d0, d0, sd);
      sd = __fmaf_rn(d1, d1, sd);
      w[2 * i + j / 2] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
  if (store) {
    uint4* o = reinterpret_cast<uint4*>(dst);
    o[0] = make_uint4(w[0], w[1], w[2], w[3]);
    o[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// One key block (rows [128 t, min(128 t + 128, L))) per CTA of 8 warps: its
// scale s_b, the fp16 rows of k / s_b, and (max ||k_p||, max ||k_p - k~_p||).
// Warp w holds rows 16w .. 16w+15 in registers (lanes 8g..8g+7: row 16w + g +
// 4j, 16 floats each), so the block is read once, every load in flight.
__device__ __forceinline__ void bt_key_block(const float* k, __half* k16, int64_t t, int64_t L, float2* kb,
                                             float* ksc, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t r_end = (t + 1) * 128 < L ? (t + 1) * 128 : L;
  float4 v[4][4];
  float am = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t row = t * 128 + 16 * w + (lane >> 3) + 4 * j;
    const float4* p = reinterpret_cast<const float4*>(k + row * 128) + (lane & 7) * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[j][i] = row < r_end ? __ldg(p + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      am = fmaxf(am, fmaxf(fmaxf(fabsf(v[j][i].x), fabsf(v[j][i].y)), fmaxf(fabsf(v[j][i].z), fabsf(v[j][i].w))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  if (lane == 0) red[w] = am;
  __syncthreads();
  am = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) am = fmaxf(am, red[i]);
  const float s = bt_scale(am), inv = 1.0f / s;   // exact: a power of two
  float mk = 0.0f, md = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t row = t * 128 + 16 * w + (lane >> 3) + 4 * j;
    float st = 0.0f, sd = 0.0f;
    bt_to_f16(v[j], s, inv, k16 + row * 128 + (lane & 7) * 16, row < r_end, st, sd);
    // ||k|| <= ||k~|| + ||k - k~||
    const float nd = bt_norm_up(bt_sum8(sd));
    mk = fmaxf(mk, __fadd_ru(bt_norm_up(bt_sum8(st)), nd));
    md = fmaxf(md, nd);
  }
  mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, 8));
  mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, 16));
  md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, 8));
  md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, 16));
  if (lane == 0) {
    red[8 + w] = mk;
    red[16 + w] = md;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) {
      mk = fmaxf(mk, red[8 + i]);
      md = fmaxf(md, red[16 + i]);
    }
    kb[t] = make_float2(fmaxf(mk, red[8]), fmaxf(md, red[16]));
    ksc[t] = s;
  }
}

// Four query rows r0..r0+3: scale sigma per row, fp16 rows of q / sigma, and
// the bound factors (||dq|| + 2^-12 (||q~|| + ||dq||), ||q~||), dq = q - q~.
__device__ __forceinline__ void bt_query_rows(const float* q, __half* q16, float2* qab, float* qsig, int64_t r0,
                                              int64_t rows) {
  const int lane = threadIdx.x & 31;
  const int64_t r = r0 + (lane >> 3);
  float4 v[4];
  const float4* p = reinterpret_cast<const float4*>(q + (r < rows ? r : 0) * 128) + (lane & 7) * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = r < rows ? __ldg(p + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  float am = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) am = fmaxf(am, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
  const float s = bt_scale(bt_max8(am)), inv = 1.0f / s;
  float st = 0.0f, sd = 0.0f;
  bt_to_f16(v, s, inv, q16 + r * 128 + (lane & 7) * 16, r < rows, st, sd);
  const float nt = bt_norm_up(bt_sum8(st)), nd = bt_norm_up(bt_sum8(sd));
  if ((lane & 7) == 0 && r < rows) {
    qab[r] = make_float2(__fmaf_ru(kBtGamma, __fadd_ru(nt, nd), nd), nt);
    qsig[r] = s;
  }
}

// Certified bound of |A_b - E_b| for a pair and a block.
__device__ __forceinline__ float bt_bound(float2 qab, float2 kb) {
  return __fadd_ru(__fmaf_ru(qab.x, kb.x, __fmul_ru(qab.y, kb.y)), kBtAbs);
}

constexpr int kBtPrepThreads = 256;

// CTA 0: counting sort of the queries by visible block count (rank -> query),
// the block count of every row tile pair, and the per-block list counters set
// to zero.  CTAs 1 .. nbm: one key block each.  The rest: 32 (query, head)
// rows each (four per warp).
__global__ void __launch_bounds__(kBtPrepThreads) bt_prep_kernel(BtProblem P, BtWs W) {
  if (blockIdx.x == 0) {
    __shared__ int32_t hist[kBtSortBins];
    __shared__ int32_t part[kBtPrepThreads];
    int shift = 0;
    while ((P.nbm >> shift) + 1 > kBtSortBins) ++shift;
    for (int i = threadIdx.x; i < kBtSortBins; i += kBtPrepThreads) hist[i] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < P.Q; i += kBtPrepThreads)
      atomicAdd(&hist[bt_nblocks(P.qpos[i], P) >> shift], 1);
    __syncthreads();
    // exclusive scan: 32 bins per thread, then the 256 partial sums
    constexpr int PER = kBtSortBins / kBtPrepThreads;
    int run = 0;
    for (int j = 0; j < PER; ++j) {
      const int v = hist[threadIdx.x * PER + j];
      hist[threadIdx.x * PER + j] = run;
      run += v;
    }
    part[threadIdx.x] = run;
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0;
      for (int t = 0; t < kBtPrepThreads; ++t) {
        const int v = part[t];
        part[t] = acc;
        acc += v;
      }
    }
    __syncthreads();
    for (int j = 0; j < PER; ++j) hist[threadIdx.x * PER + j] += part[threadIdx.x];
    for (int64_t T = threadIdx.x; T < P.nT; T += kBtPrepThreads) W.nbT[T] = 0;
    for (int64_t b = threadIdx.x; b < P.nbm; b += kBtPrepThreads) W.icnt[b] = 0;
    __syncthreads();
    // scatter; a query's rank fixes the row tile pairs its heads land in, whose block count
    // is the largest visible block count among their queries
    for (int64_t i = threadIdx.x; i < P.Q; i += kBtPrepThreads) {
      const int64_t nb = bt_nblocks(P.qpos[i], P);
      const int64_t r = atomicAdd(&hist[nb >> shift], 1);
      W.order[r] = (int32_t)i;
      const int64_t T1 = (r * P.n_kv + P.n_kv - 1) / kBtRowsT;
      for (int64_t T = r * P.n_kv / kBtRowsT; T <= T1; ++T) atomicMax(&W.nbT[T], (int32_t)nb);
    }
    return;
  }
  __shared__ float red[24];
  const int64_t cta = (int64_t)blockIdx.x - 1;
  if (cta < P.nbm) {
    bt_key_block(P.k, W.k16, cta, P.L, W.kb, W.ksc, red);
  } else {
    const int64_t r0 = (cta - P.nbm) * 32 + 4 * (threadIdx.x >> 5);
    bt_query_rows(P.q, W.q16, W.qab, W.qsig, r0, P.slots);
  }
}

// ------------------------------------------------------------ block maxima --
// Units are (row tile pair T, key block b), b < nbT[T], T-major; a CTA takes a
// contiguous range of them (balanced by count), so it reloads its 256 query
// rows only when T changes.
struct BtSched {
  int64_t T0, b0, count;
};

__device__ void bt_schedule(const BtProblem& P, const BtWs& W, BtSched* out) {
  const int lane = threadIdx.x & 31;
  int64_t total = 0;
  for (int64_t t0 = 0; t0 < P.nT; t0 += 32) {
    const int64_t t = t0 + lane;
    int64_t v = t < P.nT ? (int64_t)W.nbT[t] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    total += v;
  }
  const int64_t start = total * (int64_t)blockIdx.x / gridDim.x;
  const int64_t end = total * (int64_t)(blockIdx.x + 1) / gridDim.x;
  int64_t T0 = 0, b0 = 0;
  if (end > start) {
    int64_t run = 0;
    for (int64_t t0 = 0; t0 < P.nT; t0 += 32) {
      const int64_t t = t0 + lane;
      const int64_t v = t < P.nT ? (int64_t)W.nbT[t] : 0;
      int64_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      const int64_t chunk = __shfl_sync(0xffffffffu, incl, 31);
      if (run + chunk > start) {
        const unsigned hit = __ballot_sync(0xffffffffu, run + incl > start);
        const int first = __ffs(hit) - 1;
        const int64_t incl_f = __shfl_sync(0xffffffffu, incl, first);
        const int64_t v_f = __shfl_sync(0xffffffffu, v, first);
        T0 = t0 + first;
        b0 = start - (run + incl_f - v_f);
        break;
      }
      run += chunk;
    }
  }
  if (lane == 0) {
    out->T0 = T0;
    out->b0 = b0;
    out->count = end - start;
  }
}

struct BtUnits {
  const int32_t* nbT;
  int64_t T, b, left, nb;
  __device__ void init(const BtWs& W, const BtSched& s) {
    nbT = W.nbT;
    T = s.T0;
    b = s.b0;
    left = s.count;
    nb = left > 0 ? nbT[T] : 0;
  }
  __device__ bool valid() const { return left > 0; }
  __device__ void advance() {
    --left;
    if (left <= 0) return;
    ++b;
    while (b >= nb) {
      ++T;
      b = 0;
      nb = nbT[T];
    }
  }
};

__device__ __forceinline__ void bt_gather4(void* dst, const void* tmap, uint64_t* bar, int32_t x, int32_t y0,
                                           int32_t y1, int32_t y2, int32_t y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
      "%5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
      : "memory");
}

constexpr int kBtOffA = 0;
constexpr int kBtOffK = kBtOffA + 2 * kBtATile;
constexpr int kBtOffBar = kBtOffK + kBtKStages * kBtChunkBytes;
constexpr int kBtNBars = 2 + 2 * kBtKStages + 4 + 1;
constexpr int kBtOffMisc = kBtOffBar + kBtNBars * 8;
constexpr int kBtSmem = kBtOffMisc + 64 + 1024;
static_assert(kBtSmem <= 232448, "shared memory");

__global__ void __launch_bounds__(kBtThreads, 1)
    bt_max_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                  const BtProblem P, const BtWs W) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* sA = smem + kBtOffA;
  uint8_t* sK = smem + kBtOffK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBtOffBar);
  uint64_t* a_full = bars;
  uint64_t* a_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = k_full + kBtKStages;
  uint64_t* acc_full = k_empty + kBtKStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain_bar = acc_empty + 2;
  uint8_t* misc = smem + kBtOffMisc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  BtSched* sched = reinterpret_cast<BtSched*>(misc + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);   // the MMA-issuing thread, once per row tile pair
    for (int i = 0; i < kBtKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kBtNE);
    }
    mbar_init(&drain_bar[0], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_q);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kBtTmemCols);
  if (warp == 2) bt_schedule(P, W, sched);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const BtSched s = *sched;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    BtUnits u;
    u.init(W, s);
    int64_t cur_T = -1;
    uint32_t na = 0, nk = 0;
    bool live = true;
    while (u.valid() && live) {
      if (u.T != cur_T) {
        cur_T = u.T;
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(a_empty, (na & 1) ^ 1, abort_flag);
          if (ok) mbar_arrive_expect_tx(a_full, 2 * kBtATile);   // two tiles
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        __syncwarp();
        // lane l: rows 8l .. 8l+7 of the tile pair, four at a time, two K chunks each
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int r0 = 8 * lane + 4 * g;
          int32_t y[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int64_t slot = cur_T * kBtRowsT + r0 + i;
            y[i] = slot < P.slots ? (int32_t)bt_slot_pair(P, W, slot) : 0;
          }
          uint8_t* dst = sA + (r0 >> 7) * kBtATile + (r0 & 127) * 128;
#pragma unroll
          for (int c = 0; c < 2; ++c) bt_gather4(dst + c * kBtChunkBytes, &tmap_q, a_full, 64 * c, y[0], y[1], y[2], y[3]);
        }
        ++na;
      }
      for (int c = 0; c < 2; ++c) {
        const int st = nk % kBtKStages;
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(&k_empty[st], ((nk / kBtKStages) & 1) ^ 1, abort_flag);
          if (ok) {
            mbar_arrive_expect_tx(&k_full[st], kBtChunkBytes);
            tma_load_2d(sK + st * kBtChunkBytes, &tmap_k, &k_full[st], 64 * c, (int32_t)(u.b * 128));
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          live = false;
          break;
        }
        ++nk;
      }
      __syncwarp();
      if (live) u.advance();
    }
    // drain: the last phase issued on every barrier has landed
    if (lane == 0) {
      if (na > 0) mbar_wait_drain(a_full, (na - 1) & 1);
      for (uint32_t i = 0; i < (uint32_t)kBtKStages && i < nk; ++i) {
        const uint32_t j = nk - 1 - i;
        mbar_wait_drain(&k_full[j % kBtKStages], (j / kBtKStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    // One thread issues every unit, into accumulator stages 0 and 1 in turn (a
    // second issuing thread corrupted a few accumulator rows now and then).
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(128, 128, 0u);   // A, B fp16; D f32
      BtUnits u;
      u.init(W, s);
      int64_t cur_T = -1;
      uint32_t na = 0, nunit = 0;
      bool ok = true;
      while (u.valid() && ok) {
        if (u.T != cur_T) {
          cur_T = u.T;
          if (!(ok = mbar_wait(a_full, na & 1, abort_flag))) break;
          ++na;
        }
        {
          const uint32_t me = nunit & 1u;    // accumulator stage
          const uint32_t use = nunit >> 1;   // uses of that stage so far
          if (!(ok = mbar_wait(&acc_empty[me], (use & 1) ^ 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t d0 = tmem_base + me * 256u;
          for (int c = 0; c < 2 && ok; ++c) {
            const uint32_t nk = 2 * nunit + c;
            const int st = nk % kBtKStages;
            if (!(ok = mbar_wait(&k_full[st], (nk / kBtKStages) & 1, abort_flag))) break;
            tc_fence_after();
            const uint32_t kb = smem_u32(sK + st * kBtChunkBytes);
            const uint32_t a0 = smem_u32(sA + c * kBtChunkBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = smem_desc_sw128(kb + kk * 32);
              const uint32_t accum = (c | kk) ? 1u : 0u;
              tc_mma_f16(d0, smem_desc_sw128(a0 + kk * 32), bd, idesc, accum);
              tc_mma_f16(d0 + 128, smem_desc_sw128(a0 + kBtATile + kk * 32), bd, idesc, accum);
            }
            tc_commit(&k_empty[st]);
          }
          if (!ok) break;
          tc_commit(&acc_full[me]);
        }
        ++nunit;
        const int64_t T_this = u.T;
        u.advance();
        if (!u.valid() || u.T != T_this) tc_commit(a_empty);
      }
      // No commit may still be in flight when the CTA exits (its arrive would land
      // in the next kernel's shared memory): the thread waits for its drain commit
      // and for the last phases of the barriers its commits target.
      tc_commit(&drain_bar[0]);
      mbar_wait_drain(&drain_bar[0], 0);
      if (ok && !*abort_flag) {
        if (na > 0) mbar_wait_drain(a_empty, (na - 1) & 1);
        const uint32_t nk = 2 * nunit;
        for (uint32_t i = 0; i < (uint32_t)kBtKStages && i < nk; ++i) {
          const uint32_t j = nk - 1 - i;
          mbar_wait_drain(&k_empty[j % kBtKStages], (j / kBtKStages) & 1);
        }
      }
    }
  } else if (warp >= 2 && warp < 2 + kBtNE) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int tile = ew >> 2;
    const int row = tile * 128 + quarter * 32 + lane;
    BtUnits u;
    u.init(W, s);
    int64_t cur_T = -1, slot = 0, vis = 0;
    float sig = 1.0f;
    uint32_t nacc = 0;
    const float ninf = -__int_as_float(0x7f800000);
    while (u.valid()) {
      if (u.T != cur_T) {
        cur_T = u.T;
        slot = cur_T * kBtRowsT + row;
        vis = 0;
        if (slot < P.slots) {
          const int64_t qi = bt_slot_query(P, W, slot);
          const int64_t pos = P.qpos[qi];
          if (pos >= 0) vis = pos + 1 < P.L ? pos + 1 : P.L;
          sig = W.qsig[bt_slot_pair(P, W, slot)];
        }
      }
      const int acc = nacc & 1;
      const bool got = mbar_wait(&acc_full[acc], (nacc >> 1) & 1, abort_flag);
      __syncwarp();
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      uint32_t v0[32], v1[32], v2[32], v3[32];
      const uint32_t ta = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * 256 + tile * 128);
      tmem_ld_32x32b_x32(ta, v0);
      tmem_ld_32x32b_x32(ta + 32, v1);
      tmem_ld_32x32b_x32(ta + 64, v2);
      tmem_ld_32x32b_x32(ta + 96, v3);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      const int64_t nvis = vis - u.b * 128;
      if (nvis > 0) {
        float m0 = ninf, m1 = ninf, m2 = ninf, m3 = ninf;
        if (nvis >= 128) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            m0 = fmaxf(m0, __uint_as_float(v0[i]));
            m1 = fmaxf(m1, __uint_as_float(v1[i]));
            m2 = fmaxf(m2, __uint_as_float(v2[i]));
            m3 = fmaxf(m3, __uint_as_float(v3[i]));
          }
        } else {
          const int nv = (int)nvis;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            m0 = fmaxf(m0, i < nv ? __uint_as_float(v0[i]) : ninf);
            m1 = fmaxf(m1, i + 32 < nv ? __uint_as_float(v1[i]) : ninf);
            m2 = fmaxf(m2, i + 64 < nv ? __uint_as_float(v2[i]) : ninf);
            m3 = fmaxf(m3, i + 96 < nv ? __uint_as_float(v3[i]) : ninf);
          }
        }
        // A_b = sigma s_b max(acc): both scales are powers of two
        W.amax[slot * P.nbm + u.b] = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * (sig * W.ksc[u.b]);
      }
      ++nacc;
      u.advance();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kBtTmemCols);
  }
}

// ---------------------------------------------------------------- selection --
constexpr unsigned kFull = 0xffffffffu;

// The n-th largest (1 <= n <= count) of the keys key(i), i in [i0, i1): four
// 8-bit radix passes over a per-warp 256-bin histogram.  *need_eq: how many
// keys equal to the result belong to the top n.
template <class F>
__device__ uint32_t bt_warp_kth(const F& key, int64_t i0, int64_t i1, int64_t n, int32_t* hist, int64_t* need_eq) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0, pmask = 0;
  int64_t need = n;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    for (int64_t i = i0 + lane; i < i1; i += 32) {
      const uint32_t k = key(i);
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncwarp();
    // lane l holds digits 255 - 8l - j, j < 8 (descending)
    int c[8], csum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[255 - 8 * lane - j];
      csum += c[j];
    }
    int incl = csum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(kFull, (int64_t)incl >= need);
    const int fl = hit ? __ffs(hit) - 1 : 31;
    int digit = 0, above = 0;
    if (lane == fl) {
      int run = incl - csum;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if ((int64_t)(run + c[j]) >= need) {
          digit = 255 - 8 * lane - j;
          above = run;
          break;
        }
        run += c[j];
      }
    }
    digit = __shfl_sync(kFull, digit, fl);
    above = __shfl_sync(kFull, above, fl);
    prefix |= (uint32_t)digit << shift;
    pmask |= 255u << shift;
    need -= above;
    __syncwarp();
  }
  *need_eq = need;
  return prefix;
}

// Forced head [0, a), a middle of `mid` entries (written elsewhere) at [a, a+mid),
// the forced tail zs..n-1 after it, -1 padding; returns the count.
__device__ __forceinline__ int64_t bt_frame(int32_t* o, int Wd, int64_t a, int64_t mid, int64_t zs, int64_t n) {
  const int64_t cnt = a + mid + (n - zs);
  for (int j = threadIdx.x & 31; j < Wd; j += 32) {
    if (j < a) o[j] = j;
    else if (j >= a + mid) o[j] = j < cnt ? (int32_t)(zs + (j - a - mid)) : -1;
  }
  return cnt;
}

struct BtSlotGeom {
  int64_t qi, pair, n, a, zs, n_need;
  BlockGeom g;
};

// The route's block size is 128 and every index fits 32 bits: the geometry of
// block_geom in 32-bit arithmetic and shifts (no 64-bit division per pair).
__device__ __forceinline__ BtSlotGeom bt_slot_geom(const BtProblem& P, const BtWs& W, int64_t slot) {
  BtSlotGeom s;
  const uint32_t sl = (uint32_t)slot, nk = (uint32_t)P.n_kv;
  const uint32_t rank = sl / nk;
  s.qi = W.order[rank];
  s.pair = s.qi * P.n_kv + (int64_t)(sl - rank * nk);
  const int32_t pos = P.qpos[s.qi];
  const int32_t exist = (int32_t)P.nbm;
  const int32_t n = pos < 0 ? 0 : ((pos >> 7) + 1 < exist ? (pos >> 7) + 1 : exist);
  const int32_t init = P.c.init_blocks, local = P.c.local_blocks;
  const int32_t a = init < n ? init : n;
  int32_t zs = n - local;
  zs = zs < a ? a : zs;   // non-forced blocks: [a, zs)
  const int32_t n_forced = a + (n - zs);
  const int32_t budget = P.c.top_blocks > n_forced ? P.c.top_blocks : n_forced;
  s.g.n_blocks = n;
  s.g.n_forced = n_forced;
  s.g.budget = budget;
  s.g.scoring = n > 0 && !(n_forced >= budget || n_forced == n);
  s.n = n;
  s.a = a;
  s.zs = zs;
  s.n_need = budget - n_forced;
  return s;
}

// Lists `slot` for exact rescoring of block b.
__device__ __forceinline__ void bt_list(const BtProblem& P, const BtWs& W, int64_t slot, int64_t b) {
  const int p = atomicAdd(&W.icnt[b], 1);
  W.ilist[b * P.slots + p] = (int32_t)slot;
}

// counters: pairs scored, blocks bounded, blocks rescored, fallback pairs
// Bit-by-bit search for the n-th largest of the values v[u] (u < U, lanes
// hold lane + 32u; absent ones 0) starting from t with count(>= t) >= n and
// from bit hb down.
template <int U>
__device__ __forceinline__ uint32_t bt_bit_search(const uint32_t (&v)[8], uint32_t t, int hb, int n) {
  for (int bit = hb; bit >= 0; --bit) {
    const uint32_t cand = t | (1u << bit);
    int c = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) c += v[u] >= cand ? 1 : 0;
    if (__reduce_add_sync(kFull, c) >= n) t = cand;
  }
  return t;
}

// Candidates of a row of at most 32 R non-forced blocks [a, zs) with n <= 32,
// every bound key held in registers (lane holds blocks a + lane + 32 r): the
// cut T (the n-th largest lower bound) from the lanes' maxima and a bit search
// over the few keys above them, then the blocks with upper bound >= T written
// ascending to cb/clo/chi.  Returns their count, or -1 when the keys above the
// lanes' cut do not fit the scratch (heavy ties; the caller takes the general
// path).
template <int R>
__device__ int bt_cands_regs(const float* arow, const float2* kbs, float2 qab, int a, int zs, int n, int32_t* cb,
                             uint32_t* clo, uint32_t* chi, uint32_t* sk, uint32_t* T_out) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  uint32_t lo[R], hi[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int b = a + lane + 32 * r;
    lo[r] = 0u;
    hi[r] = 0u;
    if (b < zs) {
      const float A = arow[b], e = bt_bound(qab, kbs[b]);
      lo[r] = score_key(__fsub_rd(A, e));
      hi[r] = score_key(__fadd_ru(A, e));
    }
  }
  uint32_t mx = 0u;
#pragma unroll
  for (int r = 0; r < R; ++r) mx = lo[r] > mx ? lo[r] : mx;
  int ge = 0;
#pragma unroll
  for (int o = 0; o < 32; ++o) ge += __shfl_sync(kFull, mx, o) >= mx ? 1 : 0;
  uint32_t t0 = ge >= n ? mx : 0u, top = mx;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t u = __shfl_xor_sync(kFull, t0, o), w = __shfl_xor_sync(kFull, top, o);
    t0 = u > t0 ? u : t0;
    top = w > top ? w : top;
  }
  // the keys >= t0 (at least n of them; absent blocks hold 0 < t0 unless t0 is 0)
  int ns = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const bool in = a + lane + 32 * r < zs && lo[r] >= t0;
    const unsigned bal = __ballot_sync(kFull, in);
    if (in) {
      const int p = ns + __popc(bal & lt);
      if (p < kBtCapC) sk[p] = lo[r];
    }
    ns += __popc(bal);
  }
  if (ns > kBtCapC) return -1;
  __syncwarp();
  uint32_t v[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int i = lane + 32 * u;
    v[u] = i < ns ? sk[i] : 0u;
  }
  const int hb = (t0 ^ top) ? 31 - __clz(t0 ^ top) : -1;
  uint32_t T = hb >= 0 ? (t0 & ~((2u << hb) - 1u)) : t0;
  if (ns <= 64) T = bt_bit_search<2>(v, T, hb, n);
  else if (ns <= 128) T = bt_bit_search<4>(v, T, hb, n);
  else T = bt_bit_search<8>(v, T, hb, n);
  *T_out = T;
  // candidates: upper bound >= T, ascending
  int nc = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int b = a + lane + 32 * r;
    const bool c = b < zs && hi[r] >= T;
    const unsigned bal = __ballot_sync(kFull, c);
    if (c) {
      const int p = nc + __popc(bal & lt);
      if (p < kBtCapC) {
        cb[p] = b;
        clo[p] = lo[r];
        chi[p] = hi[r];
      }
    }
    nc += __popc(bal);
  }
  __syncwarp();
  return nc;
}

__device__ void bt_classify_slot(const BtProblem& P, const BtWs& W, int64_t slot, int32_t* out, int Wd,
                                 int32_t* out_count, int32_t* cb, uint32_t* clo, uint32_t* chi, int32_t* hist,
                                 uint32_t* sk, unsigned long long* cnt) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  const BtSlotGeom s = bt_slot_geom(P, W, slot);
  int32_t* o = out + s.pair * Wd;
  int4 st = make_int4(kBtDone, 0, 0, 0);
  int64_t count = 0;
  if (s.n == 0 || !s.g.scoring) {
    count = bt_frame(o, Wd, s.a, 0, s.zs, s.n);
  } else {
    const int64_t m = s.zs - s.a;
    if (lane == 0) {
      atomicAdd(&cnt[0], 1ull);
      atomicAdd(&cnt[1], (unsigned long long)m);
    }
    if (m <= s.n_need) {
      // every visible block is selected
      for (int j = lane; j < Wd; j += 32) o[j] = j < s.n ? j : -1;
      count = s.n;
    } else {
      const float2 qab = W.qab[s.pair];
      const float* arow = W.amax + slot * P.nbm;
      const float2* kbs = W.kb;
      int nc = -1;
      uint32_t T = 0;
      if (s.n_need <= 32) {
        if (m <= 512) nc = bt_cands_regs<16>(arow, kbs, qab, (int)s.a, (int)s.zs, (int)s.n_need, cb, clo, chi, sk, &T);
        else if (m <= 1024)
          nc = bt_cands_regs<32>(arow, kbs, qab, (int)s.a, (int)s.zs, (int)s.n_need, cb, clo, chi, sk, &T);
      }
      if (nc < 0) {
        // general rows: the cut by radix select over all blocks, then the candidates
        auto keys_of = [&](int64_t b) {
          const float A = arow[b], e = bt_bound(qab, kbs[b]);
          return make_uint2(score_key(__fsub_rd(A, e)), score_key(__fadd_ru(A, e)));
        };
        auto lo_key = [&](int64_t b) { return keys_of(b).x; };
        int64_t need_eq;
        T = bt_warp_kth(lo_key, s.a, s.zs, s.n_need, hist, &need_eq);
        nc = 0;
        for (int64_t b0 = s.a; b0 < s.zs; b0 += 32) {
          const int64_t b = b0 + lane;
          bool c = false;
          uint2 k2 = make_uint2(0u, 0u);
          if (b < s.zs) {
            k2 = keys_of(b);
            c = k2.y >= T;
          }
          const unsigned bal = __ballot_sync(kFull, c);
          if (c) {
            const int p = nc + __popc(bal & lt);
            if (p < kBtCapC) {
              cb[p] = (int32_t)b;
              clo[p] = k2.x;
              chi[p] = k2.y;
            }
          }
          nc += __popc(bal);
        }
        __syncwarp();
      }
      bool fallback = nc > kBtCapC;
      if (!fallback) {
        // certainly in: fewer than n_need other candidates reach its lower bound
        int k_in = 0;
        for (int i0 = 0; i0 < nc; i0 += 32) {
          const int i = i0 + lane;
          bool in = false;
          if (i < nc) {
            const uint32_t li = clo[i];
            int c = 0;
            for (int j = 0; j < nc; ++j) c += (j != i && chi[j] >= li) ? 1 : 0;
            in = c < s.n_need;
          }
          if (in) cb[i] |= (int32_t)0x80000000;
          k_in += __popc(__ballot_sync(kFull, in));
        }
        __syncwarp();
        const int nu = nc - k_in;
        const int64_t m_need = s.n_need - k_in;
        if (m_need == 0 || nu == m_need) {
          // decided: the certain ones (m_need == 0) or every candidate
          const bool all = m_need != 0;
          int w = 0;
          for (int i0 = 0; i0 < nc; i0 += 32) {
            const int i = i0 + lane;
            const bool sel = i < nc && (all || cb[i] < 0);
            const unsigned bal = __ballot_sync(kFull, sel);
            if (sel) o[s.a + w + __popc(bal & lt)] = cb[i] & 0x7fffffff;
            w += __popc(bal);
          }
          count = bt_frame(o, Wd, s.a, s.n_need, s.zs, s.n);
        } else if (nu > kBtCapU) {
          fallback = true;
        } else {
          // certain ones to o[a, a + k_in); undecided ones to the pair's list and the blocks' lists
          int wi = 0, wu = 0;
          for (int i0 = 0; i0 < nc; i0 += 32) {
            const int i = i0 + lane;
            const bool valid = i < nc;
            const bool in = valid && cb[i] < 0;
            const bool un = valid && !in;
            const unsigned bin = __ballot_sync(kFull, in), bun = __ballot_sync(kFull, un);
            if (in) o[s.a + wi + __popc(bin & lt)] = cb[i] & 0x7fffffff;
            if (un) {
              const int b = cb[i];
              W.ulist[slot * kBtCapU + wu + __popc(bun & lt)] = b;
              bt_list(P, W, slot, b);
            }
            wi += __popc(bin);
            wu += __popc(bun);
          }
          st = make_int4(kBtList, k_in, nu, (int)m_need);
          if (lane == 0) atomicAdd(&cnt[2], (unsigned long long)nu);
        }
      }
      if (fallback) {
        for (int64_t b = s.a + lane; b < s.zs; b += 32) bt_list(P, W, slot, b);
        st = make_int4(kBtFallback, 0, (int)m, (int)s.n_need);
        if (lane == 0) {
          atomicAdd(&cnt[2], (unsigned long long)m);
          atomicAdd(&cnt[3], 1ull);
        }
      }
    }
  }
  if (lane == 0) {
    W.sstat[slot] = st;
    if (st.x == kBtDone && out_count) out_count[s.pair] = (int32_t)count;
  }
}

constexpr int kBtWarps = 8;   // pairs per CTA in the per-pair kernels

__global__ void __launch_bounds__(32 * kBtWarps) bt_classify_kernel(BtProblem P, BtWs W, int32_t* out, int Wd,
                                                                      int32_t* out_count, block_select_stats* stats) {
  __shared__ uint32_t s_k[kBtWarps][kBtCapC];
  __shared__ int32_t s_b[kBtWarps][kBtCapC];
  __shared__ uint32_t s_lo[kBtWarps][kBtCapC];
  __shared__ uint32_t s_hi[kBtWarps][kBtCapC];
  __shared__ int32_t s_hist[kBtWarps][256];
  __shared__ unsigned long long s_cnt[4];
  if (threadIdx.x < 4) s_cnt[threadIdx.x] = 0;
  __syncthreads();
  const int wi = threadIdx.x >> 5;
  const int64_t slot = (int64_t)blockIdx.x * kBtWarps + wi;
  if (slot < P.slots)
    bt_classify_slot(P, W, slot, out, Wd, out_count, s_b[wi], s_lo[wi], s_hi[wi], s_hist[wi], s_k[wi], s_cnt);
  __syncthreads();
  if (stats && threadIdx.x < 4 && s_cnt[threadIdx.x])
    atomicAdd(&stats->pairs + threadIdx.x, s_cnt[threadIdx.x]);
}

// ------------------------------------------------------------ exact scores --
// One CTA (4 warps) per key block b.  The listed pairs go in rounds of 32:
//  1. one MMA (M = 128 positions of the block, N = 32 pairs, K = 128; the
//     same scaled fp16 operands as the block-max pass) gives A_p for every
//     position and pair, within e_b of the page's E_p;
//  2. per pair, A1 = max_p A_p; a position with A_p < A1 - 2 e_b has
//     E_p <= A_p + e_b < A1 - e_b <= E_p1 (p1 the position of A1), so the
//     block's exact maximum is among the positions with A_p >= A1 - 2 e_b
//     (usually one);
//  3. those positions are scored in the page's order (one thread per
//     (pair, position), products and sums rounded one by one) and the block
//     score E_b = max replaces A_b in the pair's row as an ordered key.
constexpr int kBtExactThreads = 128;
constexpr int kBtXN = 32;                          // pairs per round (MMA N)
constexpr int kBtXOffK = 0;                        // fp16 keys: 2 chunks x 128 rows x 128 B
constexpr int kBtXOffQ = kBtXOffK + 2 * kBtChunkBytes;   // fp16 query rows: 2 chunks x 32 rows x 128 B,
constexpr int kBtXOffT = kBtXOffQ;                       // then (the MMA done) A_p: [32 pairs][128 positions] fp32
constexpr int kBtXCap = 2048;                            // (pair, position) candidates per round
constexpr int kBtXOffL = kBtXOffT + kBtXN * 128 * 4;     // candidate list: kBtXCap x uint16
constexpr int kBtXOffM = kBtXOffL + kBtXCap * 2;         // misc
constexpr int kBtExactSmem = kBtXOffM + 1024 + 1024;

__global__ void __launch_bounds__(kBtExactThreads)
    bt_exact_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                    const BtProblem P, const BtWs W, block_select_stats* stats) {
  extern __shared__ uint8_t smem_raw[];
  const int64_t b = blockIdx.x;
  const int cnt = W.icnt[b];
  if (cnt == 0) return;
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* sK = smem + kBtXOffK;
  uint8_t* sQ = smem + kBtXOffQ;
  float* tr = reinterpret_cast<float*>(smem + kBtXOffT);
  uint16_t* lst = reinterpret_cast<uint16_t*>(smem + kBtXOffL);
  uint8_t* misc = smem + kBtXOffM;
  uint64_t* k_bar = reinterpret_cast<uint64_t*>(misc);
  uint64_t* q_bar = k_bar + 1;
  uint64_t* mma_bar = k_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 36);
  int* n_lst = reinterpret_cast<int*>(misc + 40);
  float* s_worst = reinterpret_cast<float*>(misc + 44);
  // per pair of the round
  uint32_t* ekey = reinterpret_cast<uint32_t*>(misc + 64);      // exact block score key
  float* scl = reinterpret_cast<float*>(misc + 192);             // sigma s_b
  int32_t* nvis = reinterpret_cast<int32_t*>(misc + 320);        // visible positions of the block
  int32_t* slot_of = reinterpret_cast<int32_t*>(misc + 448);     // slot
  int32_t* pair_of = reinterpret_cast<int32_t*>(misc + 576);     // pair (row of index_q, q16, qab)
  float* eb_of = reinterpret_cast<float*>(misc + 704);           // e_b
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int64_t k0 = b * 128;
  if (t == 0) {
    mbar_init(k_bar, 1);
    mbar_init(q_bar, 1);
    mbar_init(mma_bar, 1);
    *abort_flag = 0;
    *s_worst = 0.0f;
    fence_mbar_init();
    // the block's fp16 keys, needed by every round
    mbar_arrive_expect_tx(k_bar, 2 * kBtChunkBytes);
    tma_load_2d(sK, &tmap_k, k_bar, 0, (int32_t)k0);
    tma_load_2d(sK + kBtChunkBytes, &tmap_k, k_bar, 64, (int32_t)k0);
  }
  if (warp == 0) tmem_alloc(tmem_slot, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int32_t* items = W.ilist + b * P.slots;
  const float2 kb = W.kb[b];
  const float sb = W.ksc[b];
  const float ninf = -__int_as_float(0x7f800000);
  float worst = 0.0f;
  for (int base = 0, round = 0; base < cnt; base += kBtXN, ++round) {
    const int ni = cnt - base < kBtXN ? cnt - base : kBtXN;
    // ---- the round's pairs, looked up once
    if (t < kBtXN) {
      ekey[t] = 0u;
      if (t < ni) {
        const int64_t sl = items[base + t];
        const int64_t qi = bt_slot_query(P, W, sl);
        const int64_t pr = bt_slot_pair(P, W, sl);
        int64_t v = (int64_t)P.qpos[qi] + 1;
        v = v < P.L ? v : P.L;
        slot_of[t] = (int32_t)sl;
        pair_of[t] = (int32_t)pr;
        nvis[t] = (int32_t)(v - k0);
        scl[t] = W.qsig[pr] * sb;
        eb_of[t] = bt_bound(W.qab[pr], kb);
      } else {
        slot_of[t] = -1;
        pair_of[t] = 0;   // gathered but unused
        nvis[t] = 0;
        scl[t] = 0.0f;
        eb_of[t] = 0.0f;
      }
    }
    if (t == 0) *n_lst = 0;
    __syncthreads();
    // ---- operands and the MMA (one thread)
    if (warp == 0) {
      if (lane == 0) mbar_arrive_expect_tx(q_bar, 2 * kBtXN * 128);
      __syncwarp();
      if (lane < kBtXN / 4) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
          bt_gather4(sQ + c * (kBtXN * 128) + lane * 512, &tmap_q, q_bar, 64 * c, pair_of[4 * lane],
                     pair_of[4 * lane + 1], pair_of[4 * lane + 2], pair_of[4 * lane + 3]);
      }
      if (lane == 0) {
        bool ok = round > 0 || mbar_wait(k_bar, 0, abort_flag);
        ok = ok && mbar_wait(q_bar, round & 1, abort_flag);
        if (ok) {
          tc_fence_after();
          constexpr uint32_t idesc = idesc_f16(128, kBtXN, 0u);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t a0 = smem_u32(sK + c * kBtChunkBytes), b0 = smem_u32(sQ + c * (kBtXN * 128));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_f16(tmem_base, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc,
                         (c | kk) ? 1u : 0u);
          }
          tc_commit(mma_bar);
        }
      }
    }
    const bool got = mbar_wait(mma_bar, round & 1, abort_flag);
    if (!__syncthreads_and(got)) break;   // every thread leaves together
    tc_fence_after();
    // ---- A_p for this thread's position p = t and the round's pairs, transposed to [pair][position]
    {
      uint32_t v[32];
      tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(warp * 32) << 16), v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < kBtXN; ++j) tr[j * 128 + t] = t < nvis[j] ? __uint_as_float(v[j]) * scl[j] : ninf;
    }
    tc_fence_before();
    __syncthreads();
    // ---- per pair: A1, the threshold, the candidate positions
    for (int j = warp; j < ni; j += kBtExactThreads / 32) {
      const float4 a4 = *reinterpret_cast<const float4*>(tr + j * 128 + 4 * lane);
      float m = fmaxf(fmaxf(a4.x, a4.y), fmaxf(a4.z, a4.w));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      const float thr = __fsub_rd(m, __fmul_ru(2.0f, eb_of[j]));
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (av[i] >= thr) {
          const int pos = atomicAdd(n_lst, 1);
          if (pos < kBtXCap) lst[pos] = (uint16_t)((j << 7) | (4 * lane + i));
        }
      }
    }
    // A_p shares its bytes with the next round's query tile, written by TMA (the async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    // ---- the candidates in the page's order: one thread each, rows loaded 16 x 16 bytes at a time.
    // More candidates than the list holds (heavy ties): every visible position of the round's pairs.
    const int nl = *n_lst;
    const bool every = nl > kBtXCap;
    const int n_items = every ? ni * 128 : nl;
    for (int i = t; i < n_items; i += kBtExactThreads) {
      const int j = every ? i >> 7 : lst[i] >> 7, p = every ? i & 127 : lst[i] & 127;
      if (p >= nvis[j]) continue;
      const float4* qr = reinterpret_cast<const float4*>(P.q + (int64_t)pair_of[j] * 128);
      const float4* kr = reinterpret_cast<const float4*>(P.k + (k0 + p) * 128);
      float acc = 0.0f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float4 x[16], y[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          x[u] = __ldg(qr + 16 * h + u);
          y[u] = __ldg(kr + 16 * h + u);
        }
        asm volatile("" ::: "memory");   // all 32 loads issued before the serial sum consumes them
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          acc = __fadd_rn(acc, __fmul_rn(x[u].x, y[u].x));
          acc = __fadd_rn(acc, __fmul_rn(x[u].y, y[u].y));
          acc = __fadd_rn(acc, __fmul_rn(x[u].z, y[u].z));
          acc = __fadd_rn(acc, __fmul_rn(x[u].w, y[u].w));
        }
      }
      atomicMax(&ekey[j], score_key(acc));   // score_key folds -0 onto +0
    }
    __syncthreads();
    if (t < ni) {
      uint32_t* cell = reinterpret_cast<uint32_t*>(W.amax) + (int64_t)slot_of[t] * P.nbm + b;
      const float A = __uint_as_float(*cell);
      const float E = key_score(ekey[t]);
      if (eb_of[t] > 0.0f) worst = fmaxf(worst, fabsf(A - E) / eb_of[t]);
      *cell = ekey[t];
    }
    __syncthreads();
  }
  if (worst > 0.0f) atomicMax(reinterpret_cast<int*>(s_worst), __float_as_int(worst));
  tc_fence_before();
  __syncthreads();
  if (t == 0 && stats && *s_worst > 0.0f)
    atomicMax(reinterpret_cast<int*>(&stats->max_bound_use), __float_as_int(*s_worst));
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

// ---------------------------------------------------------------- resolve --
__device__ __forceinline__ int bt_count_below(const int32_t* v, int n, int32_t x) {
  int lo = 0, hi = n;   // first index with v[i] >= x (v ascending)
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(32 * kBtWarps) bt_resolve_kernel(BtProblem P, BtWs W, int32_t* out, int Wd,
                                                                     int32_t* out_count) {
  __shared__ uint32_t s_key[kBtWarps][kBtCapU];
  __shared__ int32_t s_blk[kBtWarps][kBtCapU];
  __shared__ int32_t s_win[kBtWarps][kBtCapU];
  __shared__ int32_t s_in[kBtWarps][kBtMaxTop];
  __shared__ int32_t s_hist[kBtWarps][256];
  const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  const int64_t slot = (int64_t)blockIdx.x * kBtWarps + wi;
  if (slot >= P.slots) return;
  const int4 st = W.sstat[slot];
  if (st.x == kBtDone) return;
  const BtSlotGeom s = bt_slot_geom(P, W, slot);
  const uint32_t* keys = reinterpret_cast<const uint32_t*>(W.amax) + slot * P.nbm;
  int32_t* o = out + s.pair * Wd;
  if (st.x == kBtList) {
    const int k_in = st.y, nu = st.z, m_need = st.w;
    uint32_t* sk = s_key[wi];
    int32_t* sb = s_blk[wi];
    int32_t* sw = s_win[wi];
    int32_t* si = s_in[wi];
    for (int i = lane; i < nu; i += 32) {
      const int32_t b = W.ulist[slot * kBtCapU + i];
      sb[i] = b;
      sk[i] = keys[b];
    }
    for (int i = lane; i < k_in; i += 32) si[i] = o[s.a + i];
    __syncwarp();
    // winners: rank < m_need by (exact key desc, block asc); kept ascending
    int w = 0;
    for (int i0 = 0; i0 < nu; i0 += 32) {
      const int i = i0 + lane;
      bool win = false;
      if (i < nu) {
        const uint32_t ki = sk[i];
        const int32_t bi = sb[i];
        int r = 0;
        for (int j = 0; j < nu; ++j) r += (sk[j] > ki || (sk[j] == ki && sb[j] < bi)) ? 1 : 0;
        win = r < m_need;
      }
      const unsigned bal = __ballot_sync(kFull, win);
      if (win) sw[w + __popc(bal & lt)] = sb[i];
      w += __popc(bal);
    }
    __syncwarp();
    // merge the two ascending, disjoint lists into o[a, a + n_need)
    for (int i = lane; i < k_in; i += 32) o[s.a + i + bt_count_below(sw, m_need, si[i])] = si[i];
    for (int i = lane; i < m_need; i += 32) o[s.a + i + bt_count_below(si, k_in, sw[i])] = sw[i];
  } else {
    // every non-forced block was rescored: the top n_need of [a, zs)
    int64_t need_eq;
    auto key = [&](int64_t b) { return keys[b]; };
    const uint32_t K = bt_warp_kth(key, s.a, s.zs, s.n_need, s_hist[wi], &need_eq);
    int64_t w = 0, eq_seen = 0;
    for (int64_t b0 = s.a; b0 < s.zs; b0 += 32) {
      const int64_t b = b0 + lane;
      const uint32_t k = b < s.zs ? keys[b] : 0u;
      const bool eq = b < s.zs && k == K;
      const unsigned beq = __ballot_sync(kFull, eq);
      const bool sel = (b < s.zs && k > K) || (eq && eq_seen + __popc(beq & lt) < need_eq);
      const unsigned bal = __ballot_sync(kFull, sel);
      if (sel) o[s.a + w + __popc(bal & lt)] = (int32_t)b;
      w += __popc(bal);
      eq_seen += __popc(beq);
    }
  }
  const int64_t count = bt_frame(o, Wd, s.a, s.n_need, s.zs, s.n);
  if (lane == 0 && out_count) out_count[s.pair] = (int32_t)count;
}

// ---------------------------------------------------------------- launcher --
static BtProblem bt_problem(const float* q, const float* k, const int32_t* pos, int64_t Q, int n_kv, int64_t L,
                            const block_sparse_config& c) {
  BtProblem P;
  P.q = q;
  P.k = k;
  P.qpos = pos;
  P.Q = Q;
  P.n_kv = n_kv;
  P.L = L;
  P.slots = Q * n_kv;
  P.nbm = (L + 127) / 128;
  P.nT = (P.slots + kBtRowsT - 1) / kBtRowsT;
  P.c = c;
  return P;
}

bool block_select_tc_applies(int D, const block_sparse_config& c, int64_t Q, int n_kv, int64_t L) {
  return D == 128 && c.block_size == 128 && c.top_blocks <= kBtMaxTop && n_kv > 0 &&
         Q * (int64_t)n_kv < ((int64_t)1 << 31) && L < ((int64_t)1 << 31) &&
         ((L + 127) / 128) * Q * (int64_t)n_kv < ((int64_t)1 << 40);
}

size_t block_select_tc_ws(int64_t Q, int n_kv, int64_t L, const block_sparse_config& c) {
  return bt_ws_bytes(bt_problem(nullptr, nullptr, nullptr, Q, n_kv, L, c));
}

cudaError_t launch_block_select_tc(const float* q, const float* k, const int32_t* pos, int64_t Q, int n_kv,
                                   int64_t L, const block_sparse_config& c, int32_t* out, int out_width,
                                   int32_t* out_count, void* ws, block_select_stats* stats, cudaStream_t st,
                                   const cudaEvent_t* ev) {
  const BtProblem P = bt_problem(q, k, pos, Q, n_kv, L, c);
  if (P.slots <= 0) return cudaSuccess;
  const BtWs W = bt_carve(ws, P);
  cudaError_t e;
  // ev (optional, 6 events): before prep, then after each of the five kernels
  auto mark = [&](int i) { return ev && ev[i] ? cudaEventRecord(ev[i], st) : cudaSuccess; };
  if ((e = mark(0)) != cudaSuccess) return e;
  {
    const int64_t g = 1 + P.nbm + (P.slots + 31) / 32;
    bt_prep_kernel<<<(unsigned)g, kBtPrepThreads, 0, st>>>(P, W);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = mark(1)) != cudaSuccess) return e;
  CUtensorMap tk, tq;
  if (P.nbm > 0) {
    bool ok = make_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, W.k16, 128, (uint64_t)L, 256, 64, 128);
    ok = ok && make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, W.q16, 128, (uint64_t)P.slots, 256, 64, 1);
    if (!ok) return cudaErrorInvalidValue;
    if ((e = cudaFuncSetAttribute(bt_max_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBtSmem)) !=
        cudaSuccess)
      return e;
    bt_max_kernel<<<sm_count(), kBtThreads, kBtSmem, st>>>(tk, tq, P, W);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = mark(2)) != cudaSuccess) return e;
  const unsigned gp = (unsigned)((P.slots + kBtWarps - 1) / kBtWarps);
  bt_classify_kernel<<<gp, 32 * kBtWarps, 0, st>>>(P, W, out, out_width, out_count, stats);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = mark(3)) != cudaSuccess) return e;
  if (P.nbm > 0) {
    if ((e = cudaFuncSetAttribute(bt_exact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBtExactSmem)) !=
        cudaSuccess)
      return e;
    bt_exact_kernel<<<(unsigned)P.nbm, kBtExactThreads, kBtExactSmem, st>>>(tk, tq, P, W, stats);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if ((e = mark(4)) != cudaSuccess) return e;
  bt_resolve_kernel<<<gp, 32 * kBtWarps, 0, st>>>(P, W, out, out_width, out_count);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return mark(5);
}

}  // namespace idx
