// MiniMax-M3 block-sparse selection ("ferrox_core/block_sparse.rs":
// block_sparse_select, select_for_head, dot).
//
// Two kernels:
//  1. block scores: for each (query, KV head) pair and each visible,
//     non-forced block, the max over the block's causally visible positions of
//     the raw dot q.k_p, with the page's summation order: acc starts at 0 and
//     acc = acc + q[d]*k[d] for d = 0..D-1, each product and each sum rounded
//     to fp32 on its own (no FMA).  That order is what makes the selected block
//     indices bit-exact, so this runs on the fp32 CUDA-core pipes, not the
//     tensor cores: block_score128_kernel for D = 128 (packed f32x2, two pairs
//     per lane, see below), block_score_kernel for any other D.
//  2. block_pick_kernel: per pair, forced blocks get the largest key, then the
//     exact top-`budget` of (score desc, block asc) is taken and written in
//     ascending block order.
#include <mutex>

#include "block_select.cuh"
#include "topk.cuh"

namespace idx {

constexpr int kBsThreads = 128;   // pairs per thread block
constexpr int kBsChunk = 64;      // key positions staged per round

// Any D: the query is read from global memory (L1), a chunk of keys is staged
// in shared memory, one thread per pair, scalar fp32 in the page's order.
__global__ void __launch_bounds__(kBsThreads) block_score_kernel(const float* __restrict__ q,
                                                                  const float* __restrict__ k,
                                                                  const int32_t* __restrict__ qpos, int64_t Q,
                                                                  int n_kv, int D, int64_t L,
                                                                  block_sparse_config c, int64_t nbm,
                                                                  uint32_t* __restrict__ bkey) {
  extern __shared__ __align__(16) float ks[];   // [chunk][D]
  const int64_t n_pairs = Q * n_kv;
  const int64_t pair = (int64_t)blockIdx.x * kBsThreads + threadIdx.x;
  const bool live = pair < n_pairs;
  const int64_t qi = live ? pair / n_kv : 0;
  const int64_t pos = live ? (int64_t)qpos[qi] : -1;
  const BlockGeom g = block_geom(pos, L, c);
  const int chunk = (int)max(1, min(kBsChunk, 16384 / D));
  const float* qrow = q + pair * (int64_t)D;
  for (int64_t b = blockIdx.y; b < nbm; b += gridDim.y) {
    const bool need = live && g.scoring && b < g.n_blocks && !block_forced(b, g.n_blocks, c);
    if (!__syncthreads_or(need)) continue;
    const int64_t start = b * c.block_size;
    int64_t bend = start + c.block_size;
    bend = bend < L ? bend : L;
    const int64_t vend = pos + 1 < bend ? pos + 1 : bend;   // this thread's visible end
    float best = -__int_as_float(0x7f800000);
    for (int64_t c0 = start; c0 < bend; c0 += chunk) {
      const int cl = (int)((bend - c0) < chunk ? (bend - c0) : chunk);
      __syncthreads();
      for (int i = threadIdx.x; i < cl * D; i += kBsThreads) ks[i] = __ldg(k + c0 * D + i);
      __syncthreads();
      if (!need) continue;
      int nv = (int)(vend - c0);
      nv = nv < 0 ? 0 : (nv > cl ? cl : nv);
      for (int p = 0; p < nv; ++p) {
        float a = 0.0f;
        for (int d = 0; d < D; ++d) a = __fadd_rn(a, __fmul_rn(__ldg(qrow + d), ks[p * D + d]));
        best = fmaxf(best, __fadd_rn(a, 0.0f));
      }
    }
    if (need) bkey[pair * nbm + b] = score_key(best);
  }
}

// ------------------------------------------------------------ D == 128 --
// Same scores, with packed products and half the shared-memory traffic per
// operation:
//  * one packed f32x2 multiply forms two keys' products (each half rounded as
//    the scalar instruction rounds); the two sums are scalar adds, since a
//    packed multiply feeding a packed add is fused into a packed fma by code
//    generation (see f2_add_halves);
//  * lanes 2i and 2i+1 hold the two halves (d < 64, d >= 64) of the queries of
//    two pairs, so every key value a lane loads serves two pairs.  Keys go in
//    groups of 8: the even lane sums d = 0..63 of a group while the odd lane
//    finishes d = 64..127 of the previous group from the even lane's partial
//    sums (handed over by a shuffle), so every chain is still the page's
//    sequential sum over d = 0..127.
//  * a block of up to 128 keys is staged transposed ([d][key]) so that one
//    16-byte load gives four keys' d-th elements.
constexpr int kBs128Keys = 128;   // keys staged per round

// One 8-key group, this lane's half of D: chains (keys 8g+2j, 8g+2j+1) of
// pair A in acc[j], of pair B in acc[4+j], j < 4; kcol = kt + (64 h) * 128 + 8 g.
__device__ __forceinline__ void bs128_group(const float* kcol, const float (&qa)[64], const float (&qb)[64],
                                            uint64_t (&acc)[8]) {
#pragma unroll
  for (int dd = 0; dd < 64; ++dd) {
    const float4 u = *reinterpret_cast<const float4*>(kcol + dd * kBs128Keys);
    const float4 v = *reinterpret_cast<const float4*>(kcol + dd * kBs128Keys + 4);
    const uint64_t k01 = f2_pack(u.x, u.y), k23 = f2_pack(u.z, u.w);
    const uint64_t k45 = f2_pack(v.x, v.y), k67 = f2_pack(v.z, v.w);
    const uint64_t xa = f2_pack(qa[dd], qa[dd]);
    const uint64_t xb = f2_pack(qb[dd], qb[dd]);
    acc[0] = f2_add_halves(acc[0], f2_mul(xa, k01));
    acc[1] = f2_add_halves(acc[1], f2_mul(xa, k23));
    acc[2] = f2_add_halves(acc[2], f2_mul(xa, k45));
    acc[3] = f2_add_halves(acc[3], f2_mul(xa, k67));
    acc[4] = f2_add_halves(acc[4], f2_mul(xb, k01));
    acc[5] = f2_add_halves(acc[5], f2_mul(xb, k23));
    acc[6] = f2_add_halves(acc[6], f2_mul(xb, k45));
    acc[7] = f2_add_halves(acc[7], f2_mul(xb, k67));
  }
}

__global__ void __launch_bounds__(kBsThreads) block_score128_kernel(const float* __restrict__ q,
                                                                    const float* __restrict__ k,
                                                                    const int32_t* __restrict__ qpos, int64_t Q,
                                                                    int n_kv, int64_t L, block_sparse_config c,
                                                                    int64_t nbm, uint32_t* __restrict__ bkey) {
  extern __shared__ __align__(16) float kt[];   // [128 d][128 keys]
  const int t = threadIdx.x, h = t & 1;
  const int64_t n_pairs = Q * n_kv;
  const int64_t pA = (int64_t)blockIdx.x * kBsThreads + (t & ~1), pB = pA + 1;
  const bool liveA = pA < n_pairs, liveB = pB < n_pairs;
  const int64_t posA = liveA ? (int64_t)qpos[pA / n_kv] : -1;
  const int64_t posB = liveB ? (int64_t)qpos[pB / n_kv] : -1;
  const BlockGeom gA = block_geom(posA, L, c), gB = block_geom(posB, L, c);
  float qa[64], qb[64];
  {
    const float4* ra = reinterpret_cast<const float4*>(q + pA * 128 + 64 * h);
    const float4* rb = reinterpret_cast<const float4*>(q + pB * 128 + 64 * h);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 va = liveA ? __ldg(ra + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 vb = liveB ? __ldg(rb + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      qa[4 * i] = va.x; qa[4 * i + 1] = va.y; qa[4 * i + 2] = va.z; qa[4 * i + 3] = va.w;
      qb[4 * i] = vb.x; qb[4 * i + 1] = vb.y; qb[4 * i + 2] = vb.z; qb[4 * i + 3] = vb.w;
    }
  }
  for (int64_t b = blockIdx.y; b < nbm; b += gridDim.y) {
    const bool needA = liveA && gA.scoring && b < gA.n_blocks && !block_forced(b, gA.n_blocks, c);
    const bool needB = liveB && gB.scoring && b < gB.n_blocks && !block_forced(b, gB.n_blocks, c);
    if (!__syncthreads_or(needA || needB)) continue;
    const int64_t start = b * c.block_size;
    int64_t bend = start + c.block_size;
    bend = bend < L ? bend : L;
    const int64_t vendA = posA + 1 < bend ? posA + 1 : bend;   // visible ends
    const int64_t vendB = posB + 1 < bend ? posB + 1 : bend;
    float bestA = -__int_as_float(0x7f800000), bestB = bestA;
    for (int64_t c0 = start; c0 < bend; c0 += kBs128Keys) {
      const int cl = (int)((bend - c0) < kBs128Keys ? (bend - c0) : kBs128Keys);
      __syncthreads();
      {
        // transposed staging: lanes take consecutive keys of one 16-byte column
        const float4* src = reinterpret_cast<const float4*>(k + c0 * 128);
        for (int i = t; i < cl * 32; i += kBsThreads) {
          const int key = i % cl, d4 = i / cl;
          const float4 v = __ldg(src + key * 32 + d4);
          kt[(4 * d4 + 0) * kBs128Keys + key] = v.x;
          kt[(4 * d4 + 1) * kBs128Keys + key] = v.y;
          kt[(4 * d4 + 2) * kBs128Keys + key] = v.z;
          kt[(4 * d4 + 3) * kBs128Keys + key] = v.w;
        }
      }
      __syncthreads();
      int nvA = needA ? (int)(vendA - c0) : 0, nvB = needB ? (int)(vendB - c0) : 0;
      nvA = nvA < 0 ? 0 : (nvA > cl ? cl : nvA);
      nvB = nvB < 0 ? 0 : (nvB > cl ? cl : nvB);
      const int mine = ((nvA > nvB ? nvA : nvB) + 7) >> 3;
      const int ng = __reduce_max_sync(0xffffffffu, mine);   // 8-key groups this warp runs
      uint64_t recv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) recv[j] = 0;
      // step s: the even lane takes group s, the odd lane group s - 1
      for (int st = 0; st <= ng; ++st) {
        const int g = st - h;
        const bool active = g >= 0 && g < ng;
        uint64_t acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = h ? recv[j] : 0ull;
        if (active) bs128_group(kt + (64 * h) * kBs128Keys + 8 * g, qa, qb, acc);
#pragma unroll
        for (int j = 0; j < 8; ++j) recv[j] = shfl_xor_u64(acc[j], 1);
        if (h && active) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float x0, x1, y0, y1;
            f2_unpack(acc[j], &x0, &x1);
            f2_unpack(acc[4 + j], &y0, &y1);
            const int key = 8 * g + 2 * j;
            if (key < nvA) bestA = fmaxf(bestA, __fadd_rn(x0, 0.0f));
            if (key + 1 < nvA) bestA = fmaxf(bestA, __fadd_rn(x1, 0.0f));
            if (key < nvB) bestB = fmaxf(bestB, __fadd_rn(y0, 0.0f));
            if (key + 1 < nvB) bestB = fmaxf(bestB, __fadd_rn(y1, 0.0f));
          }
        }
      }
    }
    if (h) {
      if (needA) bkey[pA * nbm + b] = score_key(bestA);
      if (needB) bkey[pB * nbm + b] = score_key(bestB);
    }
  }
}

constexpr int kPickThreads = 256;

struct BlockKeyRow {
  const uint32_t* k;
  int64_t n_blocks;
  block_sparse_config c;
  __device__ int n() const { return (int)n_blocks; }
  __device__ uint32_t key(int b) const { return block_forced(b, n_blocks, c) ? 0xffffffffu : k[b]; }
  __device__ int32_t id(int b) const { return b; }
};

__global__ void __launch_bounds__(kPickThreads) block_pick_kernel(const int32_t* __restrict__ qpos, int64_t Q,
                                                                   int n_kv, int64_t L, block_sparse_config c,
                                                                   int64_t nbm, const uint32_t* __restrict__ bkey,
                                                                   int32_t* __restrict__ out, int W,
                                                                   int32_t* __restrict__ out_count) {
  __shared__ TopkShared<kPickThreads> sh;
  extern __shared__ uint64_t sel[];
  const int64_t pair = blockIdx.x;
  const int64_t qi = pair / n_kv;
  const BlockGeom g = block_geom(qpos[qi], L, c);
  int32_t* o = out + pair * (int64_t)W;
  int count;
  if (g.n_blocks == 0) {
    count = 0;
    for (int j = threadIdx.x; j < W; j += kPickThreads) o[j] = -1;
  } else if (!g.scoring) {
    // the forced blocks are the whole selection: [0, a) then [max(n-local,0), n)
    const int64_t n = g.n_blocks;
    const int64_t a = c.init_blocks < n ? c.init_blocks : n;
    int64_t z = n - c.local_blocks;
    z = z < 0 ? 0 : z;
    const int64_t zs = z > a ? z : a;          // skip the overlap
    count = (int)(a + (n - zs));
    for (int j = threadIdx.x; j < W; j += kPickThreads) {
      int64_t v = -1;
      if (j < a) v = j;
      else if (j < count) v = zs + (j - a);
      o[j] = (int32_t)v;
    }
  } else {
    BlockKeyRow row{bkey + pair * nbm, g.n_blocks, c};
    count = block_topk<kPickThreads>(sh, sel, row, (int)g.budget, o, nullptr, true);
    for (int j = (int)g.budget + threadIdx.x; j < W; j += kPickThreads) o[j] = -1;
  }
  if (out_count && threadIdx.x == 0) out_count[pair] = count;
}

// Scratch of the CUDA-core route: one ordered key per (pair, block).
static size_t block_select_core_ws(int64_t Q, int n_kv, int64_t L, const block_sparse_config& c) {
  if (c.block_size <= 0) return 0;
  int64_t nbm = (L + c.block_size - 1) / c.block_size;
  return (size_t)(Q * n_kv) * (size_t)nbm * sizeof(uint32_t);
}

// D is not an argument of the workspace query: a configuration the tensor-core
// route may take (block size 128, D = 128) gets room for it.
size_t block_select_ws(int64_t Q, int n_kv, int64_t L, const block_sparse_config& c) {
  size_t w = block_select_core_ws(Q, n_kv, L, c);
  if (block_select_tc_applies(128, c, Q, n_kv, L)) {
    const size_t t = block_select_tc_ws(Q, n_kv, L, c);
    w = t > w ? t : w;
  }
  return w;
}

cudaError_t launch_block_select(const float* q, const float* k, const int32_t* pos, int64_t Q, int n_kv, int D,
                                int64_t L, const block_sparse_config& c, int32_t* out, int out_width,
                                int32_t* out_count, void* ws, cudaStream_t st, block_select_stats* stats,
                                bool tensor_route, const cudaEvent_t* ev) {
  const int64_t pairs = Q * n_kv;
  if (pairs <= 0) return cudaSuccess;
  if (tensor_route && block_select_tc_applies(D, c, Q, n_kv, L))
    return launch_block_select_tc(q, k, pos, Q, n_kv, L, c, out, out_width, out_count, ws, stats, st, ev);
  cudaError_t e;
  // CUDA-core route: events 0 and 5 only (before and after)
  if (ev && ev[0] && (e = cudaEventRecord(ev[0], st)) != cudaSuccess) return e;
  const int64_t nbm = c.block_size > 0 ? (L + c.block_size - 1) / c.block_size : 0;
  uint32_t* bkey = (uint32_t*)ws;
  if (nbm > 0) {
    dim3 grid((unsigned)((pairs + kBsThreads - 1) / kBsThreads), (unsigned)(nbm < 65535 ? nbm : 65535));
    if (D == 128) {
      const int smem128 = 128 * kBs128Keys * (int)sizeof(float);
      e = cudaFuncSetAttribute(block_score128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem128);
      if (e != cudaSuccess) return e;
      block_score128_kernel<<<grid, kBsThreads, smem128, st>>>(q, k, pos, Q, n_kv, L, c, nbm, bkey);
    } else {
      int chunk = D > 0 ? (16384 / D < kBsChunk ? 16384 / D : kBsChunk) : 1;
      chunk = chunk < 1 ? 1 : chunk;
      size_t smem = (size_t)chunk * D * sizeof(float);
      e = cudaFuncSetAttribute(block_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      block_score_kernel<<<grid, kBsThreads, smem, st>>>(q, k, pos, Q, n_kv, D, L, c, nbm, bkey);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  int Kmax = c.top_blocks > c.init_blocks + c.local_blocks ? c.top_blocks : c.init_blocks + c.local_blocks;
  int P = 1;
  while (P < Kmax) P <<= 1;
  size_t smem = (size_t)P * sizeof(uint64_t);
  e = cudaFuncSetAttribute(block_pick_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(IDX_MAX_K * sizeof(uint64_t)));
  if (e != cudaSuccess) return e;
  block_pick_kernel<<<(unsigned)pairs, kPickThreads, smem, st>>>(pos, Q, n_kv, L, c, nbm, bkey, out, out_width,
                                                                out_count);
  e = cudaGetLastError();
  if (e == cudaSuccess && ev && ev[5]) e = cudaEventRecord(ev[5], st);
  return e;
}

// ------------------------------------------------------- block positions --
// positions_of_blocks: one CTA per (query, head) row.  The row's block ids
// (negative entries dropped) are sorted ascending in shared memory and
// repeats removed; distinct blocks cover disjoint position ranges, ordered as
// the blocks, so concatenating each block's clipped range [b bs, min((b+1) bs,
// L, pos+1)) gives the covered positions ascending and without repeats.
constexpr int kBpThreads = 256;

__global__ void __launch_bounds__(kBpThreads) block_positions_kernel(const int32_t* __restrict__ blocks,
                                                                      const int32_t* __restrict__ counts, int W,
                                                                      int P2, const int32_t* __restrict__ qpos,
                                                                      int n_kv, int64_t L, int bs,
                                                                      int32_t* __restrict__ out, int ow,
                                                                      int32_t* __restrict__ out_count) {
  extern __shared__ int32_t sb[];   // [P2] block ids, then [P2 + 1] exclusive scan of the covered lengths
  int32_t* off = sb + P2;
  const int64_t row = blockIdx.x;
  const int t = threadIdx.x;
  int n = counts ? counts[row] : W;
  n = n < 0 ? 0 : (n > W ? W : n);
  const int64_t pos = qpos[row / n_kv];
  int64_t end_all = pos + 1 < L ? pos + 1 : L;
  end_all = end_all < 0 ? 0 : end_all;
  const int32_t* brow = blocks + row * (int64_t)W;
  for (int j = t; j < P2; j += kBpThreads) {
    const int32_t b = j < n ? brow[j] : -1;
    sb[j] = b >= 0 ? b : INT32_MAX;   // dropped entries sort last
  }
  __syncthreads();
  // bitonic sort, ascending
  for (int k = 2; k <= P2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = t; i < P2; i += kBpThreads) {
        const int x = i ^ j;
        if (x > i) {
          const int32_t a = sb[i], c = sb[x];
          const bool up = (i & k) == 0;
          if ((a > c) == up) {
            sb[i] = c;
            sb[x] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  // covered length per entry (0 for dropped entries and repeats), then an exclusive scan
  // (a single warp over P2 <= 4096 entries, 128 per lane at most)
  if (t < 32) {
    const int per = P2 / 32;
    int run = 0;
    for (int q = 0; q < per; ++q) {
      const int j = t * per + q;
      const int32_t b = sb[j];
      int len = 0;
      if (b != INT32_MAX && (j == 0 || sb[j - 1] != b) && bs > 0) {
        const int64_t st = (int64_t)b * bs;
        int64_t en = st + bs;
        en = en < end_all ? en : end_all;
        len = en > st ? (int)(en - st) : 0;
      }
      off[j] = len;
      run += len;
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (t >= o) incl += u;
    }
    int acc = incl - run;
    for (int q = 0; q < per; ++q) {
      const int j = t * per + q;
      const int len = off[j];
      off[j] = acc;
      acc += len;
    }
    if (t == 31) off[P2] = acc;
  }
  __syncthreads();
  const int total = off[P2];
  int32_t* orow = out + row * (int64_t)ow;
  // each warp writes whole blocks, lanes over consecutive positions
  const int warp = t >> 5, lane = t & 31;
  for (int j = warp; j < P2; j += kBpThreads / 32) {
    const int len = off[j + 1] - off[j];
    if (len <= 0) continue;
    const int64_t st = (int64_t)sb[j] * bs;
    for (int i = lane; i < len; i += 32) orow[off[j] + i] = (int32_t)(st + i);
  }
  for (int i = total + t; i < ow; i += kBpThreads) orow[i] = -1;
  if (out_count && t == 0) out_count[row] = total;
}

cudaError_t launch_block_positions(const int32_t* blocks, const int32_t* counts, int64_t rows, int W,
                                   const int32_t* qpos, int n_kv, int64_t L, int bs, int32_t* out, int ow,
                                   int32_t* out_count, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  int P2 = 32;
  while (P2 < W) P2 <<= 1;
  const size_t smem = (size_t)(2 * P2 + 1) * sizeof(int32_t);
  cudaError_t e = cudaFuncSetAttribute(block_positions_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  block_positions_kernel<<<(unsigned)rows, kBpThreads, smem, st>>>(blocks, counts, W, P2, qpos, n_kv, L, bs, out, ow,
                                                                   out_count);
  return cudaGetLastError();
}

}  // namespace idx

// ---------------------------------------------------------------------------
// block_select_static: the same selection with its block-score scratch in a
// file-scope device array instead of a caller workspace, for callers that
// cannot allocate device memory.  The array is part of the library's device
// image: every GPU that loads the library holds kStaticBlockScores words of it
// until the process exits.  Its device address is looked up once per device
// (cudaGetSymbolAddress, with that device current) on the first call made on
// that device.
// ---------------------------------------------------------------------------

namespace idx {

constexpr int64_t kStaticBlockScores = (int64_t)1 << 23;   // 8 Mi words = 32 MiB
static __device__ __align__(256) uint32_t g_block_scores_static[kStaticBlockScores];

constexpr int kMaxStaticDevices = 64;
static std::mutex g_static_mu;
static void* g_static_ptr[kMaxStaticDevices];

static idx_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(IDX_ERR_CUDA, "block_select_static: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxStaticDevices)
    return fail(IDX_ERR_UNSUPPORTED, "block_select_static: device ordinal %d above %d", dev, kMaxStaticDevices - 1);
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_block_scores_static);
    if (e != cudaSuccess || !p)
      return fail(IDX_ERR_CUDA, "block_select_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return IDX_OK;
}

}  // namespace idx

extern "C" idx_status block_select_static(const float* index_q, const float* index_k, const int32_t* query_pos,
                                          int64_t Q, int32_t n_kv, int32_t D, int64_t L,
                                          const block_sparse_config* cfg, int32_t* out, int32_t out_width,
                                          int32_t* out_count, void* stream) {
  using namespace idx;
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
  // Q * n_kv * ceil(L / block_size) against the fixed array, by division so that
  // no product can wrap before it is compared
  const int64_t nbm = cfg->block_size > 0 ? (L + cfg->block_size - 1) / cfg->block_size : 0;
  const bool too_big = Q > 0 && n_kv > 0 && nbm > 0 &&
                       (Q > kStaticBlockScores / n_kv || nbm > kStaticBlockScores / (Q * n_kv));
  if (too_big)
    return fail(IDX_ERR_WORKSPACE_TOO_SMALL,
                "block_select_static: Q=%lld x n_kv=%d x %lld blocks exceed the fixed %lld block scores",
                (long long)Q, n_kv, (long long)nbm, (long long)kStaticBlockScores);
  if (Q * n_kv == 0) return IDX_OK;
  if (!index_q || !query_pos || !out || (L > 0 && !index_k)) return fail(IDX_ERR_INVALID_ARG, "NULL pointer");
  void* scratch = nullptr;
  idx_status st = static_scratch(&scratch);
  if (st != IDX_OK) return st;
  cudaError_t e = launch_block_select(index_q, index_k, query_pos, Q, n_kv, D, L, *cfg, out, out_width, out_count,
                                      scratch, (cudaStream_t)stream, nullptr, false);
  if (e != cudaSuccess) return fail(IDX_ERR_CUDA, "block_select_static: %s", cudaGetErrorString(e));
  return IDX_OK;
}
