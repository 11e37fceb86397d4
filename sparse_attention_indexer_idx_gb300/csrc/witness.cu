// Segment-witness covering pass ("Segment Witnesses": sections "Object" and
// "Implementation rule and contracts").
//
// One thread block (8 warps) per row.  Occupancy is a 64-bit mask (S <= 64, as
// the fused kernel of the source pull request carries it): every thread ORs the
// segments of its share of the row (all of its loads issued first), the warps'
// masks are OR-combined in shared memory, and after a barrier -- every entry
// has been read before any slot is written -- lane s of the first two warps
// knows whether segment s is a witness and, from a popcount of the lower
// unoccupied segments, which slot it goes to.  The row is read once
// (coalesced int32) and at most B slots are written.
#include "internal.h"

namespace idx {

__device__ __forceinline__ uint64_t warp_or64(uint64_t v) {
  uint32_t lo = (uint32_t)v, hi = (uint32_t)(v >> 32);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo |= __shfl_xor_sync(0xffffffffu, lo, o);
    hi |= __shfl_xor_sync(0xffffffffu, hi, o);
  }
  return ((uint64_t)hi << 32) | lo;
}

// Segment of an entry: for 0 <= x < L, sigma(x) = floor(x S_eff / L) is the
// largest s < S_eff whose left edge e_s = ceil(s L / S_eff) is <= x (x lies in
// I_s = [e_s, e_{s+1}) exactly when sigma(x) = s).  The edges (int32, since
// L is) are computed once per row, lane l holding e_l and e_{l+32}; per entry
// a float estimate of x S_eff / L, off by at most one, is corrected against
// the edges fetched by warp shuffles -- no 64-bit division per entry.  Entries
// x >= L mark min(floor(x S_eff / L), S - 1): S - 1 when S_eff = S, else
// (S_eff = L) min(x, S - 1).
__device__ __forceinline__ int32_t edge_at(int32_t e_lo, int32_t e_hi, int s) {
  const int32_t lo = __shfl_sync(0xffffffffu, e_lo, s & 31);
  const int32_t hi = __shfl_sync(0xffffffffu, e_hi, s & 31);
  return s < 32 ? lo : hi;
}

constexpr int kWitThreads = 256;
constexpr int kWitPer = 8;        // entries per thread per round (loads in flight)

// Occupied-segment mask of one row, OR-combined over the thread block
// (entries x >= 0 mark min(sigma(x), S-1)).
__device__ __forceinline__ uint64_t row_occupancy(const int32_t* row, int topk, int64_t L, int S, int64_t s_eff,
                                                  uint64_t* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int32_t big = 0x7fffffff;
  const int32_t e_lo = lane < s_eff ? (int32_t)(((int64_t)lane * L + s_eff - 1) / s_eff) : big;
  const int32_t e_hi = lane + 32 < s_eff ? (int32_t)(((int64_t)(lane + 32) * L + s_eff - 1) / s_eff) : big;
  const float ratio = (float)s_eff / (float)L;
  const int smax = (int)s_eff - 1;
  uint64_t m = 0;
  for (int i0 = 0; i0 < topk; i0 += kWitThreads * kWitPer) {
    int32_t xv[kWitPer];
#pragma unroll
    for (int u = 0; u < kWitPer; ++u) {
      const int i = i0 + u * kWitThreads + (int)threadIdx.x;
      xv[u] = i < topk ? row[i] : -1;
    }
#pragma unroll
    for (int u = 0; u < kWitPer; ++u) {
      const int32_t x = xv[u];
      int seg = (int)((float)(x < 0 ? 0 : x) * ratio);
      seg = seg > smax ? smax : seg;
      // correct the estimate by one step either way (edges are monotone); every
      // lane takes part in both shuffles, whatever its entry
      const int nxt = seg < smax ? seg + 1 : seg;
      const int32_t e_nxt_raw = edge_at(e_lo, e_hi, nxt);
      const int32_t e_this = edge_at(e_lo, e_hi, seg);
      const int32_t e_next = seg < smax ? e_nxt_raw : big;
      if (e_next <= x) ++seg;
      else if (e_this > x && seg > 0) --seg;
      int64_t sg = seg;
      if ((int64_t)x >= L) sg = (s_eff == S) ? (int64_t)(S - 1) : ((int64_t)x < S - 1 ? (int64_t)x : (int64_t)(S - 1));
      if (x >= 0) m |= 1ull << sg;
    }
  }
  m = warp_or64(m);
  if (lane == 0) red[wid] = m;
  __syncthreads();
  uint64_t all = 0;
#pragma unroll
  for (int w = 0; w < kWitThreads / 32; ++w) all |= red[w];
  return all;
}

__global__ void __launch_bounds__(kWitThreads) witness_merge_kernel(int32_t* __restrict__ ids, int64_t rows,
                                                                     int topk, const int32_t* __restrict__ ctx,
                                                                     int keep, int S, int B) {
  __shared__ uint64_t red[kWitThreads / 32];
  const int64_t r = blockIdx.x;
  const int64_t L = ctx[r];
  if (L <= 0) return;                               // fallback: no witnesses
  const int64_t s_eff = L < S ? L : S;
  int32_t* row = ids + r * (int64_t)topk;
  const uint64_t occ = row_occupancy(row, topk, L, S, s_eff, red);
  const uint64_t part = (s_eff >= 64) ? ~0ull : ((1ull << s_eff) - 1ull);
  const uint64_t missing = ~occ & part;
  const int s = (int)threadIdx.x;                   // segments 0..63 on the first two warps
  if (s < s_eff && ((missing >> s) & 1ull)) {
    const uint64_t below = (s == 0) ? 0ull : (missing & ((1ull << s) - 1ull));
    const int rank = __popcll(below);
    if (rank < B) row[keep + rank] = (int32_t)(((int64_t)s * L + s_eff - 1) / s_eff);   // ceil(s L / S_eff)
  }
}

__global__ void __launch_bounds__(kWitThreads) witness_indices_kernel(const int32_t* __restrict__ ids, int64_t rows,
                                                                       int topk, const int32_t* __restrict__ ctx,
                                                                       int S, int32_t* __restrict__ out) {
  __shared__ uint64_t red[kWitThreads / 32];
  const int64_t r = blockIdx.x;
  const int64_t L = ctx[r];
  int32_t* o = out + r * (int64_t)S;
  if (L <= 0) {
    for (int s = threadIdx.x; s < S; s += kWitThreads) o[s] = -1;
    return;
  }
  const int64_t s_eff = L < S ? L : S;
  const uint64_t occ = row_occupancy(ids + r * (int64_t)topk, topk, L, S, s_eff, red);
  for (int s = threadIdx.x; s < S; s += kWitThreads) {
    int32_t v = -1;
    if (s < s_eff && !((occ >> s) & 1ull)) v = (int32_t)(((int64_t)s * L + s_eff - 1) / s_eff);
    o[s] = v;
  }
}

cudaError_t launch_witness_merge(int32_t* ids, int64_t rows, int topk, const int32_t* ctx, int keep, int S, int B,
                                 cudaStream_t st) {
  witness_merge_kernel<<<(unsigned)rows, kWitThreads, 0, st>>>(ids, rows, topk, ctx, keep, S, B);
  return cudaGetLastError();
}

cudaError_t launch_witness_indices(const int32_t* ids, int64_t rows, int topk, const int32_t* ctx, int S,
                                   int32_t* out, cudaStream_t st) {
  witness_indices_kernel<<<(unsigned)rows, kWitThreads, 0, st>>>(ids, rows, topk, ctx, S, out);
  return cudaGetLastError();
}

}  // namespace idx
