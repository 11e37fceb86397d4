// Segment-witness covering pass ("Segment Witnesses": sections "Object" and
// "Implementation rule and contracts").
//
// One warp per row.  Occupancy is a 64-bit mask (S <= 64, as the fused kernel
// of the source pull request carries it): every lane ORs the segments of its
// strided share of the row, then the mask is OR-reduced over the warp.  Lane s
// (two rounds of 32 lanes for S up to 64) then knows whether segment s is a
// witness and, from a popcount of the lower unoccupied segments, which slot it
// goes to.  The row is read once (coalesced int32) and at most B slots are
// written, so the kernel moves topk*4 bytes per row plus the witnesses.
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

// Occupied-segment mask of one row (entries x >= 0 mark min(x*S_eff/L, S-1)).
__device__ __forceinline__ uint64_t row_occupancy(const int32_t* row, int topk, int64_t L, int S, int64_t s_eff) {
  uint64_t m = 0;
  const int lane = threadIdx.x & 31;
  for (int i = lane; i < topk; i += 32) {
    int64_t x = row[i];
    if (x < 0) continue;
    int64_t seg = (x * s_eff) / L;
    if (seg > S - 1) seg = S - 1;
    m |= 1ull << seg;
  }
  return warp_or64(m);
}

__global__ void witness_merge_kernel(int32_t* __restrict__ ids, int64_t rows, int topk,
                                     const int32_t* __restrict__ ctx, int keep, int S, int B) {
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int lane = threadIdx.x & 31;
  const int64_t L = ctx[r];
  if (L <= 0) return;                               // fallback: no witnesses
  const int64_t s_eff = L < S ? L : S;
  int32_t* row = ids + r * (int64_t)topk;
  const uint64_t occ = row_occupancy(row, topk, L, S, s_eff);
  const uint64_t part = (s_eff >= 64) ? ~0ull : ((1ull << s_eff) - 1ull);
  const uint64_t missing = ~occ & part;
  __syncwarp();                                      // every lane has read the row
#pragma unroll
  for (int round = 0; round < 2; ++round) {
    const int s = lane + 32 * round;
    if (s < s_eff && ((missing >> s) & 1ull)) {
      const uint64_t below = (s == 0) ? 0ull : (missing & ((1ull << s) - 1ull));
      const int rank = __popcll(below);
      if (rank < B) {
        const int64_t e = ((int64_t)s * L + s_eff - 1) / s_eff;   // ceil(s L / S_eff)
        row[keep + rank] = (int32_t)e;
      }
    }
  }
}

__global__ void witness_indices_kernel(const int32_t* __restrict__ ids, int64_t rows, int topk,
                                       const int32_t* __restrict__ ctx, int S, int32_t* __restrict__ out) {
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int lane = threadIdx.x & 31;
  const int64_t L = ctx[r];
  int32_t* o = out + r * (int64_t)S;
  if (L <= 0) {
    for (int s = lane; s < S; s += 32) o[s] = -1;
    return;
  }
  const int64_t s_eff = L < S ? L : S;
  const uint64_t occ = row_occupancy(ids + r * (int64_t)topk, topk, L, S, s_eff);
  for (int s = lane; s < S; s += 32) {
    int32_t v = -1;
    if (s < s_eff && !((occ >> s) & 1ull)) v = (int32_t)(((int64_t)s * L + s_eff - 1) / s_eff);
    o[s] = v;
  }
}

cudaError_t launch_witness_merge(int32_t* ids, int64_t rows, int topk, const int32_t* ctx, int keep, int S, int B,
                                 cudaStream_t st) {
  const int warps = 8;
  const int64_t grid = (rows + warps - 1) / warps;
  witness_merge_kernel<<<(unsigned)grid, warps * 32, 0, st>>>(ids, rows, topk, ctx, keep, S, B);
  return cudaGetLastError();
}

cudaError_t launch_witness_indices(const int32_t* ids, int64_t rows, int topk, const int32_t* ctx, int S,
                                   int32_t* out, cudaStream_t st) {
  const int warps = 8;
  const int64_t grid = (rows + warps - 1) / warps;
  witness_indices_kernel<<<(unsigned)grid, warps * 32, 0, st>>>(ids, rows, topk, ctx, S, out);
  return cudaGetLastError();
}

}  // namespace idx
