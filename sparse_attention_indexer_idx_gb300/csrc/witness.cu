// Segment-witness covering pass ("Segment Witnesses": sections "Object" and
// "Implementation rule and contracts").
//
// One warp per row (eight rows per thread block) when there are enough rows to
// fill the GPU, else one whole block (eight warps) per row.  Occupancy is a
// 64-bit mask (S <= 64, as the fused kernel of the source pull request carries
// it): every lane ORs the segments of its share of the row -- 16-byte loads,
// all issued before any is used -- a butterfly of shuffles combines the lanes'
// masks and, with a block per row, shared memory and one barrier combine the
// warps'.  That combine is also the point after which every entry has been
// read, so the in-place writes that follow cannot be seen by a read.  Lane l
// of the row's first warp then handles segments l and l + 32: whether it is a
// witness and, from a popcount of the lower unoccupied segments, which slot it
// goes to.  The row is read once and at most B slots are written.
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

// Segment of an entry x >= 0: for x < L, sigma(x) = floor(x S_eff / L), from
// a float estimate (relative error a few 2^-24, so off by at most one for
// values below 64) corrected once against the exact 64-bit remainder
// x S_eff - q L; entries x >= L mark min(floor(x S_eff / L), S - 1): S - 1
// when S_eff = S, else (S_eff = L) min(x, S - 1).
__device__ __forceinline__ int segment_of(int32_t x, int64_t L, int S, int64_t s_eff, float ratio) {
  if ((int64_t)x >= L) return s_eff == S ? S - 1 : (x < S - 1 ? (int)x : S - 1);
  int q = (int)((float)x * ratio);
  q = q < (int)s_eff - 1 ? q : (int)s_eff - 1;
  const int64_t r = (int64_t)x * s_eff - (int64_t)q * L;
  if (r < 0) --q;
  else if (r >= L) ++q;
  return q;
}

constexpr int kWitRows = 8;       // rows (warps) per thread block
constexpr int kWitVec = 8;        // 16-byte loads per lane and round (in flight together)

// Occupied-segment mask of the entries of one row that thread t of the row's
// NT threads reads (entries x >= 0 mark their segment), OR-combined over the
// warp.  vec4: the row starts 16-byte aligned and topk is a multiple of 4.
template <int NT>
__device__ __forceinline__ uint64_t warp_row_occupancy(const int32_t* row, int topk, int64_t L, int S, int64_t s_eff,
                                                       bool vec4, int t) {
  const float ratio = (float)s_eff / (float)L;
  uint64_t m = 0;
  auto mark = [&](int32_t x) {
    if (x >= 0) m |= 1ull << segment_of(x, L, S, s_eff, ratio);
  };
  if (vec4) {
    const int4* r4 = reinterpret_cast<const int4*>(row);
    const int n4 = topk >> 2;
    for (int j0 = 0; j0 < n4; j0 += NT * kWitVec) {
      int4 v[kWitVec];
#pragma unroll
      for (int u = 0; u < kWitVec; ++u) {
        const int j = j0 + u * NT + t;
        v[u] = j < n4 ? r4[j] : make_int4(-1, -1, -1, -1);
      }
#pragma unroll
      for (int u = 0; u < kWitVec; ++u) {
        mark(v[u].x);
        mark(v[u].y);
        mark(v[u].z);
        mark(v[u].w);
      }
    }
  } else {
    for (int i0 = 0; i0 < topk; i0 += NT * kWitVec) {
      int32_t v[kWitVec];
#pragma unroll
      for (int u = 0; u < kWitVec; ++u) {
        const int i = i0 + u * NT + t;
        v[u] = i < topk ? row[i] : -1;
      }
#pragma unroll
      for (int u = 0; u < kWitVec; ++u) mark(v[u]);
    }
  }
  return warp_or64(m);
}

// Rows handled by one block of 8 warps: WPR warps per row (1 or 8).  Every
// warp returns or stays with its row as a whole; with WPR = 8 the block is one
// row, so the barrier below is reached by all or none of its threads.
template <int WPR>
__device__ __forceinline__ bool witness_row(const int32_t* ids, int64_t rows, int topk, const int32_t* ctx, int S,
                                            int vec4, int64_t* r_out, int64_t* L_out, int64_t* s_eff_out,
                                            uint64_t* occ_out) {
  __shared__ uint64_t red[kWitRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (kWitRows / WPR) + warp / WPR;
  if (r >= rows) return false;
  const int64_t L = ctx[r];
  if (L <= 0) return false;                         // fallback: no witnesses (uniform over the row)
  const int64_t s_eff = L < S ? L : S;
  const int t = (warp % WPR) * 32 + lane;           // this thread within the row
  uint64_t occ = warp_row_occupancy<32 * WPR>(ids + r * (int64_t)topk, topk, L, S, s_eff, vec4 != 0, t);
  if (WPR > 1) {
    if (lane == 0) red[warp] = occ;
    __syncthreads();
    occ = 0;
#pragma unroll
    for (int w = 0; w < WPR; ++w) occ |= red[w];
    if (warp != 0) return false;                    // the first warp writes
  }
  *r_out = r;
  *L_out = L;
  *s_eff_out = s_eff;
  *occ_out = occ;
  return true;
}

template <int WPR>
__global__ void __launch_bounds__(32 * kWitRows) witness_merge_kernel(int32_t* __restrict__ ids, int64_t rows,
                                                                       int topk, const int32_t* __restrict__ ctx,
                                                                       int keep, int S, int B, int vec4) {
  int64_t r, L, s_eff;
  uint64_t occ;
  if (!witness_row<WPR>(ids, rows, topk, ctx, S, vec4, &r, &L, &s_eff, &occ)) return;
  int32_t* row = ids + r * (int64_t)topk;
  const uint64_t part = (s_eff >= 64) ? ~0ull : ((1ull << s_eff) - 1ull);
  const uint64_t missing = ~occ & part;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;                    // segments 0..63
    if (s < s_eff && ((missing >> s) & 1ull)) {
      const uint64_t below = (s == 0) ? 0ull : (missing & ((1ull << s) - 1ull));
      const int rank = __popcll(below);
      if (rank < B) row[keep + rank] = (int32_t)(((int64_t)s * L + s_eff - 1) / s_eff);   // ceil(s L / S_eff)
    }
  }
}

template <int WPR>
__global__ void __launch_bounds__(32 * kWitRows) witness_indices_kernel(const int32_t* __restrict__ ids,
                                                                         int64_t rows, int topk,
                                                                         const int32_t* __restrict__ ctx, int S,
                                                                         int32_t* __restrict__ out, int vec4) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rr = (int64_t)blockIdx.x * (kWitRows / WPR) + warp / WPR;
  if (rr < rows && ctx[rr] <= 0) {
    if (warp % WPR == 0)
      for (int s = lane; s < S; s += 32) out[rr * (int64_t)S + s] = -1;
    return;
  }
  int64_t r, L, s_eff;
  uint64_t occ;
  if (!witness_row<WPR>(ids, rows, topk, ctx, S, vec4, &r, &L, &s_eff, &occ)) return;
  int32_t* o = out + r * (int64_t)S;
  for (int s = lane; s < S; s += 32) {
    int32_t v = -1;
    if (s < s_eff && !((occ >> s) & 1ull)) v = (int32_t)(((int64_t)s * L + s_eff - 1) / s_eff);
    o[s] = v;
  }
}

static int witness_vec4(const int32_t* ids, int topk) {
  return (topk % 4 == 0 && (reinterpret_cast<uintptr_t>(ids) & 15) == 0) ? 1 : 0;
}

// A warp per row once the rows fill every SM with a few blocks; a block per row below that.
static bool witness_warp_per_row(int64_t rows) { return rows >= (int64_t)4 * kWitRows * sm_count(); }

cudaError_t launch_witness_merge(int32_t* ids, int64_t rows, int topk, const int32_t* ctx, int keep, int S, int B,
                                 cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int v4 = witness_vec4(ids, topk);
  if (witness_warp_per_row(rows))
    witness_merge_kernel<1><<<(unsigned)((rows + kWitRows - 1) / kWitRows), 32 * kWitRows, 0, st>>>(
        ids, rows, topk, ctx, keep, S, B, v4);
  else
    witness_merge_kernel<kWitRows><<<(unsigned)rows, 32 * kWitRows, 0, st>>>(ids, rows, topk, ctx, keep, S, B, v4);
  return cudaGetLastError();
}

cudaError_t launch_witness_indices(const int32_t* ids, int64_t rows, int topk, const int32_t* ctx, int S,
                                   int32_t* out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int v4 = witness_vec4(ids, topk);
  if (witness_warp_per_row(rows))
    witness_indices_kernel<1><<<(unsigned)((rows + kWitRows - 1) / kWitRows), 32 * kWitRows, 0, st>>>(
        ids, rows, topk, ctx, S, out, v4);
  else
    witness_indices_kernel<kWitRows><<<(unsigned)rows, 32 * kWitRows, 0, st>>>(ids, rows, topk, ctx, S, out, v4);
  return cudaGetLastError();
}

}  // namespace idx
