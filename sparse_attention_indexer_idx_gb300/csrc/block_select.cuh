// Block geometry of MiniMax-M3 block-sparse selection ("ferrox_core/block_sparse.rs":
// causal_blocks, block_sparse_select, select_for_head) and the packed fp32
// helpers shared by the CUDA-core and tensor-core block-selection routes.
#pragma once

#include "internal.h"

namespace idx {

struct BlockGeom {
  int64_t n_blocks;
  int64_t n_forced;
  int64_t budget;
  bool scoring;  // false when the forced blocks already decide the selection
};

__device__ __forceinline__ BlockGeom block_geom(int64_t pos, int64_t L, const block_sparse_config& c) {
  BlockGeom g{0, 0, 0, false};
  if (c.block_size <= 0 || pos < 0) return g;
  int64_t causal = pos / c.block_size + 1;
  int64_t exist = (L + c.block_size - 1) / c.block_size;
  g.n_blocks = causal < exist ? causal : exist;
  const int64_t n = g.n_blocks;
  int64_t a = c.init_blocks < n ? c.init_blocks : n;              // [0, a) forced
  int64_t z = n - c.local_blocks;                                  // [max(z,0), n) forced
  z = z < 0 ? 0 : z;
  int64_t overlap = a > z ? a - z : 0;
  g.n_forced = a + (n - z) - overlap;
  g.budget = c.top_blocks > g.n_forced ? c.top_blocks : g.n_forced;
  g.scoring = !(g.n_forced >= g.budget || g.n_forced == n);
  return g;
}

__device__ __forceinline__ bool block_forced(int64_t b, int64_t n, const block_sparse_config& c) {
  int64_t z = n - c.local_blocks;
  return b < c.init_blocks || b >= (z < 0 ? 0 : z);
}

// Packed fp32 multiply: each half is the scalar IEEE product, rounded on its own.
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// acc + p, each half by a scalar rounded add.  A packed multiply feeding a
// packed add comes out of code generation as one packed fused multiply-add
// (measured: the same bits as an fma chain, with the rn modifiers, with
// contraction switched off, and with the product written as fma(a, b, -0)),
// which is not the page's order; with the adds scalar, every product and every
// sum is rounded on its own (measured bit-identical to the sequential fp32 sum).
__device__ __forceinline__ uint64_t f2_add_halves(uint64_t acc, uint64_t p) {
  float a0, a1, p0, p1;
  f2_unpack(acc, &a0, &a1);
  f2_unpack(p, &p0, &p1);
  return f2_pack(__fadd_rn(a0, p0), __fadd_rn(a1, p1));
}
__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((uint64_t)hi << 32) | lo;
}

}  // namespace idx
