// Indexer score and DoSA bound on the 5th-generation tensor cores (tcgen05,
// sm_103a), bf16 queries with bf16 keys or FP8 e4m3 keys (+ per-token scale),
// D = 128.
//
// FP8 keys go to the MMA as they are loaded (kind::f8f6f4, e4m3 x e4m3): the
// bf16 query row is split once per query group into two e4m3 vectors with one
// exact power-of-two scale sigma per row, q = sigma (hi + lo) (bf16 holds 8
// significant bits, hi takes the top 4, lo the next 4; only elements below
// 2^-2 sigma lose low bits, by less than 2^-10 sigma); hi and lo are
// separate B rows (N = 2 x vectors, so a key tile takes four MMAs of K = 32)
// and the epilogue forms sigma (acc_hi + acc_lo).  The per-key dequantisation scales travel with the key
// tile (cp.async into a shared ring, completion on the tile's barrier), so the
// epilogue never waits on a global load.
//
// Mapping.  One MMA tile is 128 keys (the M axis: key i of the tile lives in
// TMEM lane i) times N = NQ*NCOL columns (NQ queries x NCOL vectors each, all
// K-major), the full D = 128 as 8 MMAs of K = 16 (bf16) or 4 MMAs of K = 32
// (FP8, with the hi and lo rows of every vector among the N columns).  Each epilogue thread owns
// one key and reduces its own TMEM columns with no shuffles.
//
// Modes:
//  kScore   s(k) = sum_h w_h ReLU(q_h . k) ("DoSA：用安全上界减少 Indexer 的完整
//           打分", section 3), NCOL = H; the head sum is one fused-multiply-add
//           chain h = 0..H-1, so a (query, key) score has the same bits
//           wherever it is computed -- same instruction shape, same K order,
//           same chain.
//  kGather  the same score over per-row key lists: tile t of row m holds the
//           keys list[m][t*128 + i], copied by the producer warp's lanes (16-byte
//           cp.async, four rows per lane) straight into the swizzled tile; each
//           lane waits for its own copies a few tiles later, fences them for the
//           async proxy and arrives on the tile's barrier.  (TMA tile::gather4
//           moves 512 bytes per instruction and its issue rate, not bandwidth,
//           set the pace.)  Used to rescore DoSA candidates; output is indexed
//           by list position.
//  kGroup   the shared candidate stream of the same page (section 4): a group
//           of four consecutive queries over one key sequence and one list of
//           keys (list[g][i], ascending); every key of the list is scored for
//           the four queries in one tile, output indexed by list position
//           (row m = 4g + q: scores[m*ld + i]); which records a row keeps is
//           decided when the rows are merged.
//  kFilter  the dense score of every visible key of a row, kept as (id, score)
//           only when it reaches tau[m] (decode with a prior).
//  kBound   DoSA's safe upper bound (same page, sections 2, 3.1, 3.2): B holds
//           per query R retained head vectors (rows 0..R-1) and the |w|-folded
//           negative aggregate (row 31); the epilogue evaluates
//             U = sum_j w'_j ReLU(q_j . k) + coef ||k|| - ReLU(a . k)
//           (times the FP8 scale), with ||k|| read from the key tile in shared
//           memory (one query per tile) or from a per-key array (shared keys,
//           where every epilogue warp would otherwise redo it), and sets the bit of every visible non-seed key with U >= tau
//           in the row's candidate bitmap (drop only when U < tau): one warp
//           ballot is one 32-key word, stored whole, so the scan needs no atomics.
//
// Work units are (query group g, key tile t).  Shared keys (causal prefill): a
// group is NQ consecutive rows over one key sequence.  Per-row keys (decode,
// gathered lists): a group is one row.  The units are split into one
// contiguous range per CTA (persistent, one CTA per SM), balanced by the exact
// tile count of every group, which a prologue warp scans from the lengths.
//
// Warp roles:  warp 0  TMA producer (key tiles, query tiles)
//              warp 1  TMEM allocation + MMA issue (one thread)
//              warps 2..9 epilogue, two per TMEM lane quarter: they take
//                         alternate queries of a tile (several queries per
//                         tile) or alternate tiles (one query per tile):
//                         tcgen05.ld -> score / bound -> global
//              next       (FP8 only) split of each query group's bf16 rows
//                         into the e4m3 hi and lo tiles; (gathered tiles)
//                         the second producer warp
// Two layouts differ (TcCfg): the bf16 bound over several queries has sixteen
// epilogue warps (warps 2..17; over 16-vector blocks, two sets of eight taking
// alternate units), and the two-query score epilogue with its weights in
// registers has twelve warps, the epilogue being warps 4..11 (WREG).
// One thread issues every tcgen05.mma of the CTA: a build in which a second
// warp issued every other round into the same accumulators gave, in about one
// launch in twenty, a few wrong rows of one tile (repeated launches on the same
// inputs compared bit for bit): the two threads shared the query buffer's
// release barrier, which one thread's commit could complete while the other's
// MMAs still read the buffer.  With a single issuer every repeat is identical.
// Every wait is bounded (see common.cuh); on a timeout all roles stop, the
// producer and the MMA thread drain what they issued, and TMEM is released.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"

namespace idx {

enum TcMode { kScore = 0, kGather = 1, kBound = 2, kFilter = 3, kGroup = 4 };

struct TcArgs {
  idx_problem p;              // p.q is the B source: queries, or prepared vectors (kBound)
  float* scores;
  int64_t ld;
  int64_t G;                  // groups
  // kGather: row m's keys are key_base(m) + list[m*gld + i], i < cnt[m]
  // kGroup: group g's keys are list[g*gld + i], i < cnt[g]
  const int32_t* list;
  const int32_t* cnt;
  int64_t gld;
  // kBound
  const float* wfold;         // [M, 32] folded retained weights (j < R)
  const float* coef;          // [M] c + margin, multiplies ||k||
  const float* tau;           // [M]
  const float* knorm;         // kBound over shared keys: [n_keys] ||k|| (codes for FP8), rounded up
  const uint32_t* seedbits;   // seed bitmap, row stride seed_stride words (0: one shared bitmap)
  int64_t seed_stride;
  uint32_t* candbits;         // kBound: [M, cb_stride] candidate bitmap words
  int64_t cb_stride;
  int32_t* cand;              // kFilter: [M, cap] kept ids
  int32_t* cand_cnt;          // [M]
  int64_t cap;
  int32_t* status;            // [M] bit 1: candidate overflow
  float* cand_sc;             // kFilter: [M, cap] scores of the kept keys (cand: their ids)
  const int32_t* row_mask;    // optional [M]: rows with row_mask[m] == 0 are skipped
  int R;
};

__host__ __device__ constexpr int tc_pow2_cols(int c) {
  return c <= 32 ? 32 : (c <= 64 ? 64 : (c <= 128 ? 128 : (c <= 256 ? 256 : 512)));
}

template <int KDT_, int NCOL_, int NQ_, int MODE_>
struct TcCfg {
  static constexpr int KDT = KDT_;
  static constexpr int NCOL = NCOL_;          // query vectors per query: H (score) or 32 (bound)
  static constexpr int H = NCOL_;
  static constexpr int NQ = NQ_;
  static constexpr int MODE = MODE_;
  static constexpr bool FP8 = (KDT == IDX_FP8_E4M3);
  static constexpr bool GATHER = (MODE == kGather || MODE == kGroup);   // keys fetched by list entries
  static constexpr bool GROUP = (MODE == kGroup);
  static constexpr bool BOUND = (MODE == kBound);
  // kBound: ||k|| from the key tile (one query per tile: one epilogue warp reads a
  // unit) or from the per-key array (several queries per tile)
  static constexpr bool KN_TILE = BOUND && NQ_ == 1;
  static constexpr bool KN_GLOBAL = BOUND && NQ_ > 1;
  static constexpr bool FILTER = (MODE == kFilter);   // scores >= tau[m] appended as (id, score)
  static constexpr int NCOLX = FP8 ? 2 * NCOL : NCOL;   // MMA columns per query (hi, lo for FP8)
  // kBound over shared keys with at most 16 retained heads: per query a block of
  // 16 vectors (retained, zero past R), then one 16-row block holding the
  // group's aggregates (8 used): 144 columns where 8 x 32 would carry 17 terms each
  static constexpr bool AGG16 = (MODE == kBound) && NCOL_ == 16 && !FP8;
  static constexpr int QROWS = NQ * NCOL + (AGG16 ? 16 : 0);   // query-side rows of one group
  static constexpr int N = AGG16 ? QROWS : NQ * NCOLX;
  // 128-key subtiles per work unit: FP8 per-row scoring takes 256 keys (32 KB,
  // one TMA box) per unit, so every barrier round trip, commit and schedule
  // step covers as many key bytes as a bf16 tile
  static constexpr int SUB = (FP8 && (MODE == kScore || MODE == kFilter) && NQ == 1 && N <= 128) ? 2 : 1;
  static constexpr int UKEYS = 128 * SUB;
  static constexpr int A_BYTES = SUB * (FP8 ? 128 * 128 : 128 * 128 * 2);   // one unit of keys
  static constexpr int SUB_BYTES = A_BYTES / SUB;                           // one 128-key subtile
  static constexpr int BQ_BYTES = FP8 ? 0 : QROWS * 256;            // bf16 query rows as loaded
  static constexpr int B8_BYTES = FP8 ? N * 128 : 0;                 // e4m3 hi and lo rows (FP8)
  static constexpr int B_BYTES = BQ_BYTES + B8_BYTES;                // one query buffer
  static constexpr int SB = (NQ > 1) ? 1 : 2;
  static constexpr int SACC = (SUB * N >= 256) ? 2 : (4 * SUB * N <= 512 ? 4 : 3);
  // TMEM columns between accumulator stages (AGG16: 144 rounded up to 160)
  static constexpr int ACC_STRIDE = AGG16 ? 160 : SUB * N;
  // FP8: key scales of one tile; their ring is deeper than the key ring by the
  // tiles that can sit between the MMA and the epilogue, so a key slot is free
  // as soon as its MMAs complete
  static constexpr int SC_BYTES = FP8 ? 512 * SUB : 0;
  static constexpr int SA_FIT = (220 * 1024 - SB * B_BYTES - (SACC + 2) * SC_BYTES) / (A_BYTES + SC_BYTES);
  static constexpr int SA = FP8 ? (SA_FIT > 12 ? 12 : SA_FIT) : ((BQ_BYTES * SB <= 32768) ? 5 : 4);
  static constexpr int SSC = FP8 ? SA + SACC + 2 : 0;
  static constexpr int SSC_MOD = SSC > 0 ? SSC : 1;
  static constexpr int IL = (SUB == 1 && N <= 128) ? 2 : 1;   // units whose MMA chains are interleaved
  static constexpr int TMEM_COLS = tc_pow2_cols(SACC * ACC_STRIDE);
  // epilogue warps, two per TMEM lane quarter (four for the bf16 bound over
  // several queries, whose dependent chains leave two warps per quarter idle)
  static constexpr int NE = (MODE == kBound && NQ_ > 1 && KDT_ != IDX_FP8_E4M3) ? 16 : 8;
  // bf16 score tiles with at least 4 queries: an epilogue warp walks its queries
  // two at a time, both chains in one packed fma.rn.f32x2 per head
  static constexpr bool PAIR = (MODE != kBound) && (MODE != kFilter) && !FP8 && NQ >= 4;
  // the bound over 16-vector blocks keeps the folded weights of its warp's
  // queries the same way, a pair's (w_a[j], w_b[j]) adjacent, for packed chains
  static constexpr bool BPAIR = AGG16 && NQ == 8;
  // epilogue warps in two sets that take alternate units: one query per unit
  // (each set one warp per lane quarter), and the bound over 16-vector blocks
  // (each set two warps per quarter, four rows each), where one warp's
  // dependent chain from the TMEM load to the bitmap store would otherwise
  // set the pace of every unit
  static constexpr bool ALT = (NQ == 1 && SUB == 1) || (BPAIR && NE == 16);
  // epilogue warps that read one unit: half of them with alternate units, else
  // all (several queries per unit, alternating queries, or two subtiles, one
  // warp of a quarter per subtile)
  static constexpr int EPT = ALT ? NE / 2 : NE;
  static constexpr int NCONV = FP8 ? 1 : 0;   // warp that splits the query rows (FP8)
  // producer warps: gathered tiles take two (two tile rows per lane: the copies
  // of one warp alone could not keep the tensor core fed; a third or fourth
  // warp would cut the registers per thread below what the epilogue needs),
  // TMA tiles one
  static constexpr int NP = GATHER ? 2 : 1;
  static constexpr int RPL = 4 / NP;          // tile rows per producer lane
  // Two-query epilogue with its weights in registers: 2 x H per warp query pair
  // (128 for H = 64), read from shared memory in every unit they took more of its
  // bandwidth than the tensor core's operands.  The block then has twelve warps:
  // warpgroup 0 holds the producer (warp 0), the MMA thread (warp 1), the second
  // gather producer (warp 2) and an idle warp, and gives registers to the two
  // epilogue warpgroups (warps 4..11) with setmaxnreg: 80 each against 208.
  static constexpr bool WREG = PAIR;
  static constexpr int EPI0 = WREG ? 4 : 2;                  // first epilogue warp
  static constexpr int PROD1 = WREG ? 2 : 2 + NE + NCONV;    // second producer warp (NP = 2)
  static constexpr int NTHREADS = WREG ? 32 * 12 : 32 * (2 + NE + NCONV + (NP - 1));
  static constexpr int WG0_REGS = 80, EPI_REGS = 208;        // after setmaxnreg (WREG)
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + SA * A_BYTES;
  // per epilogue warp (NE private copies, so the warps never wait on each other)
  static constexpr int OFF_SC = OFF_B + SB * B_BYTES;
  static constexpr int OFF_W = OFF_SC + SSC * SC_BYTES;
  static constexpr int OFF_BASE = OFF_W + NE * NQ * NCOL * 4;
  static constexpr int OFF_LEN = OFF_BASE + NE * NQ * 8;
  static constexpr int OFF_AUX = OFF_LEN + NE * NQ * 4;        // coef, tau, sigma per query
  // FP8: ring of the per-query scales sigma, split warps -> epilogue, deeper
  // than the groups that can lie between them (SB + SACC + 1)
  static constexpr int SIGR = FP8 ? 8 : 0;
  static constexpr int SIGR_MOD = SIGR > 0 ? SIGR : 1;
  static constexpr int OFF_SIG = OFF_AUX + NE * NQ * 16;
  static constexpr int OFF_BAR = ((OFF_SIG + SIGR * NQ * 4) + 7) & ~7;
  static constexpr int NBARS = 2 * SA + 2 * SB + 2 * SACC + 1 + 2 * SIGR + 2 * SSC;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;   // + alignment slack
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "MMA N");
  static_assert(MODE != kFilter || NQ == 1, "kFilter: one query per group");
  static_assert(SACC * ACC_STRIDE <= 512, "TMEM columns");
  static_assert(!WREG || (NE == 8 && NP <= 2 && NCONV == 0), "register-weight layout: warpgroups 0, 1, 2");
  static_assert(!BPAIR || (ALT && SUB == 1 && SACC >= 2), "bound over 16-vector blocks: every other unit, one subtile");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct TcSched {
  int64_t g0;       // first group
  int64_t t0;       // first tile in it
  int64_t count;    // units in this CTA's range
};

// ------------------------------------------------------------ group helpers --
template <class C>
__device__ __forceinline__ int64_t tc_group_tiles(const TcArgs& A, int64_t g, bool report = false) {
  if (C::GATHER) {
    if (!C::GROUP && A.row_mask && !A.row_mask[g]) return 0;
    const int32_t c = A.cnt[g];
    return c > 0 ? (c + 127) / 128 : 0;
  }
  int mx = 0;
#pragma unroll 1
  for (int q = 0; q < C::NQ; ++q) {
    int64_t m = g * C::NQ + q;
    if (m >= A.p.M) break;
    int64_t off;
    int len;
    if (!row_extent(A.p, m, &off, &len) && report) atomicOr(&g_device_error, DEVERR_BAD_ROW);
    if (A.row_mask && !A.row_mask[m]) len = 0;
    mx = len > mx ? len : mx;
  }
  return (mx + C::UKEYS - 1) / C::UKEYS;
}

__device__ __forceinline__ int64_t warp_incl_scan(int64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int64_t u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// One warp: total units, this CTA's [start, end), and its first (g, t).
template <class C>
__device__ void tc_schedule(const TcArgs& A, TcSched* out) {
  const int lane = threadIdx.x & 31;
  int64_t total = 0;
  for (int64_t b = 0; b < A.G; b += 32) {
    int64_t g = b + lane;
    int64_t t = g < A.G ? tc_group_tiles<C>(A, g, blockIdx.x == 0) : 0;
    total += __shfl_sync(0xffffffffu, warp_incl_scan(t), 31);
  }
  const int64_t start = total * (int64_t)blockIdx.x / gridDim.x;
  const int64_t end = total * (int64_t)(blockIdx.x + 1) / gridDim.x;
  int64_t g0 = 0, t0 = 0;
  if (end > start) {
    int64_t run = 0;
    for (int64_t b = 0; b < A.G; b += 32) {
      int64_t g = b + lane;
      int64_t t = g < A.G ? tc_group_tiles<C>(A, g) : 0;
      int64_t incl = warp_incl_scan(t);
      int64_t chunk = __shfl_sync(0xffffffffu, incl, 31);
      if (run + chunk > start) {
        unsigned hit = __ballot_sync(0xffffffffu, run + incl > start);
        int first = __ffs(hit) - 1;
        int64_t incl_f = __shfl_sync(0xffffffffu, incl, first);
        int64_t t_f = __shfl_sync(0xffffffffu, t, first);
        g0 = b + first;
        t0 = start - (run + incl_f - t_f);
        break;
      }
      run += chunk;
    }
  }
  if (lane == 0) {
    out->g0 = g0;
    out->t0 = t0;
    out->count = end - start;
  }
}

// Walks this CTA's units in order.
template <class C>
struct TcUnits {
  const TcArgs* A;
  int64_t g, t, left, tiles_g;
  __device__ void init(const TcArgs& a, const TcSched& s) {
    A = &a;
    g = s.g0;
    t = s.t0;
    left = s.count;
    tiles_g = left > 0 ? tc_group_tiles<C>(a, g) : 0;
  }
  __device__ bool valid() const { return left > 0; }
  __device__ void advance() {
    --left;
    if (left <= 0) return;
    ++t;
    while (t >= tiles_g) {
      ++g;
      t = 0;
      tiles_g = tc_group_tiles<C>(*A, g);
    }
  }
};

// Key-row base of row m's key sequence (per-row keys: key_off, else 0).
__device__ __forceinline__ int64_t tc_key_base(const TcArgs& A, int64_t m) {
  if (!A.p.key_off) return 0;
  int64_t off;
  int len;
  row_extent(A.p, m, &off, &len);
  return off;
}

// ----------------------------------------------------------- FP8 helpers ---
// Power-of-two scale of a query row: max|q| / sigma lies in [128, 256).
__device__ __forceinline__ void row_sigma(float amax, float* sigma, float* inv) {
  if (!(amax > 0.0f)) {
    *sigma = 1.0f;
    *inv = 1.0f;
    return;
  }
  int ex;
  frexpf(amax, &ex);                      // amax = f 2^ex, f in [0.5, 1)
  *sigma = ldexpf(1.0f, ex - 8);
  *inv = ldexpf(1.0f, 8 - ex);
}

// Two floats -> two e4m3 codes (round to nearest even, saturating), x0 in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}
// Two e4m3 codes (low byte first) -> two floats, exactly.
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t codes, float* lo, float* hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)(codes & 0xffffu)));
  const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
  *lo = __low2float(hv);
  *hi = __high2float(hv);
}

// max |q| over a query's NCOL rows of 128 bf16 values (global memory): the
// epilogue's copy of the value the split used.
template <int NCOL>
__device__ __forceinline__ float query_amax(const uint16_t* q) {
  const int lane = threadIdx.x & 31;
  float mx = 0.0f;
  // 16-byte loads, eight in flight per lane
#pragma unroll 8
  for (int i = lane; i < NCOL * 16; i += 32) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(q) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mx = fmaxf(mx, fabsf(__uint_as_float(w[e] << 16)));
      mx = fmaxf(mx, fabsf(__uint_as_float(w[e] & 0xffff0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  return mx;
}

// Warp-collective: the lanes with keep set append (id, val) to row m's list
// (one atomic per warp); a list that would pass cap sets status bit 2.
__device__ __forceinline__ void tc_append(const TcArgs& A, int64_t m, bool keep, int32_t id, float val) {
  const int lane = threadIdx.x & 31;
  const unsigned mask = __ballot_sync(0xffffffffu, keep);
  if (!mask) return;
  int32_t basepos = 0;
  if (lane == 0) basepos = atomicAdd(&A.cand_cnt[m], __popc(mask));
  basepos = __shfl_sync(0xffffffffu, basepos, 0);
  if (lane == 0 && basepos + __popc(mask) > A.cap) atomicOr(&A.status[m], 2);
  if (keep) {
    const int64_t pos = basepos + __popc(mask & ((1u << lane) - 1u));
    if (pos < A.cap) {
      A.cand[m * A.cap + pos] = id;
      A.cand_sc[m * A.cap + pos] = val;
    }
  }
}

// ------------------------------------------------------------- the kernel ---
template <class C>
__global__ void __launch_bounds__(C::NTHREADS, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                    const TcArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* sA = smem + C::OFF_A;
  uint8_t* sB = smem + C::OFF_B;
  float* sScale = reinterpret_cast<float*>(smem + C::OFF_SC);
  float* sW_all = reinterpret_cast<float*>(smem + C::OFF_W);
  int32_t* sLen_all = reinterpret_cast<int32_t*>(smem + C::OFF_LEN);
  int64_t* sBase_all = reinterpret_cast<int64_t*>(smem + C::OFF_BASE);
  float* sAux_all = reinterpret_cast<float*>(smem + C::OFF_AUX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* a_full = bars;
  uint64_t* a_empty = a_full + C::SA;
  uint64_t* b_full = a_empty + C::SA;
  uint64_t* b_empty = b_full + C::SB;
  uint64_t* acc_full = b_empty + C::SB;
  uint64_t* acc_empty = acc_full + C::SACC;
  uint64_t* drain_bar = acc_empty + C::SACC;   // the MMA thread's last commit
  uint64_t* sig_full = drain_bar + 1;
  uint64_t* sig_empty = sig_full + C::SIGR;
  float* sSig = reinterpret_cast<float*>(smem + C::OFF_SIG);
  uint64_t* sc_full = sig_empty + C::SIGR;
  uint64_t* sc_empty = sc_full + C::SSC;
  uint8_t* misc = smem + C::OFF_MISC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  TcSched* sched = reinterpret_cast<TcSched*>(misc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::SA; ++i) {
      mbar_init(&a_full[i], C::GATHER ? 32 * C::NP : 1);   // gathered: every producer lane arrives
      // the bound epilogue reads ||k|| from the key tile, so its warps also release the slot
      mbar_init(&a_empty[i], C::KN_TILE ? 1 + C::EPT : 1);
    }
    for (int i = 0; i < C::SB; ++i) {
      // FP8: every lane of the split warps arrives once its rows are written
      mbar_init(&b_full[i], C::FP8 ? 32 * C::NCONV : 1);
      mbar_init(&b_empty[i], 1);                 // the MMA-issuing thread
    }
    for (int i = 0; i < C::SACC; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], C::EPT);          // one arrival per epilogue warp that read the stage
    }
    mbar_init(&drain_bar[0], 1);
    for (int i = 0; i < C::SIGR; ++i) {
      mbar_init(&sig_full[i], 1);
      mbar_init(&sig_empty[i], C::NE);
    }
    for (int i = 0; i < C::SSC; ++i) {
      mbar_init(&sc_full[i], 32 * C::NP);       // each producer lane, once its copies landed
      mbar_init(&sc_empty[i], C::EPT);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_q);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  if (warp == 2) tc_schedule<C>(args, sched);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const TcSched s = *sched;
  if constexpr (C::WREG) {
    // the launch's registers (checked on the host: 168 a thread) move from
    // warpgroup 0 to the epilogue warpgroups (their increase opens the epilogue
    // branch, so that the compiler allocates that code for it); each warpgroup
    // executes its instruction together
    if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::WG0_REGS) : "memory");
  }

  if (warp == 0 || (C::NP > 1 && warp == C::PROD1)) {
    // ------------------------------------------------------------ producer
    // producer warp pidx (warp 0 is producer 0, the only one that loads query
    // tiles) copies tile rows RPL (32 pidx + lane) .. + RPL - 1
    const int pidx = warp == 0 ? 0 : 1;
    const int rbase = C::RPL * (32 * pidx + lane);
    TcUnits<C> u;
    u.init(args, s);
    int64_t cur_g = -1;
    int64_t gbase = 0;                         // first key row of the group (kept: no global load per tile)
    int32_t gcnt = 0;                          // kGather: list length of the group
    // kGather: this lane's four list entries of the next unit, loaded one unit
    // ahead so that the list read overlaps the previous unit's gather
    int32_t pf[C::RPL];
#pragma unroll
    for (int i = 0; i < C::RPL; ++i) pf[i] = 0;
    int64_t pf_g = -1, pf_t = -1;
    uint32_t na = 0, nb = 0;
    // Gathered tiles: every producer lane arrives on the tile's barrier through
    // cp.async.mbarrier.arrive.noinc, which fires once that lane's copies have
    // landed, so the producer never waits for its own copies; the MMA thread
    // fences the async proxy after the barrier and before its MMAs read the tile.
    while (u.valid()) {
      if (u.g != cur_g) {
        cur_g = u.g;
        gbase = tc_key_base(args, cur_g);
        if (C::GATHER) gcnt = args.cnt[cur_g];
        if (!C::FP8 && pidx == 0) {
          // bf16: the group's query rows (FP8: the split warps read them from global memory)
          const int bs = nb % C::SB;
          bool ok = true;
          if (lane == 0) {
            ok = mbar_wait(&b_empty[bs], ((nb / C::SB) & 1) ^ 1, abort_flag);
            if (ok) {
              uint64_t* bar = &b_full[bs];
              mbar_arrive_expect_tx(bar, C::BQ_BYTES);
              const int32_t y = (int32_t)(cur_g * C::QROWS);
              tma_load_2d(sB + bs * C::B_BYTES, &tmap_q, bar, 0, y);
              tma_load_2d(sB + bs * C::B_BYTES + C::BQ_BYTES / 2, &tmap_q, bar, 64, y);
            }
          }
          if (!__shfl_sync(0xffffffffu, ok, 0)) break;
          ++nb;
        }
      }
      const int as = na % C::SA;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&a_empty[as], ((na / C::SA) & 1) ^ 1, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t* dst = sA + as * C::A_BYTES;
      uint64_t* fbar = &a_full[as];
      int32_t graw[C::RPL];   // gathered: list entries of this lane's tile rows rbase .. rbase + RPL - 1
#pragma unroll
      for (int i = 0; i < C::RPL; ++i) graw[i] = 0;
      if (C::GATHER) {
        if (pf_g == u.g && pf_t == u.t) {
#pragma unroll
          for (int i = 0; i < C::RPL; ++i) graw[i] = pf[i];
        } else {
          const int32_t* lst = args.list + u.g * args.gld + u.t * 128;
#pragma unroll
          for (int i = 0; i < C::RPL; ++i) graw[i] = (int)(u.t * 128) + rbase + i < gcnt ? lst[rbase + i] : 0;
        }
      }
      if constexpr (C::FP8) {
        // key scales: lane l copies those of tile rows 4l..4l+3 (rows clamped into
        // the buffer; a scale past the row's end is never used)
        const int ss = na % C::SSC_MOD;
        bool sok = true;
        if (lane == 0) sok = mbar_wait(&sc_empty[ss], ((na / C::SSC_MOD) & 1) ^ 1, abort_flag);
        if (!__shfl_sync(0xffffffffu, sok, 0)) break;
        float* sdst = sScale + ss * C::UKEYS + rbase;
#pragma unroll
        for (int i = 0; i < C::RPL * C::SUB; ++i) {
          const int pos = (int)(u.t * C::UKEYS) + 128 * (i / C::RPL) + rbase + (i % C::RPL);
          int64_t row = gbase + pos;
          if (C::GATHER) row = gbase + (int64_t)graw[i % C::RPL];
          row = row < 0 ? 0 : (row >= args.p.n_keys ? args.p.n_keys - 1 : row);
          cp_async_4(sdst + 128 * (i / C::RPL) + (i % C::RPL), args.p.key_scale + row);
        }
        cp_async_arrive_noinc(&sc_full[ss]);
      }
      if (C::GATHER) {
        // this lane's tile rows (list positions t*128 + r), 16 bytes at a time, into
        // the 128-byte-swizzled halves; rows past the list are left as they are
        // (their accumulator rows are never read)
        constexpr int RB = C::FP8 ? 128 : 256;   // bytes of one key row
        const char* kb = static_cast<const char*>(args.p.keys);
#pragma unroll
        for (int i = 0; i < C::RPL; ++i) {
          const int r = rbase + i;
          if ((int)(u.t * 128) + r >= gcnt) continue;
          int64_t row = gbase + (int64_t)graw[i];
          row = row < 0 ? 0 : (row >= args.p.n_keys ? args.p.n_keys - 1 : row);
          const char* src = kb + row * RB;
#pragma unroll
          for (int cc = 0; cc < RB / 16; ++cc)
            cp_async_16(dst + (cc >> 3) * (C::A_BYTES / 2) + r * 128 + (((cc & 7) ^ (r & 7)) << 4), src + cc * 16);
        }
        cp_async_arrive_noinc(fbar);            // counts this lane in once its copies landed
        // the next unit's entries
        TcUnits<C> nx = u;
        nx.advance();
        if (nx.valid()) {
          const int32_t cn = nx.g == u.g ? gcnt : args.cnt[nx.g];
          const int32_t* l2 = args.list + nx.g * args.gld + nx.t * 128;
#pragma unroll
          for (int i = 0; i < C::RPL; ++i) pf[i] = (int)(nx.t * 128) + rbase + i < cn ? l2[rbase + i] : 0;
          pf_g = nx.g;
          pf_t = nx.t;
        }
      } else if (lane == 0 && pidx == 0) {
        const int32_t y = (int32_t)(gbase + u.t * C::UKEYS);
        mbar_arrive_expect_tx(fbar, C::A_BYTES);
        tma_load_2d(dst, &tmap_k, fbar, 0, y);
        if (!C::FP8) tma_load_2d(dst + C::A_BYTES / 2, &tmap_k, fbar, 64, y);
      }
      __syncwarp();
      ++na;
      u.advance();
    }
    // drain: the last phase issued on every ring slot has landed
    if (C::FP8 || C::GATHER) asm volatile("cp.async.wait_all;" ::: "memory");
    if (lane == 0 && pidx == 0) {
      for (uint32_t i = 0; i < (uint32_t)C::SB && i < nb; ++i) {
        uint32_t j = nb - 1 - i;
        mbar_wait_drain(&b_full[j % C::SB], (j / C::SB) & 1);
      }
      for (uint32_t i = 0; i < (uint32_t)C::SA && i < na; ++i) {
        uint32_t j = na - 1 - i;
        mbar_wait_drain(&a_full[j % C::SA], (j / C::SA) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint64_t descA0 = smem_desc_sw128(smem_u32(sA)), descB0 = smem_desc_sw128(smem_u32(sB));
      TcUnits<C> u;
      u.init(args, s);
      int64_t cur_g = -1;
      int cur_bs = 0;
      uint32_t na = 0, nb = 0, nacc = 0;
      if constexpr (C::IL == 1 && C::SUB == 1) {
        // One unit per step: ring slots and accumulator stages as 32-bit counters
        // with their phase bits, the (group, tile) walk of TcUnits inline, one
        // descriptor add per operand and unit -- the issuing thread's own work
        // between two units is what the tensor core waits for.
        uint32_t slot = 0, a_ph = 0, st = 0, e_ph = 1;
        int64_t g = u.g, t = u.t, left = u.left, tiles_g = u.tiles_g;
        while (left > 0) {
          if (g != cur_g) {
            cur_g = g;
            cur_bs = nb % C::SB;
            if (!mbar_wait(&b_full[cur_bs], (nb / C::SB) & 1, abort_flag)) break;
            ++nb;
          }
          if (!mbar_wait(&a_full[slot], a_ph, abort_flag)) break;
          if (!mbar_wait(&acc_empty[st], e_ph, abort_flag)) break;
          tc_fence_after();
          // gathered tiles were written through the generic proxy (cp.async)
          if (C::GATHER) fence_proxy_async_smem();
          const uint64_t adesc = descA0 + (uint64_t)((slot * (uint32_t)C::A_BYTES) >> 4);
          const uint64_t bdesc = descB0 + (uint64_t)((cur_bs * C::B_BYTES) >> 4);
          const uint32_t d = tmem_base + st * (uint32_t)C::ACC_STRIDE;
          if constexpr (C::FP8) {
            constexpr uint32_t idesc = idesc_f16(128, C::N, 0u);
            const uint64_t b8 = bdesc + (uint64_t)(C::BQ_BYTES >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_f8(d, adesc + (uint64_t)(2 * k), b8 + (uint64_t)(2 * k), idesc, k > 0 ? 1u : 0u);
          } else {
            constexpr uint32_t idesc = idesc_f16(128, C::N, 1u);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t ao = (uint64_t)(((k >> 2) * (C::A_BYTES / 2) + (k & 3) * 32) >> 4);
              const uint64_t bo = (uint64_t)(((k >> 2) * (C::BQ_BYTES / 2) + (k & 3) * 32) >> 4);
              tc_mma_f16(d, adesc + ao, bdesc + bo, idesc, k > 0 ? 1u : 0u);
            }
          }
          tc_commit(&a_empty[slot]);
          tc_commit(&acc_full[st]);
          ++na;
          ++nacc;
          if (++slot == (uint32_t)C::SA) {
            slot = 0;
            a_ph ^= 1u;
          }
          if (++st == (uint32_t)C::SACC) {
            st = 0;
            e_ph ^= 1u;
          }
          // the next unit (groups without tiles are skipped)
          const int64_t g_this = g;
          if (--left > 0) {
            ++t;
            while (t >= tiles_g) {
              ++g;
              t = 0;
              tiles_g = tc_group_tiles<C>(args, g);
            }
          }
          if (left <= 0 || g != g_this) tc_commit(&b_empty[cur_bs]);
        }
        u.left = 0;   // the general loop below does not run
      }
      while (u.valid()) {
        if (u.g != cur_g) {
          cur_g = u.g;
          cur_bs = nb % C::SB;
          if (!mbar_wait(&b_full[cur_bs], (nb / C::SB) & 1, abort_flag)) break;
          ++nb;
        }
        // up to IL consecutive tiles of this group: their MMA chains are issued
        // interleaved (a chain of small-N MMAs on one accumulator runs at the
        // accumulate latency, two independent chains fill the gaps); each
        // accumulator still sees the same instructions in the same order
        int n = 1;
        TcUnits<C> nx = u;
        if (C::IL > 1) {
          nx.advance();
          if (nx.valid() && nx.g == u.g) n = 2;
        }
        bool ok = true;
        for (int i = 0; i < n && ok; ++i) {
          ok = mbar_wait(&a_full[(na + i) % C::SA], ((na + i) / C::SA) & 1, abort_flag);
          if (ok) ok = mbar_wait(&acc_empty[(nacc + i) % C::SACC], (((nacc + i) / C::SACC) & 1) ^ 1, abort_flag);
        }
        if (!ok) break;
        tc_fence_after();
        // gathered tiles were written through the generic proxy (cp.async); make
        // them visible to the tensor core's async-proxy reads
        if (C::GATHER) fence_proxy_async_smem();
        // descriptors: the ring's base descriptors plus offsets (the start-address
        // field is the byte address >> 4 and every offset stays inside shared
        // memory, so adding offset >> 4 moves the operand), built once per unit
        // so that each MMA costs one add per operand
        const uint64_t bdesc = descB0 + (uint64_t)((cur_bs * C::B_BYTES) >> 4);
        // two independent chains: two units (IL), or the two subtiles of one unit
        uint64_t adesc[2];
        uint32_t d[2];
        if (C::SUB > 1) {
          n = 2;
          adesc[0] = descA0 + (uint64_t)(((na % C::SA) * C::A_BYTES) >> 4);
          adesc[1] = adesc[0] + (uint64_t)(C::SUB_BYTES >> 4);
          d[0] = tmem_base + (uint32_t)((nacc % C::SACC) * C::ACC_STRIDE);
          d[1] = d[0] + C::N;
        } else {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            adesc[i] = descA0 + (uint64_t)((((na + i) % C::SA) * C::A_BYTES) >> 4);
            d[i] = tmem_base + (uint32_t)(((nacc + i) % C::SACC) * C::ACC_STRIDE);
          }
        }
        // the unit's MMAs, one chain or two interleaved (no branch between MMAs)
        auto issue = [&](auto two) {
          constexpr bool TWO = decltype(two)::value;
          if constexpr (C::FP8) {
            // e4m3 x e4m3, K = 32 per instruction: four steps of 32 bytes along the 128-byte rows
            constexpr uint32_t idesc = idesc_f16(128, C::N, 0u);   // same layout; format 0 = E4M3 here
            const uint64_t b8 = bdesc + (uint64_t)(C::BQ_BYTES >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              tc_mma_f8(d[0], adesc[0] + (uint64_t)(2 * k), b8 + (uint64_t)(2 * k), idesc, k > 0 ? 1u : 0u);
              if constexpr (TWO)
                tc_mma_f8(d[1], adesc[1] + (uint64_t)(2 * k), b8 + (uint64_t)(2 * k), idesc, k > 0 ? 1u : 0u);
            }
          } else {
            constexpr uint32_t idesc = idesc_f16(128, C::N, 1u);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t ao = (uint64_t)(((k >> 2) * (C::A_BYTES / 2) + (k & 3) * 32) >> 4);
              const uint64_t bo = (uint64_t)(((k >> 2) * (C::BQ_BYTES / 2) + (k & 3) * 32) >> 4);
              tc_mma_f16(d[0], adesc[0] + ao, bdesc + bo, idesc, k > 0 ? 1u : 0u);
              if constexpr (TWO) tc_mma_f16(d[1], adesc[1] + ao, bdesc + bo, idesc, k > 0 ? 1u : 0u);
            }
          }
        };
        if (n > 1)
          issue(std::true_type{});
        else
          issue(std::false_type{});
        if (C::SUB > 1) n = 1;                 // one unit
        for (int i = 0; i < n; ++i) {
          tc_commit(&a_empty[(na + i) % C::SA]);
          tc_commit(&acc_full[(nacc + i) % C::SACC]);
        }
        na += n;
        nacc += n;
        const int64_t g_this = u.g;
        if (n > 1) u = nx;
        u.advance();
        if (!u.valid() || u.g != g_this) tc_commit(&b_empty[cur_bs]);
      }
      // No commit may still be in flight when the CTA exits: its arrive would land
      // on whatever the next kernel on this SM keeps at that shared-memory address.
      // So the thread commits the drain barrier and waits for it, then for the last
      // phases of the slot and query-buffer barriers it commits to.
      tc_commit(&drain_bar[0]);
      mbar_wait_drain(&drain_bar[0], 0);
      if (!*abort_flag) {
        for (uint32_t i = 0; i < (uint32_t)C::SA && i < na; ++i) {
          const uint32_t j = na - 1 - i;
          mbar_wait_drain(&a_empty[j % C::SA], (j / C::SA) & 1);
        }
        for (uint32_t i = 0; i < (uint32_t)C::SB && i < nb; ++i) {
          const uint32_t j = nb - 1 - i;
          mbar_wait_drain(&b_empty[j % C::SB], (j / C::SB) & 1);
        }
      }
    }
  } else if (warp >= C::EPI0 && warp < C::EPI0 + C::NE) {
    // ------------------------------------------------------------ epilogue
    if constexpr (C::WREG) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::EPI_REGS) : "memory");
    const int ew = warp - C::EPI0;             // epilogue warp index
    const int quarter = warp & 3;              // TMEM lanes this warp may read
    // first query of this warp in a tile, and the warps per lane quarter that
    // read one unit (its queries are qfirst, qfirst + QSTEP, ...)
    const int qfirst = C::NQ > 1 ? ((ew % C::EPT) >> 2) : 0;
    constexpr int QSTEP = C::NQ > 1 ? C::EPT / 4 : 1;
    const int tile_par = ew / C::EPT;          // alternate units: the parity of the units this warp takes
    const int sub = C::SUB > 1 ? (ew >> 2) : 0;   // two subtiles per unit: the one this warp reads
    const int row_in_tile = quarter * 32 + lane;
    float* sW = sW_all + ew * C::NQ * C::NCOL;
    int32_t* sLen = sLen_all + ew * C::NQ;
    int64_t* sBase = sBase_all + ew * C::NQ;
    float* sAux = sAux_all + ew * C::NQ * 4;   // coef, tau, sigma per query
    TcUnits<C> u;
    u.init(args, s);
    int64_t cur_g = -1;
    uint32_t nacc = 0, ngrp = 0;
    // two-query epilogue: this warp's query pairs' weights, (w_a[h], w_b[h]) packed
    constexpr int PPW = C::PAIR ? C::NQ / QSTEP / 2 : 1;   // query pairs of this warp
    static_assert(!C::PAIR || C::H % 16 == 0, "two-query epilogue: whole TMEM loads");
    uint64_t wreg[C::PAIR ? PPW * C::H : 1];
#pragma unroll
    for (int i = 0; i < (C::PAIR ? PPW * C::H : 1); ++i) wreg[i] = 0;
    if constexpr (C::BPAIR) {
      // The bound over 16-vector blocks.  This warp's set takes every other unit
      // of the CTA's range (those of parity tile_par), so the walk of TcUnits
      // steps two units at a time, on 32-bit counters like the stage and its
      // phase, and lanes 0..BQ-1 store the bitmap words of the warp's BQ rows.
      constexpr int BQ = C::NQ / QSTEP;        // rows of a group this warp reads
      static_assert(BQ % 2 == 0 && BQ <= 32, "rows in pairs, one storing lane each");
      int bq_len[BQ];
      float bq_coef[BQ], bq_tau[BQ];
      int32_t g = (int32_t)u.g, t = (int32_t)u.t, tiles_g = (int32_t)u.tiles_g, gcur = -1;
      int64_t left = u.left;
      if (tile_par == 1 && left > 0 && --left > 0) {
        // the set's first unit is the range's second
        ++t;
        while (t >= tiles_g) {
          ++g;
          t = 0;
          tiles_g = (int32_t)tc_group_tiles<C>(args, g);
        }
      }
      uint32_t st = (uint32_t)tile_par, f_ph = 0;   // accumulator stage of the unit, its phase
      uint32_t* cb_row = nullptr;                   // lane b < BQ: row b's candidate bitmap
      while (left > 0) {
        if (g != gcur) {
          gcur = g;
          __syncwarp();
          // folded weights of the warp's rows, pair c = rows 2c, 2c + 1 stored
          // (w_a[h], w_b[h]) adjacent
          for (int i = lane; i < BQ * C::NCOL; i += 32) {
            const int r = i / C::NCOL, h = i % C::NCOL;
            const int64_t m = (int64_t)g * C::NQ + qfirst + r * QSTEP;
            sW[(r >> 1) * 2 * C::NCOL + 2 * h + (r & 1)] = m < args.p.M ? args.wfold[m * 32 + h] : 0.0f;
          }
          __syncwarp();
#pragma unroll
          for (int b = 0; b < BQ; ++b) {
            const int64_t m = (int64_t)g * C::NQ + qfirst + b * QSTEP;
            int64_t off = 0;
            int len = 0;
            if (m < args.p.M) {
              row_extent(args.p, m, &off, &len);
              if (args.row_mask && !args.row_mask[m]) len = 0;
            }
            bq_len[b] = len;
            bq_coef[b] = m < args.p.M ? args.coef[m] : 0.0f;
            bq_tau[b] = m < args.p.M ? args.tau[m] : 0.0f;
          }
          const int64_t ml = (int64_t)g * C::NQ + qfirst + lane * QSTEP;
          cb_row = (lane < BQ && ml < args.p.M) ? args.candbits + ml * args.cb_stride : nullptr;
        }
        const int key = t * C::UKEYS + row_in_tile;
        const uint32_t kbit = 1u << (key & 31);
        // ||k|| and the seed words of this lane's key, read before the wait so that
        // the loads overlap it (words cover max_key_len keys)
        float knorm = 0.0f;
        uint32_t sword = 0u, sw2[BQ];
#pragma unroll
        for (int b = 0; b < BQ; ++b) sw2[b] = 0u;
        if (key < args.p.max_key_len) {
          knorm = __ldg(args.knorm + key);
          if (args.seed_stride == 0) sword = __ldg(args.seedbits + (key >> 5));
        }
        if (args.seed_stride != 0) {
#pragma unroll
          for (int b = 0; b < BQ; ++b) {
            const int64_t m = (int64_t)g * C::NQ + qfirst + b * QSTEP;
            if (key < bq_len[b]) sw2[b] = __ldg(args.seedbits + m * args.seed_stride + (key >> 5));
          }
        }
        const bool got = mbar_wait(&acc_full[st], f_ph, abort_flag);
        __syncwarp();                         // tcgen05.ld below is warp-collective
        if (!__all_sync(0xffffffffu, got)) break;
        tc_fence_after();
        // 16 retained vectors per query, rows qfirst + b * QSTEP of the group, taken
        // in pairs (2c, 2c + 1): the halves of packed chains, two per pair (heads
        // 2i and 2i + 1) so that each dependent sequence is 8 deep, then their sum.
        // The summation order differs from the scalar chain by a few ulp, far
        // inside the margin coef[m] already carries for the bf16 operands.
        constexpr int NPR = BQ / 2;
        const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + st * (uint32_t)C::ACC_STRIDE;
        float chain[BQ];
        uint32_t agg[BQ];
#pragma unroll
        for (int c = 0; c < NPR; ++c) {
          // rows 2c and 2c + 1: columns 0..15 of each (one TMEM wait per pair, so
          // that only one pair's values are live)
          uint32_t v[2][32];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int q = qfirst + (2 * c + e) * QSTEP;
            tmem_ld_32x32b_x16(tbase + (uint32_t)(q * C::NCOL), v[e]);
            agg[2 * c + e] = tmem_ld_32x32b_x1(tbase + (uint32_t)(C::NQ * C::NCOL + q));
          }
          tmem_ld_wait();
          // weights of pair c stored (w_a[h], w_b[h]) adjacent: one 16-byte load
          // gives the operand pairs of heads j and j + 1
          const float4* w4 = reinterpret_cast<const float4*>(sW + c * 2 * C::NCOL);
          uint64_t se = f2_pack(0.0f, 0.0f), so = f2_pack(0.0f, 0.0f);
#pragma unroll
          for (int j2 = 0; j2 < 8; ++j2) {
            const float4 ww = w4[j2];
            const int j = 2 * j2;
            se = f2_fma(f2_pack(ww.x, ww.y),
                        f2_pack(fmaxf(__uint_as_float(v[0][j]), 0.0f), fmaxf(__uint_as_float(v[1][j]), 0.0f)), se);
            so = f2_fma(f2_pack(ww.z, ww.w),
                        f2_pack(fmaxf(__uint_as_float(v[0][j + 1]), 0.0f), fmaxf(__uint_as_float(v[1][j + 1]), 0.0f)),
                        so);
          }
          float e0, e1, o0, o1;
          f2_unpack(se, &e0, &e1);
          f2_unpack(so, &o0, &o1);
          chain[2 * c] = e0 + o0;
          chain[2 * c + 1] = e1 + o1;
        }
        unsigned mine = 0u;
#pragma unroll
        for (int b = 0; b < BQ; ++b) {
          float ub = chain[b] - fmaxf(__uint_as_float(agg[b]), 0.0f);
          ub = __fmaf_rn(bq_coef[b], knorm, ub);
          const uint32_t word = args.seed_stride ? sw2[b] : sword;
          const bool is_cand = key < bq_len[b] && !(word & kbit) && !(ub < bq_tau[b]);
          const unsigned mk = __ballot_sync(0xffffffffu, is_cand);
          if (lane == b) mine = mk;
        }
        // the warp's 32 keys are one bitmap word (key - lane is a multiple of 32)
        const int64_t wd = (int64_t)t * (C::UKEYS / 32) + quarter;
        if (cb_row && wd < args.cb_stride) cb_row[wd] = mine;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[st]);
        // this set's next unit, two on (groups without tiles are skipped)
        st += 2;
        if (st >= (uint32_t)C::SACC) {
          st -= C::SACC;
          f_ph ^= 1u;
        }
        left -= 2;
        if (left > 0) {
          t += 2;
          while (t >= tiles_g) {
            t -= tiles_g;
            ++g;
            tiles_g = (int32_t)tc_group_tiles<C>(args, g);
          }
        }
      }
    }
    while (!C::BPAIR && u.valid()) {
      if (u.g != cur_g) {
        cur_g = u.g;
        __syncwarp();
        if constexpr (C::FP8) {
          // the group's sigma per query, as the split warps used it
          const int sl = ngrp % C::SIGR;
          bool ok = true;
          if (lane == 0) ok = mbar_wait(&sig_full[sl], (ngrp / C::SIGR) & 1, abort_flag);
          if (!__shfl_sync(0xffffffffu, ok, 0)) break;
          if (lane < C::NQ) sAux[4 * lane + 2] = sSig[sl * C::NQ + lane];
          __syncwarp();
          if (lane == 0) mbar_arrive(&sig_empty[sl]);
          ++ngrp;
        }
        for (int i = lane; i < C::NQ * C::NCOL; i += 32) {
          const int qi = i / C::NCOL, h = i % C::NCOL;
          const int64_t m = cur_g * C::NQ + qi;
          float wv = 0.0f;
          if (m < args.p.M) wv = C::BOUND ? args.wfold[m * 32 + h] : args.p.w[m * C::H + h];
          if constexpr (C::PAIR) {
            // this warp's r-th query goes to pair r/2, half r%2: [pair][h][2]
            if ((qi - qfirst) % QSTEP != 0) continue;
            const int r = (qi - qfirst) / QSTEP;
            sW[(r >> 1) * 2 * C::NCOL + 2 * h + (r & 1)] = wv;
          } else {
            sW[i] = wv;
          }
        }
        if (!C::FP8 && lane < C::NQ) sAux[4 * lane + 2] = 1.0f;
        if (lane < C::NQ) {
          const int64_t m = cur_g * C::NQ + lane;
          int64_t off = 0;
          int len = 0;
          if (m < args.p.M) {
            if (C::GROUP) {
              len = args.cnt[cur_g];               // every row of the group: the group's list
            } else if (C::GATHER) {
              len = args.cnt[m];
              off = tc_key_base(args, m);
            } else {
              row_extent(args.p, m, &off, &len);
            }
            if (args.row_mask && !args.row_mask[m]) len = 0;
          }
          sLen[lane] = len;
          sBase[lane] = off;
          if (C::BOUND) sAux[4 * lane] = m < args.p.M ? args.coef[m] : 0.0f;
          if (C::BOUND || C::FILTER) sAux[4 * lane + 1] = m < args.p.M ? args.tau[m] : 0.0f;
        }
        __syncwarp();
        if constexpr (C::PAIR) {
#pragma unroll
          for (int i = 0; i < PPW * C::H; ++i)
            wreg[i] = reinterpret_cast<const uint64_t*>(sW + (i / C::H) * 2 * C::NCOL)[i % C::H];
        }
      }
      if (C::ALT && (int)(nacc & 1) != tile_par) {
        ++nacc;
        u.advance();
        continue;
      }
      const int acc = nacc % C::SACC;
      const int key = (int)(u.t * C::UKEYS) + sub * 128 + row_in_tile;
      // kBound with one seed bitmap for all rows: this key's word, read before the
      // wait so that the load overlaps it (words cover max_key_len keys)
      uint32_t sword = 0;
      if (C::BOUND && args.seed_stride == 0 && key < args.p.max_key_len) sword = __ldg(args.seedbits + (key >> 5));
      float knorm = 0.0f;
      if (C::KN_GLOBAL && key < args.p.max_key_len) knorm = __ldg(args.knorm + key);
      bool got = mbar_wait(&acc_full[acc], (nacc / C::SACC) & 1, abort_flag);
      // the key-tile slot of this unit (bound: read below for ||k||, so the slot is
      // held until this warp releases it) and its scale slot (FP8)
      const int slot = nacc % C::SA;
      const int sslot = nacc % C::SSC_MOD;
      if (C::KN_TILE && got) got = mbar_wait(&a_full[slot], (nacc / C::SA) & 1, abort_flag);
      if (C::FP8 && got) got = mbar_wait(&sc_full[sslot], (nacc / C::SSC_MOD) & 1, abort_flag);
      __syncwarp();                           // tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      // FP8: all queries of a group read the same key sequence, so one scale serves them all
      const float kscale = C::FP8 ? sScale[sslot * C::UKEYS + sub * 128 + row_in_tile] : 1.0f;
      if (C::KN_TILE) {
        // ||k|| of this lane's key (codes for FP8) from the MMA-ready tile
        const uint8_t* at = sA + slot * C::A_BYTES;
        float ss = 0.0f;
        constexpr int HALVES = C::FP8 ? 1 : 2;
#pragma unroll
        for (int h = 0; h < HALVES; ++h) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(at + h * (C::A_BYTES / 2) + row_in_tile * 128 +
                                                            ((c ^ (row_in_tile & 7)) << 4));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (C::FP8) {
                float x0, x1, x2, x3;
                e4m3x2_to_f32(w4[e], &x0, &x1);
                e4m3x2_to_f32(w4[e] >> 16, &x2, &x3);
                ss = __fmaf_rn(x0, x0, ss);
                ss = __fmaf_rn(x1, x1, ss);
                ss = __fmaf_rn(x2, x2, ss);
                ss = __fmaf_rn(x3, x3, ss);
              } else {
                const float lo = __uint_as_float(w4[e] << 16);
                const float hi = __uint_as_float(w4[e] & 0xffff0000u);
                ss = __fmaf_rn(lo, lo, ss);
                ss = __fmaf_rn(hi, hi, ss);
              }
            }
          }
        }
        knorm = __fsqrt_ru(ss);
      }
      if (C::KN_TILE || C::FP8) {
        __syncwarp();
        if (lane == 0) {
          if (C::KN_TILE) mbar_arrive(&a_empty[slot]);
          if (C::FP8) mbar_arrive(&sc_empty[sslot]);
        }
      }
      // kBound: U of this lane's key for query qi (row m) from its 32 accumulator
      // columns, and the warp's 32 candidate bits as one bitmap word
      // (the retained-head chain sum_j w'_j ReLU(acc_j) is computed by the callers:
      // rows R..30 of the prepared vectors and their folded weights are zero, so a
      // chain that stops anywhere at or past R has the same value)
      auto bound_finish = [&](int qi, int64_t m, float chain, uint32_t agg) {
        float ub = chain - fmaxf(__uint_as_float(agg), 0.0f);
        if (C::FP8) ub = ub * sAux[4 * qi + 2];
        ub = __fmaf_rn(sAux[4 * qi], knorm, ub);
        bool is_cand = false;
        if (key < sLen[qi]) {
          if (C::FP8) ub = ub * kscale;
          const uint32_t word = args.seed_stride ? args.seedbits[m * args.seed_stride + (key >> 5)] : sword;
          const bool seed = (word >> (key & 31)) & 1u;
          is_cand = !seed && !(ub < sAux[4 * qi + 1]);
        }
        // the warp's 32 keys are one bitmap word (key - lane is a multiple of 32)
        const unsigned mask = __ballot_sync(0xffffffffu, is_cand);
        const int64_t wd = key >> 5;
        if (lane == 0 && wd < args.cb_stride) args.candbits[m * args.cb_stride + wd] = mask;
      };
      auto bound_word = [&](int qi, int64_t m, const uint32_t (&v)[32]) {
        float ub = 0.0f;
        const float4* w4 = reinterpret_cast<const float4*>(sW + qi * C::NCOL);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 ww = w4[j4];
          const int j = 4 * j4;
          ub = __fmaf_rn(ww.x, fmaxf(__uint_as_float(v[j]), 0.0f), ub);
          ub = __fmaf_rn(ww.y, fmaxf(__uint_as_float(v[j + 1]), 0.0f), ub);
          ub = __fmaf_rn(ww.z, fmaxf(__uint_as_float(v[j + 2]), 0.0f), ub);
          if (j4 < 7) ub = __fmaf_rn(ww.w, fmaxf(__uint_as_float(v[j + 3]), 0.0f), ub);
        }
        bound_finish(qi, m, ub, v[31]);
      };
      if constexpr (C::BOUND && !C::FP8 && C::NQ > 1 && (C::NQ == 4 * QSTEP || C::NQ == 2 * QSTEP)) {
        constexpr int QPW = C::NQ / QSTEP;     // queries of this warp in a tile
        const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * C::ACC_STRIDE);
        if (args.R <= 16) {
          // at most 16 retained heads: columns 0..15 of each of this warp's four
          // queries and their aggregates (column 31 of the query), one TMEM wait;
          // two packed chains (queries 0|1 and 2|3 of the warp in the halves of
          // fma.rn.f32x2, each rounding as fmaf)
          uint32_t v[QPW][32], agg[QPW];
#pragma unroll
          for (int b = 0; b < QPW; ++b) {
            const int q = qfirst + b * QSTEP;
            const uint32_t col = tbase + (uint32_t)(q * C::NCOLX);
            tmem_ld_32x32b_x16(col, v[b]);
            agg[b] = tmem_ld_32x32b_x1(col + 31);
          }
          tmem_ld_wait();
          // queries 2c and 2c + 1 of this warp in the halves of chain c
          uint64_t sc2[QPW / 2];
#pragma unroll
          for (int c = 0; c < QPW / 2; ++c) sc2[c] = f2_pack(0.0f, 0.0f);
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
#pragma unroll
            for (int c = 0; c < QPW / 2; ++c) {
              const float4 a = reinterpret_cast<const float4*>(sW + (qfirst + (2 * c) * QSTEP) * C::NCOL)[j4];
              const float4 b = reinterpret_cast<const float4*>(sW + (qfirst + (2 * c + 1) * QSTEP) * C::NCOL)[j4];
              const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int j = 4 * j4 + e;
                sc2[c] = f2_fma(f2_pack(av[e], bv[e]),
                                f2_pack(fmaxf(__uint_as_float(v[2 * c][j]), 0.0f),
                                        fmaxf(__uint_as_float(v[2 * c + 1][j]), 0.0f)),
                                sc2[c]);
              }
            }
          }
          float u[QPW];
#pragma unroll
          for (int c = 0; c < QPW / 2; ++c) f2_unpack(sc2[c], &u[2 * c], &u[2 * c + 1]);
#pragma unroll
          for (int b = 0; b < QPW; ++b) {
            const int qi = qfirst + b * QSTEP;
            const int64_t m = cur_g * C::NQ + qi;
            if (m < args.p.M) bound_finish(qi, m, u[b], agg[b]);
          }
        } else {
          // more retained heads: the whole 31-column chain, two queries per TMEM wait
#pragma unroll 1
          for (int qi = qfirst; qi < C::NQ; qi += 2 * QSTEP) {
            const int64_t ma = cur_g * C::NQ + qi;
            if (ma >= args.p.M) break;
            const int qb = qi + QSTEP;
            const int64_t mb = cur_g * C::NQ + qb;
            uint32_t va[32], vb[32];
            tmem_ld_32x32b_x32(tbase + (uint32_t)(qi * C::NCOLX), va);
            tmem_ld_32x32b_x32(tbase + (uint32_t)(qb * C::NCOLX), vb);
            tmem_ld_wait();
            bound_word(qi, ma, va);
            if (mb < args.p.M) bound_word(qb, mb, vb);
          }
        }
      } else if constexpr (C::PAIR) {
        // queries qi and qi + QSTEP, chains packed (a in the low half, b in the
        // high half), the weight pairs from registers (loaded at the group change)
        const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * C::ACC_STRIDE);
#pragma unroll
        for (int pp = 0; pp < PPW; ++pp) {
          const int qi = qfirst + 2 * pp * QSTEP, qb = qi + QSTEP;
          const int64_t ma = cur_g * C::NQ + qi, mb = cur_g * C::NQ + qb;
          if (ma >= args.p.M) break;
          const uint32_t ta = tbase + (uint32_t)(qi * C::NCOLX), tb = tbase + (uint32_t)(qb * C::NCOLX);
          constexpr int CW = 16;                        // heads per TMEM wait
          uint64_t s2 = 0;
#pragma unroll
          for (int c = 0; c < C::H / CW; ++c) {
            uint32_t va[32], vb[32];   // columns 0..CW-1 used
            tmem_ld_32x32b_x16(ta + CW * c, va);
            tmem_ld_32x32b_x16(tb + CW * c, vb);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < CW; ++j)
              s2 = f2_fma(wreg[pp * C::H + CW * c + j],
                          f2_pack(fmaxf(__uint_as_float(va[j]), 0.0f), fmaxf(__uint_as_float(vb[j]), 0.0f)), s2);
          }
          float sa, sb;
          f2_unpack(s2, &sa, &sb);
          if (key < sLen[qi]) args.scores[ma * args.ld + key] = sa;
          if (mb < args.p.M && key < sLen[qb]) args.scores[mb * args.ld + key] = sb;
        }
      } else
#pragma unroll 1
      for (int qi = qfirst; qi < C::NQ; qi += QSTEP) {
        const int64_t m = cur_g * C::NQ + qi;
        if (m >= args.p.M) break;
        const uint32_t tcol = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                              (uint32_t)(acc * C::ACC_STRIDE + sub * C::N + qi * C::NCOLX);
        const float* wq = sW + qi * C::NCOL;
        const int len = sLen[qi];
        if (!C::BOUND) {
          float sc = 0.0f;
          constexpr int NCH = (C::H + 31) / 32;      // 32-head chunks per query
          constexpr int CW = C::H < 32 ? C::H : 32;  // heads per chunk
          if constexpr (C::FP8) {
            // head h: hi column h plus lo column H + h
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
              uint32_t vh[32], vl[32];
              if (C::H >= 32) {
                tmem_ld_32x32b_x32(tcol + 32 * c, vh);
                tmem_ld_32x32b_x32(tcol + C::H + 32 * c, vl);
              } else {
                tmem_ld_32x32b_x16(tcol, vh);
                tmem_ld_32x32b_x16(tcol + C::H, vl);
              }
              tmem_ld_wait();
              const float4* w4 = reinterpret_cast<const float4*>(wq + 32 * c);
#pragma unroll
              for (int j4 = 0; j4 < CW / 4; ++j4) {
                const float4 ww = w4[j4];
                const float wv[4] = {ww.x, ww.y, ww.z, ww.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int j = 4 * j4 + e;
                  sc = __fmaf_rn(wv[e], fmaxf(__uint_as_float(vh[j]) + __uint_as_float(vl[j]), 0.0f), sc);
                }
              }
            }
          } else {
            constexpr int GRP = NCH < 2 ? NCH : 2;     // loads in flight before one wait
            // head chain h = 0 .. H-1, weights four at a time (broadcast loads)
#pragma unroll
            for (int c0 = 0; c0 < NCH; c0 += GRP) {
              uint32_t v[GRP][32];
#pragma unroll
              for (int c = 0; c < GRP; ++c) {
                if (C::H >= 32) {
                  tmem_ld_32x32b_x32(tcol + 32 * (c0 + c), v[c]);
                } else {
                  tmem_ld_32x32b_x16(tcol, v[c]);
                }
              }
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < GRP; ++c) {
                const float4* w4 = reinterpret_cast<const float4*>(wq + 32 * (c0 + c));
#pragma unroll
                for (int j4 = 0; j4 < CW / 4; ++j4) {
                  const float4 ww = w4[j4];
                  sc = __fmaf_rn(ww.x, fmaxf(__uint_as_float(v[c][4 * j4 + 0]), 0.0f), sc);
                  sc = __fmaf_rn(ww.y, fmaxf(__uint_as_float(v[c][4 * j4 + 1]), 0.0f), sc);
                  sc = __fmaf_rn(ww.z, fmaxf(__uint_as_float(v[c][4 * j4 + 2]), 0.0f), sc);
                  sc = __fmaf_rn(ww.w, fmaxf(__uint_as_float(v[c][4 * j4 + 3]), 0.0f), sc);
                }
              }
            }
          }
          const float val = C::FP8 ? (sc * sAux[4 * qi + 2]) * kscale : sc;
          if constexpr (C::FILTER) {
            // the same value the dense mode writes; kept iff >= tau (warp ballot, one atomic per warp)
            tc_append(args, m, key < len && !(val < sAux[4 * qi + 1]), key, val);
          } else if (key < len) {
            args.scores[m * args.ld + key] = val;
          }
        } else {
          uint32_t v[32], vl[32];
          tmem_ld_32x32b_x32(tcol, v);
          if (C::FP8) tmem_ld_32x32b_x32(tcol + 32, vl);
          tmem_ld_wait();
          if (C::FP8) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(vl[j]));
          }
          bound_word(qi, m, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      ++nacc;
      u.advance();
    }
  } else if (C::FP8 && warp < 2 + C::NE + C::NCONV) {
    // ------------------------------------------------------------ query split
    // Per query group, once the MMA has released the buffer: bf16 row v of query
    // qi (global memory, 256 bytes, one coalesced warp load) -> e4m3 B rows
    // qi*2*NCOL + v (hi) and qi*2*NCOL + NCOL + v (lo) (128-byte rows, 128-byte
    // swizzle); rows of queries past M are zero.
    const int cw = warp - 2 - C::NE;           // split warp 0..NCONV-1
    TcUnits<C> u;
    u.init(args, s);
    int64_t cur_g = -1;
    uint32_t nb = 0;
    while (u.valid()) {
      if (u.g != cur_g) {
        cur_g = u.g;
        const int bs = nb % C::SB;
        bool ok = mbar_wait(&b_empty[bs], ((nb / C::SB) & 1) ^ 1, abort_flag);
        const int sl = nb % C::SIGR_MOD;
        if (cw == 0 && ok && lane == 0) ok = mbar_wait(&sig_empty[sl], ((nb / C::SIGR_MOD) & 1) ^ 1, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
        uint8_t* b8 = sB + bs * C::B_BYTES;
        for (int qi = 0; qi < C::NQ; ++qi) {
          const int64_t m = cur_g * C::NQ + qi;
          const bool live = m < args.p.M;
          const uint16_t* qrow = (const uint16_t*)args.p.q + (live ? m : 0) * C::NCOL * 128;
          float sig = 1.0f, inv = 1.0f;
          if (live) row_sigma(query_amax<C::NCOL>(qrow), &sig, &inv);
          if (cw == 0 && lane == 0) sSig[sl * C::NQ + qi] = sig;
#pragma unroll 8
          for (int v = cw; v < C::NCOL; v += C::NCONV) {
            uint2 q4 = make_uint2(0u, 0u);
            if (live) q4 = __ldg(reinterpret_cast<const uint2*>(qrow + v * 128) + lane);
            // elements 4*lane .. 4*lane+3
            const float x[4] = {__uint_as_float(q4.x << 16) * inv, __uint_as_float(q4.x & 0xffff0000u) * inv,
                                __uint_as_float(q4.y << 16) * inv, __uint_as_float(q4.y & 0xffff0000u) * inv};
            const uint32_t h01 = e4m3x2(x[0], x[1]), h23 = e4m3x2(x[2], x[3]);
            float hv[4];
            e4m3x2_to_f32(h01, &hv[0], &hv[1]);
            e4m3x2_to_f32(h23, &hv[2], &hv[3]);
            const uint32_t l01 = e4m3x2(x[0] - hv[0], x[1] - hv[1]);
            const uint32_t l23 = e4m3x2(x[2] - hv[2], x[3] - hv[3]);
            const uint32_t hi = h01 | (h23 << 16), lo = l01 | (l23 << 16);
            // byte 4*lane of a 128-byte row: 16-byte chunk lane/4, offset 4*(lane%4)
            const int rh = qi * 2 * C::NCOL + v, rl = rh + C::NCOL;
            *reinterpret_cast<uint32_t*>(b8 + rh * 128 + (((lane >> 2) ^ (rh & 7)) << 4) + 4 * (lane & 3)) = hi;
            *reinterpret_cast<uint32_t*>(b8 + rl * 128 + (((lane >> 2) ^ (rl & 7)) << 4) + 4 * (lane & 3)) = lo;
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&b_full[bs]);
        if (cw == 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&sig_full[sl]);
        }
        ++nb;
      }
      u.advance();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// 2-D tensor map over a row-major [rows, inner] matrix, 128-byte swizzle.
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows);

// Launches one configuration.  Query rows are a.p.q viewed as [M * NCOL, 128] bf16.
template <class C>
cudaError_t launch_tc(const TcArgs& a_in, cudaStream_t st) {
  TcArgs a = a_in;
  const idx_problem& p = a.p;
  if (p.M <= 0 || p.n_keys <= 0) return cudaSuccess;
  if (!C::GATHER && p.max_key_len <= 0) return cudaSuccess;
  if (p.n_keys >= ((int64_t)1 << 31) || p.M * C::NCOL >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  CUtensorMap tk, tq;
  bool ok;
  // gathered modes copy key rows with cp.async and never read through this map
  const uint32_t krows = C::GATHER ? 1u : (uint32_t)C::UKEYS;
  if (C::FP8)
    ok = make_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.keys, 128, (uint64_t)p.n_keys, 128, 128, krows);
  else
    ok = make_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.keys, 128, (uint64_t)p.n_keys, 256, 64, krows);
  a.G = (p.M + C::NQ - 1) / C::NQ;
  // query-side rows: M x NCOL, or (AGG16) QROWS per group
  const uint64_t qrows = C::AGG16 ? (uint64_t)(a.G * C::QROWS) : (uint64_t)(p.M * C::NCOL);
  ok = ok && make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, 128, qrows, 256, 64, C::QROWS);
  if (!ok) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if constexpr (C::WREG) {
    // setmaxnreg moves registers within the block: the epilogue warpgroups'
    // increase must not exceed what warpgroup 0 gives back from the launch count
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, score_tc_kernel<C>);
    if (e != cudaSuccess) return e;
    if (4 * C::WG0_REGS + 8 * C::EPI_REGS > 12 * fa.numRegs || fa.numRegs > C::EPI_REGS) return cudaErrorInvalidConfiguration;
  }
  score_tc_kernel<C><<<sm_count(), C::NTHREADS, C::SMEM_BYTES, st>>>(tk, tq, a);
  return cudaGetLastError();
}

}  // namespace idx
