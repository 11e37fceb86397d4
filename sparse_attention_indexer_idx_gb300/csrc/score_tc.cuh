// Indexer score and DoSA bound on the 5th-generation tensor cores (tcgen05,
// sm_103a), bf16 queries with bf16 keys or FP8 e4m3 keys (+ per-token scale),
// D = 128.
//
// Mapping.  One MMA tile is 128 keys (the M axis: key i of the tile lives in
// TMEM lane i) times N = NQ*NCOL columns (NQ queries x NCOL vectors each, all
// K-major), the full D = 128 as 8 MMAs of K = 16.  Each epilogue thread owns
// one key and reduces its own TMEM columns with no shuffles.
//
// Modes:
//  kScore   s(k) = sum_h w_h ReLU(q_h . k) ("DoSA：用安全上界减少 Indexer 的完整
//           打分", section 3), NCOL = H; the head sum is one fused-multiply-add
//           chain h = 0..H-1, so a (query, key) score has the same bits
//           wherever it is computed -- same instruction shape, same K order,
//           same chain.
//  kGather  the same score over per-row key lists: tile t of row m holds the
//           keys list[m][t*128 + i], fetched by TMA tile::gather4 (four rows
//           per instruction) straight into the swizzled tile.  Used to rescore
//           DoSA candidates; output is indexed by list position.
//  kBound   DoSA's safe upper bound (same page, sections 2, 3.1, 3.2): B holds
//           per query R retained head vectors (rows 0..R-1) and the |w|-folded
//           negative aggregate (row 31); the epilogue evaluates
//             U = sum_j w'_j ReLU(q_j . k) + coef ||k|| - ReLU(a . k)
//           (times the FP8 scale), with ||k|| read from the key tile in shared
//           memory, and appends every visible non-seed key with U >= tau to the
//           row's candidate list (drop only when U < tau).
//
// Work units are (query group g, key tile t).  Shared keys (causal prefill): a
// group is NQ consecutive rows over one key sequence.  Per-row keys (decode,
// gathered lists): a group is one row.  The units are split into one
// contiguous range per CTA (persistent, one CTA per SM), balanced by the exact
// tile count of every group, which a prologue warp scans from the lengths.
//
// Warp roles:  warp 0  TMA producer (key tiles, query tiles)
//              warp 1  TMEM allocation + MMA issue (one thread)
//              warps 2..  epilogue (4, or 8 when a tile holds several queries:
//                         two per TMEM lane quarter, alternating queries):
//                         tcgen05.ld -> score / bound -> global
//              last 4     (FP8 only) e4m3 -> f16 conversion of key tiles into
//                         the swizzled MMA layout, bf16 -> f16 of query tiles
// Every wait is bounded (see common.cuh); on a timeout all roles stop, the
// producer and the MMA thread drain what they issued, and TMEM is released.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace idx {

enum TcMode { kScore = 0, kGather = 1, kBound = 2 };

struct TcArgs {
  idx_problem p;              // p.q is the B source: queries, or prepared vectors (kBound)
  float* scores;
  int64_t ld;
  int64_t G;                  // groups
  // kGather: row m's keys are key_base(m) + list[m*gld + i], i < cnt[m]
  const int32_t* list;
  const int32_t* cnt;
  int64_t gld;
  // kBound
  const float* wfold;         // [M, 32] folded retained weights (j < R)
  const float* coef;          // [M] c + margin, multiplies ||k||
  const float* tau;           // [M]
  const uint32_t* seedbits;   // seed bitmap, row stride seed_stride words (0: one shared bitmap)
  int64_t seed_stride;
  int32_t* cand;              // [M, cap] candidate ids
  int32_t* cand_cnt;          // [M]
  int64_t cap;
  int32_t* status;            // [M] bit 1: candidate overflow
  const int32_t* row_mask;    // optional [M]: rows with row_mask[m] == 0 are skipped
  int R;
};

__host__ __device__ constexpr int tc_pow2_cols(int c) {
  return c <= 32 ? 32 : (c <= 64 ? 64 : (c <= 128 ? 128 : (c <= 256 ? 256 : 512)));
}

template <int KDT_, int NCOL_, int NQ_, int MODE_>
struct TcCfg {
  static constexpr int KDT = KDT_;
  static constexpr int NCOL = NCOL_;          // H (score) or 32 (bound)
  static constexpr int H = NCOL_;
  static constexpr int NQ = NQ_;
  static constexpr int MODE = MODE_;
  static constexpr bool FP8 = (KDT == IDX_FP8_E4M3);
  static constexpr bool GATHER = (MODE == kGather);
  static constexpr bool BOUND = (MODE == kBound);
  static constexpr int N = NQ * NCOL;
  static constexpr int A_BYTES = 128 * 128 * 2;
  static constexpr int B_BYTES = N * 128 * 2;
  static constexpr int RAW_BYTES = 128 * 128;
  static constexpr int SB = (NQ > 1) ? 1 : 2;
  // FP8: two converted (f16) tiles are enough for the MMA; every other byte of
  // shared memory holds raw tiles in flight from HBM
  static constexpr int SA = FP8 ? 2 : ((B_BYTES * SB <= 32768) ? 5 : 4);
  static constexpr int SRAW_FIT = (212 * 1024 - SA * A_BYTES - SB * B_BYTES) / RAW_BYTES;
  static constexpr int SRAW = FP8 ? (SRAW_FIT > 8 ? 8 : SRAW_FIT) : 0;
  static constexpr int SRAW_MOD = SRAW > 0 ? SRAW : 1;   // ring index arithmetic
  static constexpr int SACC = (N >= 256) ? 2 : 4;
  static constexpr int TMEM_COLS = tc_pow2_cols(SACC * N);
  // epilogue warps: two per TMEM lane quarter when a tile holds several queries
  // (each takes every other query), else one
  static constexpr int NE = (NQ > 1) ? 8 : 4;
  static constexpr int NTHREADS = 32 * (2 + NE + (FP8 ? 4 : 0));
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + SA * A_BYTES;
  static constexpr int OFF_RAW = OFF_B + SB * B_BYTES;
  // per epilogue warp (NE private copies, so the warps never wait on each other)
  static constexpr int OFF_W = OFF_RAW + SRAW * RAW_BYTES;
  static constexpr int OFF_BASE = OFF_W + NE * N * 4;
  static constexpr int OFF_LEN = OFF_BASE + NE * NQ * 8;
  static constexpr int OFF_AUX = OFF_LEN + NE * NQ * 4;        // coef, tau per query (bound)
  static constexpr int OFF_BAR = ((OFF_AUX + NE * NQ * 8) + 7) & ~7;
  static constexpr int NBARS = 2 * SA + 3 * SB + 2 * SRAW + 2 * SACC + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;   // + alignment slack
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "MMA N");
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
    if (A.row_mask && !A.row_mask[g]) return 0;
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
  return (mx + 127) / 128;
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

__device__ __forceinline__ void tma_gather4(void* dst, const void* tmap, uint64_t* bar, int32_t x, int32_t y0,
                                            int32_t y1, int32_t y2, int32_t y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
      "%5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
      : "memory");
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
  uint8_t* sRaw = smem + C::OFF_RAW;
  float* sW_all = reinterpret_cast<float*>(smem + C::OFF_W);
  int32_t* sLen_all = reinterpret_cast<int32_t*>(smem + C::OFF_LEN);
  int64_t* sBase_all = reinterpret_cast<int64_t*>(smem + C::OFF_BASE);
  float* sAux_all = reinterpret_cast<float*>(smem + C::OFF_AUX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* a_full = bars;
  uint64_t* a_empty = a_full + C::SA;
  uint64_t* b_full = a_empty + C::SA;
  uint64_t* b_empty = b_full + C::SB;
  uint64_t* b_loaded = b_empty + C::SB;
  uint64_t* raw_full = b_loaded + C::SB;
  uint64_t* raw_empty = raw_full + C::SRAW;
  uint64_t* acc_full = raw_empty + C::SRAW;
  uint64_t* acc_empty = acc_full + C::SACC;
  uint64_t* drain_bar = acc_empty + C::SACC;
  uint8_t* misc = smem + C::OFF_MISC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  TcSched* sched = reinterpret_cast<TcSched*>(misc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int kConvThreads = 128;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::SA; ++i) {
      mbar_init(&a_full[i], C::FP8 ? kConvThreads : 1);
      // the bound epilogue reads ||k|| from the key tile, so its 4 warps also release it
      mbar_init(&a_empty[i], C::BOUND ? 1 + C::NE : 1);
    }
    for (int i = 0; i < C::SB; ++i) {
      mbar_init(&b_full[i], C::FP8 ? kConvThreads : 1);
      mbar_init(&b_empty[i], 1);
      mbar_init(&b_loaded[i], 1);
    }
    for (int i = 0; i < C::SRAW; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kConvThreads);
    }
    for (int i = 0; i < C::SACC; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 32 * C::NE);
    }
    mbar_init(drain_bar, 1);
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
  volatile int no_abort_storage = 0;
  volatile int* no_abort = &no_abort_storage;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    TcUnits<C> u;
    u.init(args, s);
    int64_t cur_g = -1;
    uint32_t na = 0, nb = 0, nr = 0;
    while (u.valid()) {
      if (u.g != cur_g) {
        cur_g = u.g;
        const int bs = nb % C::SB;
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(&b_empty[bs], ((nb / C::SB) & 1) ^ 1, abort_flag);
          if (ok) {
            uint64_t* bar = C::FP8 ? &b_loaded[bs] : &b_full[bs];
            mbar_arrive_expect_tx(bar, C::B_BYTES);
            const int32_t y = (int32_t)(cur_g * C::N);
            tma_load_2d(sB + bs * C::B_BYTES, &tmap_q, bar, 0, y);
            tma_load_2d(sB + bs * C::B_BYTES + C::B_BYTES / 2, &tmap_q, bar, 64, y);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        ++nb;
      }
      // the ring slot this tile goes to, and its barrier
      uint8_t* dst;
      uint64_t* fbar;
      bool ok = true;
      if (C::FP8) {
        const int rs = nr % C::SRAW_MOD;
        if (lane == 0) ok = mbar_wait(&raw_empty[rs], ((nr / C::SRAW_MOD) & 1) ^ 1, abort_flag);
        dst = sRaw + rs * C::RAW_BYTES;
        fbar = &raw_full[rs];
      } else {
        const int as = na % C::SA;
        if (lane == 0) ok = mbar_wait(&a_empty[as], ((na / C::SA) & 1) ^ 1, abort_flag);
        dst = sA + as * C::A_BYTES;
        fbar = &a_full[as];
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const uint32_t tile_bytes = C::FP8 ? C::RAW_BYTES : C::A_BYTES;
      if (C::GATHER) {
        // lane l fetches tile rows 4l..4l+3 (list positions t*128 + 4l + i)
        const int64_t m = u.g;
        const int64_t base = tc_key_base(args, m);
        const int32_t cntm = args.cnt[m];
        const int32_t* lst = args.list + m * args.gld + u.t * 128;
        int32_t y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int pos = (int)(u.t * 128) + 4 * lane + i;
          int64_t id = pos < cntm ? (int64_t)lst[4 * lane + i] : 0;
          int64_t row = base + id;
          row = row < 0 ? 0 : (row >= args.p.n_keys ? args.p.n_keys - 1 : row);
          y[i] = (int32_t)row;
        }
        if (lane == 0) mbar_arrive_expect_tx(fbar, tile_bytes);
        __syncwarp();
        tma_gather4(dst + lane * 512, &tmap_k, fbar, 0, y[0], y[1], y[2], y[3]);
        if (!C::FP8) tma_gather4(dst + C::A_BYTES / 2 + lane * 512, &tmap_k, fbar, 64, y[0], y[1], y[2], y[3]);
      } else if (lane == 0) {
        const int32_t y = (int32_t)(tc_key_base(args, u.g) + u.t * 128);
        mbar_arrive_expect_tx(fbar, tile_bytes);
        tma_load_2d(dst, &tmap_k, fbar, 0, y);
        if (!C::FP8) tma_load_2d(dst + C::A_BYTES / 2, &tmap_k, fbar, 64, y);
      }
      __syncwarp();
      if (C::FP8) ++nr;
      else ++na;
      u.advance();
    }
    // drain: the last phase issued on every ring slot has landed
    if (lane == 0) {
      for (uint32_t i = 0; i < (uint32_t)C::SB && i < nb; ++i) {
        uint32_t j = nb - 1 - i;
        mbar_wait(C::FP8 ? &b_loaded[j % C::SB] : &b_full[j % C::SB], (j / C::SB) & 1, no_abort);
      }
      if (!C::FP8) {
        for (uint32_t i = 0; i < (uint32_t)C::SA && i < na; ++i) {
          uint32_t j = na - 1 - i;
          mbar_wait(&a_full[j % C::SA], (j / C::SA) & 1, no_abort);
        }
      }
      if constexpr (C::FP8) {
        for (uint32_t i = 0; i < (uint32_t)C::SRAW_MOD && i < nr; ++i) {
          uint32_t j = nr - 1 - i;
          mbar_wait(&raw_full[j % C::SRAW_MOD], (j / C::SRAW_MOD) & 1, no_abort);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(128, C::N, C::FP8 ? 0u : 1u);
      TcUnits<C> u;
      u.init(args, s);
      int64_t cur_g = -1;
      int cur_bs = 0;
      uint32_t na = 0, nb = 0, nacc = 0;
      bool issued = false;
      while (u.valid()) {
        if (u.g != cur_g) {
          cur_g = u.g;
          cur_bs = nb % C::SB;
          if (!mbar_wait(&b_full[cur_bs], (nb / C::SB) & 1, abort_flag)) break;
          ++nb;
        }
        const int as = na % C::SA;
        if (!mbar_wait(&a_full[as], (na / C::SA) & 1, abort_flag)) break;
        const int acc = nacc % C::SACC;
        if (!mbar_wait(&acc_empty[acc], ((nacc / C::SACC) & 1) ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + as * C::A_BYTES);
        const uint32_t b0 = smem_u32(sB + cur_bs * C::B_BYTES);
        const uint32_t d = tmem_base + (uint32_t)(acc * C::N);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t ao = a0 + (k >> 2) * (C::A_BYTES / 2) + (k & 3) * 32;
          const uint32_t bo = b0 + (k >> 2) * (C::B_BYTES / 2) + (k & 3) * 32;
          tc_mma_f16(d, smem_desc_sw128(ao), smem_desc_sw128(bo), idesc, k > 0 ? 1u : 0u);
        }
        issued = true;
        tc_commit(&a_empty[as]);
        tc_commit(&acc_full[acc]);
        ++na;
        ++nacc;
        const int64_t g_this = u.g;
        u.advance();
        if (!u.valid() || u.g != g_this) tc_commit(&b_empty[cur_bs]);
      }
      if (issued) {
        tc_commit(drain_bar);
        mbar_wait(drain_bar, 0, no_abort);
      }
    }
  } else if (warp >= 2 && warp < 2 + C::NE) {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                   // epilogue warp index
    const int quarter = warp & 3;              // TMEM lanes this warp may read
    const int qfirst = ew >> 2;                // first query of this warp in a tile
    constexpr int QSTEP = C::NE / 4;
    const int row_in_tile = quarter * 32 + lane;
    float* sW = sW_all + ew * C::N;
    int32_t* sLen = sLen_all + ew * C::NQ;
    int64_t* sBase = sBase_all + ew * C::NQ;
    float* sAux = sAux_all + ew * C::NQ * 2;
    TcUnits<C> u;
    u.init(args, s);
    int64_t cur_g = -1;
    uint32_t nacc = 0;
    while (u.valid()) {
      if (u.g != cur_g) {
        cur_g = u.g;
        __syncwarp();
        for (int i = lane; i < C::N; i += 32) {
          const int64_t m = cur_g * C::NQ + i / C::NCOL;
          float wv = 0.0f;
          if (m < args.p.M) wv = C::BOUND ? args.wfold[m * 32 + (i % 32)] : args.p.w[m * C::H + (i % C::H)];
          sW[i] = wv;
        }
        if (lane < C::NQ) {
          const int64_t m = cur_g * C::NQ + lane;
          int64_t off = 0;
          int len = 0;
          if (m < args.p.M) {
            if (C::GATHER) {
              len = args.cnt[m];
              off = tc_key_base(args, m);
            } else {
              row_extent(args.p, m, &off, &len);
            }
            if (args.row_mask && !args.row_mask[m]) len = 0;
          }
          sLen[lane] = len;
          sBase[lane] = off;
          if (C::BOUND) {
            sAux[2 * lane] = m < args.p.M ? args.coef[m] : 0.0f;
            sAux[2 * lane + 1] = m < args.p.M ? args.tau[m] : 0.0f;
          }
        }
        __syncwarp();
      }
      const int acc = nacc % C::SACC;
      const int key = (int)(u.t * 128) + row_in_tile;
      // FP8: fetch this key's dequantisation scale before waiting for the
      // accumulator, so the global load overlaps the wait (all queries of a
      // group read the same key sequence, so one scale serves them all)
      float kscale = 1.0f;
      if constexpr (C::FP8) {
        const int64_t m0 = cur_g * C::NQ + qfirst;
        if (m0 < args.p.M) {
          int64_t kid = key;
          if (C::GATHER) kid = key < sLen[qfirst] ? (int64_t)args.list[m0 * args.gld + key] : -1;
          const int64_t row = sBase[qfirst] + kid;
          if (kid >= 0 && row < args.p.n_keys) kscale = __ldg(args.p.key_scale + row);
        }
      }
      const bool got = mbar_wait(&acc_full[acc], (nacc / C::SACC) & 1, abort_flag);
      __syncwarp();                           // tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      float knorm = 0.0f;
      if (C::BOUND) {
        // ||k|| of this lane's key from the MMA-ready tile (128-byte swizzle), then release the tile
        const uint8_t* at = sA + (nacc % C::SA) * C::A_BYTES;
        float ss = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(at + h * (C::A_BYTES / 2) + row_in_tile * 128 +
                                                            ((c ^ (row_in_tile & 7)) << 4));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float lo, hi;
              if (C::FP8) {
                const __half2 h2 = *reinterpret_cast<const __half2*>(&w4[e]);
                lo = __low2float(h2);
                hi = __high2float(h2);
              } else {
                lo = __uint_as_float(w4[e] << 16);
                hi = __uint_as_float(w4[e] & 0xffff0000u);
              }
              ss = __fmaf_rn(lo, lo, ss);
              ss = __fmaf_rn(hi, hi, ss);
            }
          }
        }
        knorm = __fsqrt_ru(ss);
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_empty[nacc % C::SA]);
      }
#pragma unroll 1
      for (int qi = qfirst; qi < C::NQ; qi += QSTEP) {
        const int64_t m = cur_g * C::NQ + qi;
        if (m >= args.p.M) break;
        const uint32_t tcol = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * C::N + qi * C::NCOL);
        const float* wq = sW + qi * C::NCOL;
        const int len = sLen[qi];
        if (!C::BOUND) {
          float sc = 0.0f;
          constexpr int NCH = (C::H + 31) / 32;      // 32-column TMEM loads per query
          constexpr int CW = C::H < 32 ? C::H : 32;  // columns per load
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
          if (key < len) args.scores[m * args.ld + key] = C::FP8 ? sc * kscale : sc;
        } else {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tcol, v);
          tmem_ld_wait();
          const int R = args.R;
          float ub = 0.0f;
#pragma unroll
          for (int j = 0; j < 31; ++j)
            if (j < R) ub = __fmaf_rn(wq[j], fmaxf(__uint_as_float(v[j]), 0.0f), ub);
          ub = __fmaf_rn(sAux[2 * qi], knorm, ub);
          ub = ub - fmaxf(__uint_as_float(v[31]), 0.0f);
          bool is_cand = false;
          if (key < len) {
            if (C::FP8) ub = ub * kscale;
            const uint32_t* bits = args.seedbits + (args.seed_stride ? m * args.seed_stride : 0);
            const bool seed = (bits[key >> 5] >> (key & 31)) & 1u;
            is_cand = !seed && !(ub < sAux[2 * qi + 1]);
          }
          const unsigned mask = __ballot_sync(0xffffffffu, is_cand);
          if (mask) {
            int32_t basepos = 0;
            if (lane == 0) basepos = atomicAdd(&args.cand_cnt[m], __popc(mask));
            basepos = __shfl_sync(0xffffffffu, basepos, 0);
            if (lane == 0 && basepos + __popc(mask) > args.cap) atomicOr(&args.status[m], 2);
            if (is_cand) {
              const int64_t pos = basepos + __popc(mask & ((1u << lane) - 1u));
              if (pos < args.cap) args.cand[m * args.cap + pos] = key;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
      ++nacc;
      u.advance();
    }
  } else if (C::FP8) {
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - 32 * (2 + C::NE);   // 0..127
    TcUnits<C> u;
    u.init(args, s);
    int64_t cur_g = -1;
    uint32_t na = 0, nb = 0, nr = 0;
    while (u.valid()) {
      if (u.g != cur_g) {
        cur_g = u.g;
        const int bs = nb % C::SB;
        if (!mbar_wait(&b_loaded[bs], (nb / C::SB) & 1, abort_flag)) break;
        uint4* bp = reinterpret_cast<uint4*>(sB + bs * C::B_BYTES);
        for (int i = ct; i < C::B_BYTES / 16; i += kConvThreads) {
          uint4 v = bp[i];
          uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16);
            const float hi = __uint_as_float(w[j] & 0xffff0000u);
            __half2 h2 = __floats2half2_rn(lo, hi);
            w[j] = *reinterpret_cast<uint32_t*>(&h2);
          }
          bp[i] = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&b_full[bs]);
        ++nb;
      }
      const int rs = nr % C::SRAW_MOD;
      if (!mbar_wait(&raw_full[rs], (nr / C::SRAW_MOD) & 1, abort_flag)) break;
      const int as = na % C::SA;
      if (!mbar_wait(&a_empty[as], ((na / C::SA) & 1) ^ 1, abort_flag)) break;
      const uint8_t* src = sRaw + rs * C::RAW_BYTES;
      uint8_t* dst = sA + as * C::A_BYTES;
#pragma unroll 2
      for (int it = 0; it < 8; ++it) {
        const int item = it * kConvThreads + ct;   // (row r, 16-byte source chunk j)
        const int r = item >> 3, j = item & 7;
        const uint4 raw = *reinterpret_cast<const uint4*>(src + r * 128 + ((j ^ (r & 7)) << 4));
        const uint32_t* rw = reinterpret_cast<const uint32_t*>(&raw);
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t lo, hi;
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((unsigned short)(rw[q] & 0xffffu)));
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((unsigned short)(rw[q] >> 16)));
          o[2 * q] = lo;
          o[2 * q + 1] = hi;
        }
        // elements 16j..16j+15 of row r -> half j/4, 16-byte chunks 2j%8 and 2j%8+1
        uint8_t* hbase = dst + (j >> 2) * (C::A_BYTES / 2) + r * 128;
        const int c0 = (2 * j) & 7;
        *reinterpret_cast<uint4*>(hbase + ((c0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(hbase + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&raw_empty[rs]);
      mbar_arrive(&a_full[as]);
      ++nr;
      ++na;
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

// Launches one configuration.  B rows are a.p.q viewed as [M * NCOL, 128] bf16.
template <class C>
cudaError_t launch_tc(const TcArgs& a_in, cudaStream_t st) {
  TcArgs a = a_in;
  const idx_problem& p = a.p;
  if (p.M <= 0 || p.n_keys <= 0) return cudaSuccess;
  if (!C::GATHER && p.max_key_len <= 0) return cudaSuccess;
  if (p.n_keys >= ((int64_t)1 << 31) || p.M * C::NCOL >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  CUtensorMap tk, tq;
  bool ok;
  const uint32_t krows = C::GATHER ? 1u : 128u;     // gather4 wants a one-row box
  if (C::FP8)
    ok = make_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.keys, 128, (uint64_t)p.n_keys, 128, 128, krows);
  else
    ok = make_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.keys, 128, (uint64_t)p.n_keys, 256, 64, krows);
  ok = ok && make_tmap_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, 128, (uint64_t)(p.M * C::NCOL), 256, 64, C::N);
  if (!ok) return cudaErrorInvalidValue;
  a.G = (p.M + C::NQ - 1) / C::NQ;
  cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  score_tc_kernel<C><<<sm_count(), C::NTHREADS, C::SMEM_BYTES, st>>>(tk, tq, a);
  return cudaGetLastError();
}

}  // namespace idx
