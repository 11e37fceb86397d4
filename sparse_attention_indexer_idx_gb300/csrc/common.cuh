// Shared device helpers for the indexer kernels (sm_103a).
//
// * ordered keys: fp32 scores mapped to uint32 so that unsigned comparison is
//   the float order (after -0.0 -> +0.0), used by every top-K in the library;
// * bounded waits: every spin on an mbarrier gives up after a time limit,
//   records the failure in a device-global error word and tells the other
//   warps of the CTA to stop, so a broken pipeline returns instead of hanging;
// * thin inline-PTX wrappers for mbarriers, TMA (cp.async.bulk.tensor) and the
//   5th-generation tensor core (tcgen05 alloc / mma / commit / ld).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace idx {

// ----------------------------------------------------------------- errors --
// Device-side error word: 0 = clean.  Set (atomicOr) by kernels that hit a
// bounded wait's limit or an internal inconsistency; read and cleared by the
// host through idx_device_error().
enum : uint32_t {
  DEVERR_WAIT_TIMEOUT = 1u << 0,
  DEVERR_BAD_ROW = 1u << 1,
  DEVERR_CAPACITY = 1u << 2,
};
// Each translation unit has its own word (the library is compiled without
// relocatable device code); every unit registers a host-side reader at load
// time and idx_device_error() ORs them together.
void register_error_word(uint32_t (*take)());
}  // namespace idx

static __device__ uint32_t g_device_error = 0;

static uint32_t idx_take_unit_error() {
  uint32_t v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  cudaMemcpyToSymbol(g_device_error, &z, sizeof(z));
  return v;
}
static struct IdxErrorWordRegistrar {
  IdxErrorWordRegistrar() { idx::register_error_word(&idx_take_unit_error); }
} idx_error_word_registrar;

namespace idx {

// Default limit of a single mbarrier wait, in globaltimer nanoseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// Setter of this translation unit's pipeline wait limit (see idx_set_wait_limit_ns).
void register_wait_limit_setter(cudaError_t (*set)(uint64_t));
}  // namespace idx

// The pipeline wait limit of the kernels of this translation unit (one copy per
// unit, like the error word); idx_set_wait_limit_ns() sets every copy.
static __device__ uint64_t g_wait_limit_ns = idx::kWaitLimitNs;

static cudaError_t idx_set_unit_wait_limit(uint64_t ns) {
  return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns));
}
static struct IdxWaitLimitRegistrar {
  IdxWaitLimitRegistrar() { idx::register_wait_limit_setter(&idx_set_unit_wait_limit); }
} idx_wait_limit_registrar;

namespace idx {

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------ ordered keys --
// Score -> key: larger score <=> larger key.  -0.0 is folded onto +0.0 first
// (x + 0.0f), so the two zeros are one key.  Inputs are assumed finite.
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}
// Ids rank ascending: smaller id <=> larger tie key.
__device__ __forceinline__ uint32_t id_key(int32_t id) { return 0xffffffffu - (uint32_t)id; }
__device__ __forceinline__ int32_t key_id(uint32_t k) { return (int32_t)(0xffffffffu - k); }

// ---------------------------------------------------------------- mbarrier --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Same test, but a thread whose phase is not complete may sleep until it
// completes or `hint_ns` nanoseconds pass (so a waiting warp takes no issue
// slots from the warps that work).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Bounded pipeline wait: returns false (and flags the CTA and the device) when
// the phase did not complete within the unit's wait limit (g_wait_limit_ns,
// 2 s unless the host set another) or another warp already aborted.
// The limit is checked before every sleep, so a limit of 0 gives up at the
// first wait whose phase is not already complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t limit = *(volatile uint64_t*)&g_wait_limit_ns;
  const uint64_t t0 = global_ns();
  while (true) {
    if (*abort_flag) return false;
    if (global_ns() - t0 >= limit) {
      *abort_flag = 1;
      atomicOr(&g_device_error, DEVERR_WAIT_TIMEOUT);
      return false;
    }
    if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
  }
}
// Drain wait at the end of a kernel (copies and MMAs this thread issued that
// must land before the CTA exits): always the fixed 2 s limit, whatever the
// pipeline limit, so that an aborted CTA still waits for its work in flight.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_device_error, DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// Bulk prefetch of [src, src + bytes) into L2 (src 16-byte aligned, bytes a
// multiple of 16): a hint, no data is returned.
__device__ __forceinline__ void l2_prefetch_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ------------------------------------------------------------------ tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Packed fp32 pairs (low half, high half) and the packed fused multiply-add:
// each half is one IEEE fma rounded once, exactly as fmaf on that half.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float* lo, float* hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(*lo), "=f"(*hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (A and B both bf16 or both f16).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 4-byte asynchronous global -> shared copy (both addresses 4-byte aligned).
__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
// 16-byte asynchronous global -> shared copy through L2 (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's committed cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy accesses (TMA, tcgen05.mma operands).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Arrive on `bar` (counted against its expected arrivals) once every cp.async
// this thread issued so far has completed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4 (formats from the instruction descriptor).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::tf32 (32-bit operands read as tf32).
__device__ __forceinline__ void tc_mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (base lane + i), columns [col, col+32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 16 consecutive 32-bit columns (r[0..15]).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 32 lanes x 1 32-bit column.
__device__ __forceinline__ uint32_t tmem_ld_32x32b_x1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
  return r;
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms of 1024 bytes (stride
// between atoms = 1024 B).  `addr` must lie in a 1024-byte aligned tile; moving
// along K inside the 128-byte row is done by adding the byte offset to addr.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3ffffu) >> 4);          // start address
  d |= (uint64_t)(16u >> 4) << 16;                  // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset: one 8-row atom
  d |= (uint64_t)1 << 46;                           // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                           // swizzle mode: 128 B
  return d;
}

// Instruction descriptor, fp32 accumulate, A and B K-major.  ab_type: for
// kind::f16 0 = f16, 1 = bf16; for kind::tf32 2 = tf32; for kind::f8f6f4
// 0 = e4m3 (same bit layout).
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N, uint32_t ab_type) {
  return (1u << 4)                 // D format f32
         | (ab_type << 7)          // A format
         | (ab_type << 10)         // B format
         | ((N >> 3) << 17)        // N >> 3
         | ((M >> 4) << 24);       // M >> 4
}

}  // namespace idx
