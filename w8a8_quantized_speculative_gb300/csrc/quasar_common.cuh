// Shared device/host helpers for libquasar (sm_103a).
//
// Device side: thin inline-PTX wrappers for mbarrier, TMA bulk-tensor loads,
// tcgen05 (TMEM alloc / MMA / ld / st / commit) and bounded waits.  Every
// wait in this library is bounded: after the configured limit it records a
// site code in the library's error word and returns false, and the caller
// unwinds without trapping.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/quasar.h"

#define QUASAR_DEVICE_INLINE __device__ __forceinline__

namespace quasar {

// ---------------------------------------------------------------- host side

// Library error word and wait limit, owned by quasar_capi.cu.
unsigned int* device_error_word();          // device address for the current device, or nullptr
unsigned long long wait_limit_ns();
int sm_count();                             // SMs of the current device (cached)
quasar_status_t cuda_status(cudaError_t e); // maps a CUDA error to a status

// 2-D tensor map over a row-major uint8 matrix [outer][inner] (row stride =
// inner bytes, a multiple of 16), 128B-swizzled boxes of box_outer rows x
// box_inner bytes; out-of-range elements read as zero.
bool encode_2d_u8(CUtensorMap* map, const void* base, int inner, int outer, int box_inner, int box_outer);

// 2-D tensor map over a row-major BF16 matrix [outer][inner] whose rows are
// `ld` elements apart (ld * 2 a multiple of 16 bytes), 128B-swizzled boxes of
// box_outer rows x box_inner elements (box_inner * 2 <= 128); out-of-range
// elements read as zero.
bool encode_2d_bf16(CUtensorMap* map, const void* base, int inner, int outer, long long ld, int box_inner,
                    int box_outer);

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Error site codes recorded in the device error word (low 16 bits = site,
// high 16 bits = block index modulo 65536, for debugging).
enum : unsigned int {
  SITE_GEMM_FULL1 = 1,
  SITE_GEMM_EMPTY1 = 2,
  SITE_GEMM_FULL2 = 3,
  SITE_GEMM_EMPTY2 = 4,
  SITE_GEMM_ACCFULL = 5,
  SITE_GEMM_ACCEMPTY = 6,
  SITE_GEMM_DRAIN = 7,
  SITE_SKINNY_FULL = 8,
  SITE_SKINNY_EMPTY = 9,
  SITE_SKINNY_DRAIN = 10,
  SITE_SKINNY_ROWS = 11,
  SITE_SELFTEST = 12,
  SITE_LMH_FULL = 13,
  SITE_LMH_EMPTY = 14,
  SITE_LMH_ACCFULL = 15,
  SITE_LMH_ACCFREE = 16,
  SITE_LMH_DRAIN = 17,
};

// ---------------------------------------------------------------- device side

QUASAR_DEVICE_INLINE uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

QUASAR_DEVICE_INLINE unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

QUASAR_DEVICE_INLINE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

QUASAR_DEVICE_INLINE void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

QUASAR_DEVICE_INLINE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

QUASAR_DEVICE_INLINE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

QUASAR_DEVICE_INLINE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on the phase with the given parity.  Gives up when the CTA's
// abort flag is raised by another role, or after `limit_ns`; in the latter
// case it raises the abort flag and records `site` in the error word.
QUASAR_DEVICE_INLINE bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                    unsigned int* err, unsigned int site, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        if (err) atomicCAS(err, 0u, site | ((blockIdx.x & 0xFFFFu) << 16));
        return false;
      }
    }
  }
}

// 2-D TMA tile load into shared memory, completing on `bar` (tx bytes).
QUASAR_DEVICE_INLINE void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 1-D bulk copy global -> shared memory, completing on `bar` (tx bytes).
// Both addresses 16-byte aligned, size a multiple of 16.
QUASAR_DEVICE_INLINE void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// independent prologue now / wait until the previous kernel's writes are
// visible.  Both are no-ops for a launch without the PDL attribute.
QUASAR_DEVICE_INLINE void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
QUASAR_DEVICE_INLINE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named-barrier synchronisation of `count` threads (whole warps) that also
// returns the OR of every participant's `pred`; involves no memory access.
QUASAR_DEVICE_INLINE bool named_barrier_or(int id, int count, uint32_t pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\t"
      "setp.ne.b32 pin, %1, 0;\n\t"
      "barrier.red.or.pred pout, %2, %3, pin;\n\t"
      "selp.u32 %0, 1, 0, pout;\n\t}"
      : "=r"(out)
      : "r"(pred), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

QUASAR_DEVICE_INLINE uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

QUASAR_DEVICE_INLINE uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

QUASAR_DEVICE_INLINE void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

QUASAR_DEVICE_INLINE void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- tcgen05 -----------------------------------------------------------------

QUASAR_DEVICE_INLINE void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

QUASAR_DEVICE_INLINE void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

QUASAR_DEVICE_INLINE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

QUASAR_DEVICE_INLINE void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

QUASAR_DEVICE_INLINE void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

QUASAR_DEVICE_INLINE void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16 (fp16 operands, fp32 accumulate).
QUASAR_DEVICE_INLINE void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

QUASAR_DEVICE_INLINE void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
QUASAR_DEVICE_INLINE void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Store 32 consecutive 32-bit columns of this warp's 32 TMEM lanes.
QUASAR_DEVICE_INLINE void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Store 16 consecutive 32-bit columns of this warp's 32 TMEM lanes.
QUASAR_DEVICE_INLINE void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Load 4 consecutive 32-bit columns of this warp's 32 TMEM lanes.
QUASAR_DEVICE_INLINE void tmem_ld4(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}

// Load 8 consecutive 32-bit columns of this warp's 32 TMEM lanes.
QUASAR_DEVICE_INLINE void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

// Load 16 consecutive 32-bit columns of this warp's 32 TMEM lanes.
QUASAR_DEVICE_INLINE void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Load 32 consecutive 32-bit columns of this warp's 32 TMEM lanes.
QUASAR_DEVICE_INLINE void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Per-warpgroup register budget (every warp of a warpgroup executes these
// together).  `dec` returns registers to the CTA's pool, `inc` waits until the
// pool can grant the increase: a split must never ask for more than the
// warpgroups give back, or the increase waits forever.
template <int N>
QUASAR_DEVICE_INLINE void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
QUASAR_DEVICE_INLINE void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// ---- thread-block clusters ------------------------------------------------------

QUASAR_DEVICE_INLINE uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

QUASAR_DEVICE_INLINE uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

// Cluster-wide barrier of every thread of every CTA in the cluster
// (warp-converged callers only): release on arrive, acquire on wait, so the
// shared-memory writes before it are visible to every CTA after it.
QUASAR_DEVICE_INLINE void cluster_sync_full() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same barrier ordering execution only: no CTA passes before every
// thread of the cluster has arrived (remote loads issued before it have
// returned their values by then), without waiting for this thread's global
// stores to become visible.
QUASAR_DEVICE_INLINE void cluster_sync_exec() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// Split form of cluster_sync_exec: arrive now, wait later.
QUASAR_DEVICE_INLINE void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
QUASAR_DEVICE_INLINE void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Address of the same shared-memory offset in cluster CTA `rank`.
QUASAR_DEVICE_INLINE uint32_t map_to_rank(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  return remote;
}

// ---- bit helpers ---------------------------------------------------------------

// Four signed bytes -> two fp16x2 words, exactly.  Each byte b is re-biased
// to b + 128 in [0, 255] and placed in the low mantissa byte of the fp16
// number 1024 + (b + 128) (exponent field 0x64: ulp 1 on [1024, 2048));
// subtracting 1152 = 1024 + 128 leaves b.  Integer-valued fp16 arithmetic
// in this range is exact.
QUASAR_DEVICE_INLINE void u8x4_to_f16x4(uint32_t u, uint32_t& lo, uint32_t& hi);
QUASAR_DEVICE_INLINE void s8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  u8x4_to_f16x4(w ^ 0x80808080u, lo, hi);
}

// Four bytes holding code + 128 (code in [-128, 127]) -> two fp16x2 words
// holding the codes, exactly (same construction as above without the bias
// flip).
QUASAR_DEVICE_INLINE void u8x4_to_f16x4(uint32_t u, uint32_t& lo, uint32_t& hi) {
  uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);  // bytes: u0, 0x64, u1, 0x64
  uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);  // bytes: u2, 0x64, u3, 0x64
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// Four bytes, each holding a 4-bit code + 8 (code in [-8, 7]) -> two fp16x2
// words holding the codes exactly: the byte goes into the low mantissa of
// 1024 (0x6400) and 1032 = 1024 + 8 is subtracted.
QUASAR_DEVICE_INLINE void n4x4_to_f16x4(uint32_t u, uint32_t& lo, uint32_t& hi) {
  uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
  uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

}  // namespace quasar
