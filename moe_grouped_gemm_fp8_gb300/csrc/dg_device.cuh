// Device-side building blocks for sm_103a: mbarriers, TMA, tcgen05 (UMMA,
// TMEM), bounded waits and the device error word.  Written against the PTX
// ISA descriptions of these instructions; inline PTX only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dg_internal.h"

namespace dg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Records the first device-side condition of a launch: code in bits 0-7,
// site in bits 8-23, block index in bits 32-63.  Never traps.
__device__ __forceinline__ void record_error(unsigned long long* word, uint32_t code,
                                             uint32_t site) {
  unsigned long long v = (unsigned long long)(code & 0xFFu) |
                         ((unsigned long long)(site & 0xFFFFu) << 8) |
                         ((unsigned long long)blockIdx.x << 32);
  atomicCAS(word, 0ull, v);
}

// Device checks of the debug build (compiled with DG_DEBUG_CHECKS=1, the
// library libdg_debug.so): a violated bound records DG_ERR_DEVICE_CHECK with
// its site in the error word and never traps.  TMA loads outside a tensor
// zero-fill and TMA stores clip, so those accesses still happen; row stores
// the check rejects are skipped.  Compiled out of the release library.
#ifndef DG_DEBUG_CHECKS
#define DG_DEBUG_CHECKS 0
#endif
#define DG_CHECK(err, cond, site)                                             \
  do {                                                                        \
    if (DG_DEBUG_CHECKS && !(cond)) ::dg::record_error((err), DG_ERR_DEVICE_CHECK, (site)); \
  } while (0)

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete yet
// is suspended for at most HINT_NS nanoseconds before the test is repeated
// (HINT_NS = 0: the form without a hint, whose suspend limit is left to the
// hardware).  Measured on the single-CTA pipeline, a 32 ns limit shortens the
// producer / MMA hand-offs.
template <uint32_t HINT_NS>
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity) {
  if (HINT_NS == 0) return mbar_try_wait(bar, parity);
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(HINT_NS)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) when the shared abort flag is raised by another role, or
// after `timeout_ns`, or after a fixed iteration cap; in the two last cases
// it records DG_ERR_DEVICE_TIMEOUT with `site` and raises the abort flag.
// wait_bounded keeps this slow path out of line; kernels that move registers
// between warpgroups with setmaxnreg cannot call an out-of-line function (the
// register allocator rejects the call), so they inline wait_bounded_body.
template <uint32_t HINT_NS = 0>
__device__ __forceinline__ bool wait_bounded_body(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t timeout_ns, unsigned long long* err,
                                                  uint32_t site) {
  if (mbar_try_wait_hint<HINT_NS>(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_hint<HINT_NS>(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns || it >= (1u << 30)) {
        record_error(err, DG_ERR_DEVICE_TIMEOUT, site);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

template <uint32_t HINT_NS = 0>
static __device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns, unsigned long long* err,
                                          uint32_t site) {
  return wait_bounded_body<HINT_NS>(bar, parity, abort_flag, timeout_ns, err, site);
}

// ---------------------------------------------------------------- flags in global memory

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits until the word at `flag` (written by another CTA) is non-zero, with
// acquire semantics.  Bounded like wait_bounded: gives up when the abort flag
// is raised, or after `timeout_ns` (recording DG_ERR_DEVICE_TIMEOUT with
// `site` and raising the abort flag).  Inlined (usable under setmaxnreg).
__device__ __forceinline__ bool wait_flag_gpu(const uint32_t* flag, volatile int* abort_flag,
                                              uint64_t timeout_ns, unsigned long long* err,
                                              uint32_t site) {
  if (ld_acquire_gpu(flag) != 0u) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire_gpu(flag) != 0u) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns || it >= (1u << 28)) {
        record_error(err, DG_ERR_DEVICE_TIMEOUT, site);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- programmatic dependent launch

// Waits until the grids this launch depends on programmatically have completed
// and their memory writes are visible.  Without such a dependency (PDL off, or
// the previous work on the stream not launched by this library with PDL) it
// returns at once.  Every thread that reads global memory another kernel may
// have written executes it first.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the launches that depend on this grid start their own set-up (they
// still wait for this grid's completion before reading its outputs).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- proxies

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// TMA store of a 2-D box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until at most N bulk groups of this thread are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- tcgen05

// Allocation is warp-wide; the TMEM base address is written to smem `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives (once) on `bar` when every tcgen05 async operation issued so far by
// this thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), descriptor version 1 at bit 46, layout
// type in bits 61-63 (0 = no swizzle, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}

// K-major operand tile with rows of 128 bytes, 128-byte swizzle (as written by
// a TMA load with CU_TENSOR_MAP_SWIZZLE_128B): 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_kmajor_sw128(uint32_t saddr) {
  return smem_desc(saddr, 16, 1024, 2);
}

// MN-major operand tile with 128-byte swizzle, as written by TMA boxes of 128
// bytes (along M or N) x 128 rows (along K): a swizzle atom is 8 K rows of
// 128 bytes (1024 bytes, 8-row K groups 1024 bytes apart: SBO); atoms along
// the MN dimension are 16 KB apart (LBO: the next 128-column box).  Checked
// on the hardware with exact small-integer operands.
__device__ __forceinline__ uint64_t smem_desc_mnmajor_sw128(uint32_t saddr) {
  return smem_desc(saddr, 16384, 1024, 2);
}

// Instruction-descriptor bits marking A / B as MN-major ("transposed").
constexpr uint32_t kIdescMnMajorA = 1u << 15;
constexpr uint32_t kIdescMnMajorB = 1u << 16;

// 32 rows x 16 bytes, row r at byte 16 r, no swizzle (source of a
// 32x128b tcgen05.cp).  Core matrices (8 rows x 16 B) are 128 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sf_chunk(uint32_t saddr) {
  return smem_desc(saddr, 128, 128, 0);
}

// Copies a 32x128b chunk from shared memory into TMEM columns
// [taddr, taddr + 4) and repeats it in all four 32-lane quarters.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Block-scaled FP8 MMA (E4M3 x E4M3 -> FP32 in TMEM, UE8M0 scales read from
// TMEM, one scale per 32 K elements per row): D (+)= (A * sA) (B * sB)^T for a
// 128 x N x 32 step.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: E4M3 A and B
// (format code 0), both K-major, N >> 3 in bits 17-22, UE8M0 scale type
// (bit 23), M >> 4 in bits 24-28, scale-factor byte selectors for B (bits
// 4-5) and A (bits 29-30).
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3(uint32_t m, uint32_t n, uint32_t sfa_id,
                                                       uint32_t sfb_id) {
  return ((sfb_id & 3u) << 4) | (0u << 7) | (0u << 10) | ((n >> 3) << 17) | (1u << 23) |
         ((m >> 4) << 24) | ((sfa_id & 3u) << 29);
}

// 32 lanes x 32 columns of 32-bit TMEM cells into registers; thread t of the
// warp receives lane (quarter base + t), columns taddr .. taddr + 31.
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Waits for this thread's tcgen05.ld and ties the 32 destination registers to
// the wait, so no use of them can be scheduled before it.
__device__ __forceinline__ void tc_wait_ld_regs(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}


// ---------------------------------------------------------------- clusters / CTA pairs

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Whole-cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Whole-cluster barrier whose arrive carries no ordering but whose wait
// acquires: paired with fence_acq_rel_cluster() before it in the threads that
// have something to publish (release pattern), it orders only their writes.
__device__ __forceinline__ void cluster_arrive_relaxed_wait_acquire() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Orders this thread's earlier memory accesses (shared memory of other CTAs of
// the cluster included) before its later ones, at cluster scope.
__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// 16-byte store into the shared memory of a CTA of the cluster.
__device__ __forceinline__ void st_shared_cluster_v4(uint32_t cluster_addr, uint32_t a, uint32_t b,
                                                     uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Arrive on an mbarrier given by its cluster address (possibly the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait with cluster-scope acquire (for barriers other CTAs arrive on).
static __device__ __noinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                         volatile int* abort_flag,
                                                         uint64_t timeout_ns,
                                                         unsigned long long* err, uint32_t site) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns || it >= (1u << 30)) {
        record_error(err, DG_ERR_DEVICE_TIMEOUT, site);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// TMA loads whose completion is signalled on an mbarrier of either CTA of the
// pair (the leader's), given by its cluster address.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// tcgen05 on a CTA pair: the TMEM allocation is joint (one warp of each CTA
// executes it and both receive the same address); copies, MMAs and commits
// are issued by the leader CTA only.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Each CTA's 32x128b chunk (same shared-memory offset) into its own TMEM.
__device__ __forceinline__ void tc_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// 256 x N x 32 block-scaled MMA over the pair: A rows 0-127 from the leader's
// shared memory, 128-255 from the peer's; B rows split in halves the same
// way; D rows split likewise across the two TMEMs.  Every CTA's TMEM holds
// the A scales of its own rows and the B scales of all N rows.
__device__ __forceinline__ void tc_mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t sfa_tmem,
                                                 uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Arrives on the mbarrier at shared offset `bar` of both CTAs of the pair once
// every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

// Arrives on the mbarrier at shared offset `bar` of both CTAs of a 2-CTA
// cluster (single-CTA MMAs) once every tcgen05 operation issued so far by
// this thread has completed.
__device__ __forceinline__ void tc_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

// TMA load of a 2-D box into the shared memory of both CTAs of a 2-CTA
// cluster, at the same offset `dst` in each, counted (complete_tx) on the
// mbarrier at offset `bar` of each.
__device__ __forceinline__ void tma_load_2d_both(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "h"((uint16_t)3)
      : "memory");
}

// TMA load of a 3-D box into the shared memory of both CTAs of a 2-CTA
// cluster, at the same offset `dst` in each, counted (complete_tx) on the
// mbarrier at offset `bar` of each.
__device__ __forceinline__ void tma_load_3d_both(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "h"((uint16_t)3)
      : "memory");
}

// ---------------------------------------------------------------- numerics

// Two FP32 values -> two E4M3 codes (round to nearest even, saturating to the
// largest finite magnitude); `lo` lands in the low byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^e as an FP32 for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23)
                   : __uint_as_float(1u << (e + 149));
}

// Smallest integer e with 448 * 2^e >= amax, clamped to [-127, 127];
// amax == 0 (or NaN) gives 0.  448 = 1.75 * 2^8, so for a normal
// amax = f * 2^E (f in [1, 2)) the answer is E - 8, plus one when f > 1.75.
__device__ __forceinline__ int scale_exponent(float amax) {
  if (!(amax > 0.0f)) return 0;
  const uint32_t bits = __float_as_uint(amax);
  const int biased = (int)((bits >> 23) & 0xFFu);
  const uint32_t frac = bits & 0x7FFFFFu;
  int e;
  if (biased == 0) e = -127;          // subnormal amax: 448 * 2^-127 already exceeds it
  else if (biased == 255) e = 127;    // infinity
  else e = biased - 127 - 8 + (frac > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// x * 2^-e exactly (both factors normal; the product can only lose bits when
// it falls below 2^-126, far under half the smallest E4M3 subnormal).
__device__ __forceinline__ float scale_down(float x, int e) {
  const int h = -e / 2;
  return (x * pow2f(h)) * pow2f(-e - h);
}

}  // namespace dg
