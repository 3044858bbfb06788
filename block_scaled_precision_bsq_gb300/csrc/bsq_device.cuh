// bsq_device.cuh -- inline-PTX helpers for sm_103a: mbarriers with bounded waits, TMA
// (tensor and bulk copies), tcgen05 (TMEM allocation, block-scaled MMA, scale-factor copy,
// TMEM loads) and low-precision conversions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "bsq.h"

namespace bsq {

// Longest time any mbarrier wait may take before the kernel gives up (nanoseconds of
// %globaltimer). A healthy wait in these kernels lasts microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitSuspendHintNs = 20000;  // one suspended try_wait: at most 20 us

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// Index checks of the checked build (compiled with BSQ_DEVICE_CHECKS=1): an access whose computed
// index falls outside its buffer records BSQ_ERR_DEVICE_CHECK in the status word and is skipped
// (`if (in_bounds(...)) access`). In the normal build the test compiles to nothing.
#ifndef BSQ_DEVICE_CHECKS
#define BSQ_DEVICE_CHECKS 0
#endif
__device__ __forceinline__ bool in_bounds(bool ok, int* status) {
#if BSQ_DEVICE_CHECKS
  if (!ok) atomicCAS(status, 0, BSQ_ERR_DEVICE_CHECK);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}

__device__ __forceinline__ bool elect_lane0() { return (threadIdx.x & 31u) == 0u; }

// Programmatic dependent launch. A kernel launched with programmatic stream serialization
// may start while the previous kernel in the stream is still running; grid_dependency_wait()
// blocks until that kernel has completed and its memory operations are visible, so every
// global read of inputs and every global write must come after it. launch_dependents() lets
// the next kernel in the stream be launched (it waits the same way before touching memory).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// One lane of the (converged) warp, chosen by elect.sync. The warp's other lanes keep running the
// same loop, so addresses and descriptors computed there stay warp-uniform.
__device__ __forceinline__ bool elect_one_sync() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .b32 r;\n\t.reg .pred p;\n\telect.sync r|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ---------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: a waiting thread sleeps until the phase completes (or
// the hint expires) instead of spinning and taking issue slots from the working warps.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity), "r"(kWaitSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed. Gives up when `*abort` becomes
// non-zero (another role gave up) or after `limit_ns`; on a timeout it raises `*abort`,
// records BSQ_ERR_TIMEOUT in the device status word and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  int* status, uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(addr, parity)) return true;
    if ((it & 7u) == 0u) {
      if (abort != nullptr && *abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        if (abort != nullptr) *abort = 1;
        atomicCAS(status, 0, BSQ_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Whole-warp form of mbar_wait_bounded: every lane waits (bounded) and the warp agrees on the
// outcome, so a timeout seen by any lane sends the whole warp down the same path.
__device__ __forceinline__ bool mbar_wait_bounded_warp(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                                                       uint64_t limit_ns = kWaitLimitNs) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort, status, limit_ns)) != 0;
}

// Before a CTA that loads by TMA into a ring of `stages` buffers exits, every load it issued must
// have landed (a copy still in flight would write into shared memory a later CTA may own). The
// producer armed `armed` stages in ring order from stage 0, phase 0; for each stage this waits
// (bounded, ignoring the abort flag) for the phase of its last arming. Phases already completed
// return at once, so on the normal path this costs nothing.
__device__ __forceinline__ void wait_armed_stages(uint64_t* full_bar, int stages, int64_t armed, int* status,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  for (int s = 0; s < stages && s < armed; ++s) {
    const int64_t arms = (armed - s + stages - 1) / stages;  // times stage s was armed
    mbar_wait_bounded(&full_bar[s], static_cast<uint32_t>((arms - 1) & 1), nullptr, status, limit_ns);
  }
}

// ---------------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Contiguous global -> shared copy; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// 3-D tile load: with the view (128 bytes of a K chunk, rows, K chunks) one copy brings several
// 128-byte-swizzled K chunks of a row block at once (fewer, larger TMA operations).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 3-D tile load into this CTA's shared memory whose completion is signalled on the mbarrier of
// the pair's leader CTA (`leader_bar`: a shared address with the CTA-rank bit cleared; in a
// cluster, bit 24 of a CTA's shared addresses holds its rank).
__device__ __forceinline__ void tma_load_3d_to_leader(void* smem_dst, const void* tmap, uint32_t leader_bar, int32_t x,
                                                      int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(leader_bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// The same 3-D load with an L2 cache policy (createpolicy) on the global reads.
__device__ __forceinline__ void tma_load_3d_to_leader(void* smem_dst, const void* tmap, uint32_t leader_bar, int32_t x,
                                                      int32_t y, int32_t z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(leader_bar), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}
// 2-D form of tma_load_3d_to_leader.
__device__ __forceinline__ void tma_load_2d_to_leader(void* smem_dst, const void* tmap, uint32_t leader_bar, int32_t x,
                                                      int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(leader_bar), "r"(x), "r"(y)
      : "memory");
}
// The same 2-D load with an L2 cache policy (createpolicy) on the global reads.
__device__ __forceinline__ void tma_load_2d_to_leader(void* smem_dst, const void* tmap, uint32_t leader_bar, int32_t x,
                                                      int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(leader_bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
constexpr uint32_t kClusterRankBit = 1u << 24;

// L2 policy that keeps the lines it covers resident ahead of normally cached lines.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* smem_src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y)
               : "memory");
}

// 5-D tile store (coordinates innermost first).
__device__ __forceinline__ void tma_store_5d(const void* tmap, const void* smem_src, int32_t c0, int32_t c1,
                                             int32_t c2, int32_t c3, int32_t c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until at most N of this thread's committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make generic-proxy shared-memory writes visible to the async proxy (TMA store source).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_holder)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Copy a 32-row x 128-bit block from shared memory into TMEM, replicated into all four
// 32-lane quadrants: lane 32q + i, column j receives bytes [4j, 4j + 4) of row i.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading / stride byte
// offsets (16-byte units), version 1 at bit 46, swizzle mode at bits 61..63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle_mode & 7u) << 61;
  return d;
}
constexpr uint32_t kSwizzleNone = 0, kSwizzle128B = 2;

// Block-scaled MMA, A and B from shared memory, D and the scale factors in TMEM.
template <int KIND>
__device__ __forceinline__ void tc_mma_block_scaled(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                    uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate);

// KIND 1: kind::mxf8f6f4 (E4M3 x E4M3, one UE8M0 scale per 32 K)
template <>
__device__ __forceinline__ void tc_mma_block_scaled<1>(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
// KIND 2: kind::mxf4nvf4 with four E4M3 scales per 64 K (NVFP4)
template <>
__device__ __forceinline__ void tc_mma_block_scaled<2>(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
// KIND 3: kind::mxf4 with two UE8M0 scales per 64 K (MXFP4)
template <>
__device__ __forceinline__ void tc_mma_block_scaled<3>(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM cells: thread i receives row (lane) i, columns c..c+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------- CTA pairs
// Two CTAs of a (2, 1, 1) cluster cooperate on one tile: the 2-SM forms (.cta_group::2) of
// the tcgen05 instructions. All tcgen05 instructions of a kernel use the same cta_group.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Full cluster barrier (every thread of both CTAs), release/acquire at cluster scope.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster (a plain arrive: the data it stands for
// is ordered by the producer's own completion wait; a cluster-scope release here costs ~1 us).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_holder)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// Arrive on `bar` (same offset) in every CTA of `mask` once the pair's prior tcgen05 work is done.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}
// Issued by one thread of the leader CTA: each CTA's TMEM receives its own shared-memory bytes.
__device__ __forceinline__ void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// 2-SM block-scaled MMA (M = 256 across the pair): A rows and B columns split between the CTAs'
// shared memory at the same offsets, D and scale factors in each CTA's TMEM.
template <int KIND>
__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t acc);
template <>
__device__ __forceinline__ void tc_mma_pair<1>(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                               uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
template <>
__device__ __forceinline__ void tc_mma_pair<2>(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                               uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
template <>
__device__ __forceinline__ void tc_mma_pair<3>(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                               uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

// ---------------------------------------------------------------------------- conversions
// E4M3 code (sign bit ignored) -> its fp32 value, exact.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t E = (c >> 3) & 15u, m = c & 7u;
  if (E == 0u) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9, exact
  return __uint_as_float(((E + 120u) << 23) | (m << 20));
}

// Two fp32 -> two E4M3 codes (round to nearest even, saturate to +-448); `lo` lands in
// bits 0..7 of the result, `hi` in bits 8..15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 -> two e2m1 codes (round to nearest even, saturate to +-6); `lo` in bits 0..3.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Eight fp32 -> eight e2m1 codes packed in one word (element i in bits 4i..4i+3), same
// rounding as cvt_e2m1x2; the four code bytes are assembled with one vector move.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Four fp32 -> four E4M3 codes packed in one word (element i in byte i), same rounding as
// cvt_e4m3x2.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h0, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h1, %4, %3;\n\t"
      "mov.b32 %0, {h0, h1};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// ---------------------------------------------------------------------------- packed fp32 pairs
// Two fp32 values in one 64-bit operand (`lo` in bits 0..31) of the f32x2 instructions, each lane
// rounded to nearest even exactly like the scalar operation.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_splat(float v) { return f2(v, v); }

// ---------------------------------------------------------------------------- IEEE quotients
// NVFP4 divides every element of a block by one fp32 divisor d and rounds the IEEE quotient
// fp32(x / d). With r = fp32(1 / d) correctly rounded (computed once per divisor), the quotient
// follows from one multiply and two fused multiply-adds by Markstein's remainder step
// (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000 processor",
// IBM J. Res. Develop. 34(1), 1990: from a correctly rounded reciprocal and a quotient within an
// ulp, one exact remainder and one fused correction give the correctly rounded quotient):
//   q0 = fp32(x r),  e = q0 d - x (exact in one fma),  q = fp32(q0 - e r).
// The remainder is taken as q0 d - x rather than x - q0 d so that x = -0 keeps its sign.
// Valid while nothing overflows or underflows: d in [2^-92, 2^100) and |x| r below 2^100
// (markstein_ok); quotients far below the smallest value any code of the target format rounds
// away from zero (2^-10 for E4M3, 2^-3 for e2m1) can carry an underflowed remainder but still
// round to a zero code, exactly as the IEEE quotient does.
__device__ __forceinline__ float markstein_quotient(float x, float d, float r) {
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(q0, d, -x);
  return __fmaf_rn(-e, r, q0);
}
// True when markstein_quotient(x, d, r) is the IEEE quotient for every |x| <= xmax.
__device__ __forceinline__ bool markstein_ok(float d, float r, float xmax) {
  const uint32_t db = __float_as_uint(d);
  return db >= (35u << 23) && db < (227u << 23) && __fmul_rn(xmax, r) < 0x1p100f;
}

}  // namespace bsq
