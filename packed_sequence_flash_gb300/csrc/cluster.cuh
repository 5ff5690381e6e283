// cluster.cuh -- inline-PTX wrappers for thread-block clusters on sm_103a:
// cluster ids, shared-memory addresses of the other CTAs (mapa), stores and
// mbarrier arrivals into them, cluster-scope phase tests and the cluster
// barrier. Only the kernels that run as clusters include it.
#pragma once

#include "common.cuh"

namespace psf {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address, in the cluster's shared window, of local shared address `a` in the
// CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t a, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(rank));
  return d;
}
// Every thread of every CTA of the cluster: release this CTA's prior memory
// operations, then wait until all threads of the cluster have arrived.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
// 16-byte store into another CTA's shared memory (cluster address `raddr`);
// its 16 bytes complete as transactions on that CTA's mbarrier at cluster
// address `rbar`.
__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint4 v, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(raddr),
      "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
      : "memory");
}
// Shared-memory matrix descriptor for a 64-byte-swizzled operand (atoms of
// 8 rows x 64 bytes): for a K-major operand `sbo` is the distance between
// 8-row groups; for an MN-major one `lbo` is the distance between 32-element
// MN blocks and `sbo` the distance between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)4 << 61;  // 64-byte swizzle
  return d;
}
// Arrive on another CTA's mbarrier (cluster address), releasing this thread's
// prior memory operations at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t rbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar) : "memory");
}
// Arrive on another CTA's mbarrier without ordering this thread's earlier
// memory operations: for a signal that only says "values this thread has
// already loaded into registers may be overwritten", which must not wait for
// the thread's own stores still in flight.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t rbar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar) : "memory");
}
// Phase tests with cluster-scope acquire, for barriers that other CTAs of the
// cluster arrive on or store against.
__device__ __forceinline__ bool mbar_test_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_sleep_cl(uint64_t* bar, uint32_t parity, uint32_t suspend_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}
// wait_bar with cluster-scope acquire (bounded in the same way).
__device__ __forceinline__ bool wait_bar_cl(uint64_t* bar, uint32_t parity, const Ctl& c) {
  if (mbar_test_cl(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_test_sleep_cl(bar, parity, 20000)) return true;
    if (*c.abort_flag) return false;
    if (globaltimer_ns() - t0 > c.limit_ns) {
      atomicCAS(c.status, 0, kStatusTimeout);
      *c.abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

}  // namespace psf
