// Thread-block-cluster helpers (inline PTX): the CTA's rank in its cluster,
// addresses in a peer CTA's shared memory, stores and mbarrier arrivals
// there, cluster-scope acquire waits and the cluster-wide barrier.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace mla {
namespace cl {

__device__ __forceinline__ uint32_t rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of `saddr` (a shared::cta address of this
// CTA's layout) in CTA `peer` of the cluster.
__device__ __forceinline__ uint32_t map(uint32_t saddr, uint32_t peer) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(peer));
  return r;
}

__device__ __forceinline__ void st_v4(uint32_t caddr, uint32_t a, uint32_t b, uint32_t c,
                                      uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(caddr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

// Asynchronous 16-byte store into a peer CTA's shared memory that counts its
// bytes on the peer's mbarrier (complete_tx): the peer sees the data once the
// barrier phase, armed there with expect_tx, completes.
__device__ __forceinline__ void st_async_v4(uint32_t caddr, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d, uint32_t bar_caddr) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          caddr),
      "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar_caddr)
      : "memory");
}

// Bulk copy (TMA engine) of `bytes` from this CTA's shared memory to a peer
// CTA's, counted on the peer's mbarrier (complete_tx). One thread issues it;
// `commit` groups it for wait_read.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst_caddr, uint32_t src_saddr,
                                             uint32_t bytes, uint32_t bar_caddr) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_caddr),
      "r"(src_saddr), "r"(bytes), "r"(bar_caddr)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed bulk groups still read their source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Arrive (relaxed, cluster scope) on an mbarrier given by its cluster address:
// no fence. For signalling that this thread's earlier shared-memory reads --
// whose values it has already used -- are done.
__device__ __forceinline__ void arrive_remote_relaxed(uint32_t bar_caddr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_caddr)
               : "memory");
}

// Arrive (release, cluster scope) on an mbarrier given by its cluster address.
__device__ __forceinline__ void arrive_remote(uint32_t bar_caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_caddr)
               : "memory");
}

// try_wait with cluster-scope acquire: data a peer CTA stored before its
// release arrival is visible once this returns true.
__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity) {
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

// Every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

}  // namespace cl
}  // namespace mla
