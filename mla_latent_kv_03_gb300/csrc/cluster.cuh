// Thread-block-cluster helpers (inline PTX): the CTA's rank in its cluster,
// addresses in a peer CTA's shared memory, bulk copies and mbarrier arrivals
// into it, and the cluster-wide barrier.
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

// Bulk copy (TMA engine) of `bytes` from this CTA's shared memory to a peer
// CTA's, counted on the peer's mbarrier (complete_tx): the peer sees the data
// once that barrier's phase, armed there with expect_tx, completes. One
// thread issues it; `bulk_commit` groups it for `bulk_wait_read`.
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

// Every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

}  // namespace cl
}  // namespace mla
