// Thread-block-cluster helpers: bulk copies into a peer CTA's shared memory
// (DSMEM), relaxed remote mbarrier arrivals, cluster-scope acquire waits, and
// the cluster barrier.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace metis {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

// Bulk copy (async proxy) of `bytes` from this CTA's shared memory into a peer
// CTA's shared memory, signalling complete_tx(bytes) on the peer's mbarrier.
// Addresses 16-byte aligned, bytes a multiple of 16.  The source must have been
// made visible to the async proxy (fence.proxy.async) by the threads that wrote it.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster_addr, uint32_t src_smem_addr, uint32_t bytes,
                                                  uint32_t cluster_bar_addr) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster_addr),
      "r"(src_smem_addr), "r"(bytes), "r"(cluster_bar_addr)
      : "memory");
}

// Relaxed arrive on an mbarrier of another CTA: no fence, so it does not wait
// for this thread's earlier memory operations (or bulk copies) to complete.  Use
// it only where the arrival orders nothing but reads that have already returned.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_bar_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar_addr) : "memory");
}

// try_wait with cluster-scope acquire: makes the peers' released writes visible.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
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

// 16-byte store into a peer CTA's shared memory (address from dsmem_map).
__device__ __forceinline__ void st_cluster_v4(uint32_t cluster_addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Asynchronous 16-byte store into a peer CTA's shared memory that signals
// complete_tx(16) on the peer's mbarrier `cluster_bar_addr` when it lands (the
// receiver arms the barrier with expect_tx for the bytes it awaits; a thread
// that sees the phase complete sees the data).  The sender does not wait.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t cluster_bar_addr) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   cluster_addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(cluster_bar_addr)
               : "memory");
}

// Arrive on an mbarrier of another CTA with release semantics at cluster scope:
// this thread's earlier stores into that CTA's shared memory are visible to a
// thread that observes the phase completing with an acquire.cluster wait.
__device__ __forceinline__ void mbar_arrive_remote_release(uint32_t cluster_bar_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar_addr) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace metis
