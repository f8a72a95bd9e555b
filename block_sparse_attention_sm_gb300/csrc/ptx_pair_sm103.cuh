// Inline-PTX building blocks for kernels that run on a pair of CTAs in a
// thread-block cluster of two (sm_103a): cluster rank and barrier, shared
// addresses of the peer CTA, remote mbarrier arrivals and stores, and the
// two-SM (cta_group::2) forms of TMEM allocation, MMA, commit and TMA loads.
// Written from the public PTX ISA description of these instructions.
//
// In the two-SM form one thread of the even CTA (the "leader") issues an MMA
// that both SMs execute: each SM supplies half of the rows of A (its own
// shared memory or TMEM at the same address) and half of the columns of B
// (its own shared memory at the same address), and writes its own half of
// the rows of D into its own TMEM.  A commit can arrive on the mbarrier at
// the same offset in both CTAs (multicast).  A TMA load issued by either CTA
// into its own shared memory may signal the leader's mbarrier, so the leader
// sees one barrier complete when both halves of an operand have landed.
#pragma once
#include <cstdint>

#include "ptx_sm103.cuh"

namespace ssattn {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs: release this CTA's prior shared-memory writes
// and mbarrier initialisations to the cluster, then wait for the peer.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the object at shared::cta address `local` in
// the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t map_shared(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// Arrive (release at cluster scope) on an mbarrier given by its
// shared::cluster address: this CTA's or the peer's.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   bar_cluster_addr)
               : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Asynchronous 4-byte store into a CTA of the cluster that completes 4 bytes
// of transaction count on the mbarrier `bar_cluster_addr` of that CTA: the
// waiter that sees the barrier's phase complete sees the value.  Unlike a
// store followed by a cluster-scope release, the issuing thread does not wait
// for the store to be performed.
__device__ __forceinline__ void st_async_u32(uint32_t cluster_addr, uint32_t v,
                                             uint32_t bar_cluster_addr) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(
                   cluster_addr),
               "r"(v), "r"(bar_cluster_addr)
               : "memory");
}

// Test / wait with cluster-scope acquire: pairs with arrivals released at
// cluster scope by the peer CTA (so its prior stores are visible).
__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
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

// Bounded wait.  On expiry the wait raises this CTA's abort flag and the
// peer's (`peer_abort`: shared::cluster address of the peer's flag), so that
// every waiter of the pair gives up promptly.  CLUSTER selects a
// cluster-scope acquire, needed only where the phase was completed by the
// peer's release of data this thread then reads; barriers completed by
// tcgen05 commits or by this CTA's own threads use the CTA-scope form, which
// is much cheaper (a cluster-scope acquire or release costs a memory barrier).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_pair(uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag, uint32_t peer_abort) {
  auto test = [&]() { return CLUSTER ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity); };
  auto wait = [&]() { return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (test()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (wait()) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      st_cluster_u32(peer_abort, 1u);
      return false;
    }
  }
}

// Producer side of a named barrier: count this thread's arrival without
// waiting.  Memory operations before it are visible to the threads that
// complete the same phase with bar.sync.
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- tcgen05, two SMs
// Executed by one warp of EACH CTA of the pair: the allocation is made on
// both SMs' tensor memory and its address written to each CTA's `smem_dst`.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_dst)),
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

// D (+)= A * B over both SMs (M = 256: 128 rows per SM), A and B from each
// CTA's shared memory at the descriptors' addresses.
__device__ __forceinline__ void mma2_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same with A read from each SM's tensor memory.
__device__ __forceinline__ void mma2_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at `bar`'s offset in every CTA of `cta_mask` once
// all two-SM tcgen05 operations issued so far by this thread are done.
__device__ __forceinline__ void mma2_commit_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// 3-D tiled TMA load into this CTA's shared memory that completes its bytes
// on the mbarrier at shared::cluster address `bar_cluster_addr`, which may be
// the peer's (two-SM form).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster_addr, int c0, int c1,
                                                 int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

}  // namespace ssattn
