// Inline-PTX helpers beyond ptx.cuh used by the two-CTA (cluster) MLA kernel:
// thread-block cluster addressing and barriers, stores and bulk copies into a peer
// CTA's shared memory counted on its mbarrier, cluster-scope mbarrier waits, 64-byte-swizzled
// shared-memory matrix descriptors, the tensor-memory-A form of tcgen05.mma and a
// 2-D TMA tile load.
#pragma once

#include "ptx.cuh"

namespace pda {
namespace ptx {

// ------------------------------------------------------------------ thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// All threads of all CTAs of the cluster; orders every CTA's earlier memory accesses
// (accesses to peers' shared memory included) before everyone's later ones.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16 bytes into a peer CTA's shared memory (cluster address); the store counts its
// bytes as completed transactions on the peer's mbarrier `rbar` (cluster address).
__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          raddr),
      "r"(a), "r"(b), "r"(c), "r"(d), "r"(rbar)
      : "memory");
}

// Arrive on an mbarrier of a peer CTA (cluster address), releasing this thread's earlier
// accesses at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t rbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar)
               : "memory");
}

// Arrive on an mbarrier of a peer CTA with no ordering of this thread's earlier memory
// accesses: for signalling that a buffer the peer writes has been read, without waiting
// for this thread's own outstanding stores to the peer (release semantics would). Each
// caller says how its reads of the buffer come before the arrive: acquire loads
// (ld_shared_v4_acquire), which keep every later operation after them, or loads whose
// values are consumed before a __syncwarp that precedes the one lane's arrive.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t rbar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar)
               : "memory");
}

// Like mbar_try_wait, acquiring at cluster scope (for phases completed by a peer CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// A shared-memory load with acquire semantics at cluster scope: no later memory operation
// of this thread (a relaxed remote arrive that tells the peer the buffer may be
// overwritten, in particular) is performed before this load.
__device__ __forceinline__ float4 ld_shared_v4_acquire(uint32_t saddr) {
  float4 v;
  asm volatile("ld.acquire.cluster.shared::cta.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(saddr)
               : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_shared_v4(uint32_t saddr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(saddr)
               : "memory");
  return v;
}

// Bulk copy (async proxy) of `bytes` (a multiple of 16) from this CTA's shared memory
// into a peer CTA's shared memory (cluster address); completion is counted as
// transaction bytes on the peer's mbarrier `rbar` (cluster address).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src_cta,
                                                  uint32_t bytes, uint32_t rbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src_cta), "r"(bytes), "r"(rbar)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's committed bulk copies have finished reading their sources.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's committed bulk copies have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t saddr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// ------------------------------------------------------------------ tcgen05 additions
// Shared-memory matrix descriptor with a 64-byte swizzle (rows of 32 16-bit elements);
// fields as in umma_desc_sw128, swizzle mode 4 in bits 61-63.
__device__ __forceinline__ uint64_t umma_desc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFF);
  d |= uint64_t((lbo >> 4) & 0x3FFF) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFF) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(4) << 61;
  return d;
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M x 16, two 16-bit elements per 32-bit column with
// the lower K index in the low half, row i in lane i) is read from tensor memory.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// Arrive once on the mbarrier at shared-memory offset `bar` of every CTA in `cta_mask`
// when all tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void umma_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(cta_mask)
      : "memory");
}

// 4 bytes into a peer CTA's shared memory, counted on the peer's mbarrier (cluster addresses).
__device__ __forceinline__ void st_async_b32(uint32_t raddr, uint32_t v, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr),
               "r"(v), "r"(rbar)
               : "memory");
}

// 2-D tiled load global -> shared; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar)),
      "l"(cache_policy)
      : "memory");
}

}  // namespace ptx
}  // namespace pda
