// sv_cluster.cuh -- thread-block-cluster primitives for sm_103a: the CTA's
// place in its cluster, the cluster barrier, and loads from another CTA's
// shared memory (distributed shared memory).
//
// A cluster of CTAs works on one logit row at a time, each CTA holding a
// contiguous slice of the vocabulary in its own shared memory; the CTAs
// combine their slices' statistics by reading each other's exchange
// records after a cluster barrier.  The hardware schedules a cluster's
// CTAs together, so the barrier never waits on a CTA that is not running.
#pragma once

#include "sv_device.cuh"

namespace sv {

__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Cluster barrier, every thread of every CTA of the cluster.  arrive has
// release semantics (this thread's shared-memory writes become visible to
// the cluster), wait has acquire semantics.
__device__ __forceinline__ void cl_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_sync() {
  cl_arrive();
  cl_wait();
}

// The shared::cluster address of `p` (an address in this CTA's shared
// memory) in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t cl_map(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ uint4 cl_ld_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t cl_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

}  // namespace sv

