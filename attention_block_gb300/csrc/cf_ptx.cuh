// cf_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, TMA tensor
// loads, distributed-shared-memory (DSMEM) addressing and asynchronous
// remote stores, cluster barriers, and bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cf_params.h"

namespace cf {

// A wait that has not completed after this many SM cycles (about one second
// at the GB300 boost clock) gives up, sets kDevErrTimeout and returns, so a
// lost transaction can never hang the GPU.
constexpr long long kWaitLimitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier (every non-exited thread of every CTA must call it,
// warp-converged).  Release/acquire orders shared-memory traffic across it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Cluster barrier before the CTAs exit: no CTA leaves while a peer may still
// access its shared memory.  Every remote access has completed by then (each
// pushed store was waited for by its receiver, each pulled load was consumed
// by its issuer before the issuer arrives), so the arrival needs no release
// ordering, which would wait for the thread's outstanding global stores.
__device__ __forceinline__ void cluster_sync_exit() {
  asm volatile(
      "barrier.cluster.arrive.relaxed.aligned;\n\t"
      "barrier.cluster.wait.aligned;" ::: "memory");
}

// Named barrier among `nthreads` threads (a multiple of 32) with id `id`.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------- mbarriers --
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// `count` arrivals at once (the phase completes when the expected count is
// reached, so arrivals still outstanding keep it open).
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cta(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar,
                                                      uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase with the given parity.  On expiry (after
// `limit` SM cycles) it records kDevErrTimeout and returns false; once any
// CTA has recorded a timeout the other waits give up quickly, so the whole
// grid drains instead of hanging.
template <bool kCluster>
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            int* errflag, long long limit) {
  const long long t0 = clock64();
  for (uint32_t spins = 1;; ++spins) {
    bool ok = kCluster ? mbar_try_wait_cluster(bar, parity)
                       : mbar_try_wait_cta(bar, parity);
    if (ok) return true;
    if ((spins & 1023u) == 0) {
      if (*reinterpret_cast<volatile int*>(errflag) & kDevErrTimeout) return false;
      if (clock64() - t0 > limit) {
        atomicOr(errflag, kDevErrTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          int* errflag) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cta(a, parity)) return true;
  return mbar_wait_slow<false>(a, parity, errflag, kWaitLimitCycles);
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  int* errflag,
                                                  long long limit = kWaitLimitCycles) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cluster(a, parity)) return true;
  return mbar_wait_slow<true>(a, parity, errflag, limit);
}

// Bounded wait until the global counter reaches `target` (blocks of the same,
// fully resident grid are the only writers).  On expiry it records
// kDevErrTimeout and returns false.
static __device__ __noinline__ bool wait_count_at_least(const int* ctr, int target, int* errflag) {
  const long long t0 = clock64();
  for (uint32_t spins = 1;; ++spins) {
    if (*reinterpret_cast<const volatile int*>(ctr) >= target) return true;
    if ((spins & 255u) == 0) {
      if (*reinterpret_cast<volatile int*>(errflag) & kDevErrTimeout) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        atomicOr(errflag, kDevErrTimeout);
        return false;
      }
    }
    __nanosleep(32);
  }
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's async-proxy global-memory accesses (bulk copies and
// reductions it has waited for) with its later generic-proxy accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Tiled tensor reduction (add, in the tensor map's element type) of a box in
// this CTA's shared memory into global memory, tracked by the issuing
// thread's bulk async-group.  Both coordinates are non-negative and the
// innermost one is a multiple of 16 bytes (host-checked layouts); elements
// outside the tensor map are not written.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* tm, int x, int y,
                                                  const void* src) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];"
      ::"l"(tm), "r"(x), "r"(y), "r"(smem_u32(src))
      : "memory");
}

// Closes this thread's current bulk async-group.
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every bulk async-group of this thread is complete (the writes
// to global memory performed, not only the shared-memory reads).
__device__ __forceinline__ void bulk_wait_group_0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------ TMA loads --
// Contiguous bulk copy global -> this CTA's shared memory of `bytes` bytes
// (both addresses 16-byte aligned, bytes a multiple of 16), completing on
// `bar` with complete_tx of `bytes`.
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Tiled tensor copies global -> this CTA's shared memory, completing on `bar`
// with complete_tx of the box's byte count.  The innermost coordinate x is
// always a multiple of 16 bytes (host-checked layouts).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm,
                                            int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* tm,
                                            int x, int y, int z, int w,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2-only prefetch of one tensor box (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* tm, int x, int y,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.2d.L2.global.tile.L2::cache_hint [%0, {%1, %2}], %3;" ::"l"(tm),
      "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* tm, int x, int y, int z, int w,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.4d.L2.global.tile.L2::cache_hint [%0, {%1, %2, %3, %4}], %5;" ::"l"(
          tm),
      "r"(x), "r"(y), "r"(z), "r"(w), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}

// ----------------------------------------------------------------- DSMEM --
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// Asynchronous 8- or 16-byte store into a remote CTA's shared memory that
// signals the remote mbarrier `rbar` with complete_tx of its byte count.
__device__ __forceinline__ void st_async_v2(uint32_t raddr, float2 v, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
          raddr),
      "f"(v.x), "f"(v.y), "r"(rbar)
      : "memory");
}
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float4 v, uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          raddr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(rbar)
      : "memory");
}

// Arrive on the mbarrier at cluster shared address `rbar` (usually another
// CTA's) with release semantics at cluster scope: this thread's earlier
// memory operations, and those it has observed, are visible to a thread
// that then completes an acquire wait on that barrier.
__device__ __forceinline__ void mbar_remote_arrive(uint32_t rbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar)
               : "memory");
}

// Release fence at cluster scope restricted to shared::cta accesses: orders
// this thread's earlier shared-memory writes, and those it has observed
// through a CTA barrier, before its later relaxed arrivals on peers'
// mbarriers (an acquiring wait on such a barrier then sees the writes).
// The unrestricted release also waits for the thread's other memory traffic.
__device__ __forceinline__ void fence_release_smem_cluster() {
  asm volatile("fence.release.sync_restrict::shared::cta.cluster;" ::: "memory");
}

// Relaxed arrival on the mbarrier at cluster shared address `rbar`; pair with
// fence_release_smem_cluster() for release ordering.
__device__ __forceinline__ void mbar_remote_arrive_relaxed(uint32_t rbar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar)
               : "memory");
}

// 16-byte loads from (possibly another CTA's) shared memory at a cluster
// shared address.
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint4 ld_dsmem_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

}  // namespace cf
