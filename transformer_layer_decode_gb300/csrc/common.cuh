// Device helpers shared by the decode kernels: bulk-copy (TMA) staging with
// mbarriers, programmatic dependent launch, bounded waits and bf16 unpacking.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace tld {

// Bounded waits: a wait that legitimately takes more than a few milliseconds
// means something is broken; the kernel then raises the error flag and leaves.
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

enum ErrBits : int {
  ERR_FULL_WAIT = 1,
  ERR_EMPTY_WAIT = 2,
  ERR_DRAIN = 4,
  ERR_SPLITS = 8,
  ERR_GRID_WAIT = 16,
  ERR_BOUNDS = 32,  // debug builds: an index check failed; err[1] holds the source line
  ERR_CLUSTER_WAIT = 64
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of `bar` to complete.  Gives up (returns false)
// once kWaitLimitNs of wall time have passed (measured on %globaltimer,
// whatever each try_wait's own suspension time is), after kWaitLimit tries, or
// as soon as *abort (an error flag some other wait already raised) is set.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const int* abort = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
      if (abort && *reinterpret_cast<const volatile int*>(abort)) return false;
    }
  }
  return false;
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 cache policies for bulk copies: the weight stream of the running kernel is
// read once (evict first); prefetched data of the next kernel should stay.
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

// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Ticket for the last-arrival pattern: release this thread's prior writes and
// acquire the other arrivals' writes in one atomic.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Programmatic dependent launch: wait for the preceding grid's completion and
// memory, and let the following grid start its prologue early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}


// Timeline probe of one launch (ns, %globaltimer): [0] first CTA start,
// [1] last CTA end, [2] / [3] first / last return from griddepcontrol.wait,
// [4] last CTA to receive its first stage, [5] / [6] first / last CTA to end
// its main loop, [7] first CTA end.
__device__ __forceinline__ void tl_mark_min(uint64_t* tl, int i) {
  if (tl) atomicMin(reinterpret_cast<unsigned long long*>(tl + i), (unsigned long long)globaltimer_ns());
}
__device__ __forceinline__ void tl_mark_max(uint64_t* tl, int i) {
  if (tl) atomicMax(reinterpret_cast<unsigned long long*>(tl + i), (unsigned long long)globaltimer_ns());
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- thread-block clusters (distributed shared memory) -------------------------
// Every non-exited thread of every CTA of the cluster arrives; shared-memory
// writes before the barrier are visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync_all() {
  __syncwarp();  // the .aligned forms want the whole warp converged
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Split form of the cluster barrier: arrive now (no ordering), wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  __syncwarp();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}

__device__ __forceinline__ float dsmem_ld(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ void dsmem_st(uint32_t a, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// Arrive on an mbarrier of a CTA of the cluster (address from dsmem_addr),
// releasing this thread's prior writes (and those ordered before it by a CTA
// barrier) at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait with cluster-scope acquire: the writes released by the other
// CTAs' arrivals are visible after it.  Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  const int* abort = nullptr) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i < kWaitLimit; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
      if (abort && *reinterpret_cast<const volatile int*>(abort)) return false;
    }
  }
  return false;
}

// Two bf16 packed in a 32-bit word -> two fp32 (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void raise_error(int* flag, int bits) {
  if (flag) atomicOr(flag, bits);
}

// Index checks of the debug build (TLD_DEBUG_CHECKS): a failed check raises
// ERR_BOUNDS, keeps the first failing source line in err[1] and returns false,
// and the caller skips the access.  Release builds compile every check to true.
__device__ __noinline__ inline bool bounds_failed(int* err, int line) {
  if (err) {
    atomicOr(err, ERR_BOUNDS);
    atomicCAS(err + 1, 0, line);
  }
  return false;
}
#ifdef TLD_DEBUG_CHECKS
#define TLD_IN_BOUNDS(cond, err) ((cond) ? true : ::tld::bounds_failed((err), __LINE__))
#else
#define TLD_IN_BOUNDS(cond, err) true
#endif

// ---- grid-wide synchronisation inside one launch ---------------------------------
// Only for launches whose CTAs are all resident at once (one CTA per SM, grid no
// larger than the SM count): every wait is bounded in wall time and by the error
// flag, so a CTA that never arrives costs a timeout and an error flag, not a hang.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Makes generic-proxy writes visible to later bulk copies (async proxy) of this thread.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Spins until *ctr >= target (bounded by wall time and by the error flag).
__device__ __forceinline__ bool spin_until(const int* ctr, int target, int* err) {
  if (ld_acquire_gpu(ctr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire_gpu(ctr) >= target) return true;
    if ((i & 63) == 0) {
      if (*reinterpret_cast<volatile int*>(err)) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        raise_error(err, ERR_GRID_WAIT);
        return false;
      }
    }
  }
}

// Grid barrier of the consumer threads (nthreads of each CTA, named barrier
// `bar_id`): every CTA adds one to *ctr once its consumers are done with the
// phase; all wait until the count reaches `target`.  The named barrier orders
// every consumer thread's writes before thread 0's release; thread 0's acquire
// orders the other CTAs' writes before every thread's reads after the second
// named barrier.
__device__ __forceinline__ void grid_sync(int* ctr, int target, int* err, int tid, int bar_id,
                                          int nthreads, uint64_t* tl = nullptr) {
  named_barrier(bar_id, nthreads);
  if (tid == 0) {
    tl_mark_min(tl, 0);
    red_release_gpu_add(ctr, 1);
    spin_until(ctr, target, err);
    tl_mark_min(tl, 2);
    tl_mark_max(tl, 3);
  }
  named_barrier(bar_id, nthreads);
}

}  // namespace tld
