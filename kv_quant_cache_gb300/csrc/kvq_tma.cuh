// kvq_tma.cuh -- the bulk-copy (TMA) staging primitives shared by the staged
// launch shapes of both operators: mbarrier set-up and bounded waits, 1-D
// bulk copies global -> shared with an L2 evict-first policy, the proxy
// fence, and the host-side helpers (pointer kind, per-device shared-memory
// opt-in).  Inline PTX for sm_103a.
#pragma once

#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {

// Polls of a stage barrier after which a warp of a staged launch shape stops
// staging and finishes its items from global memory; read at each launch
// (kvq_set_stage_wait_limit).  Defined in kvq_api.cu.
uint32_t stage_wait_limit();
uint32_t set_stage_wait_limit(uint32_t polls);

namespace tma {

// Stage-wait limits: a warp gives up staging after `stage_wait_limit()`
// polls or kWaitNs; the copies it still has in flight then get kDrainPolls
// polls or kDrainNs each.
constexpr uint64_t kWaitNs = 20000000;    // 20 ms
constexpr uint32_t kDrainPolls = 1u << 22;
constexpr uint64_t kDrainNs = 100000000;  // 100 ms

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes initialised barriers visible to the bulk-copy engine.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One arrival that also announces `bytes` of copies completing on the barrier.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
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

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Polls the completion of the barrier phase with parity `parity` at most
// `limit` times and for about `ns` nanoseconds at most (the clock is read
// every 64 polls); the result is the same on every lane of the warp.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint32_t limit,
                                               uint64_t ns) {
  bool done = limit > 0 && mbar_test(bar, parity);
  if (!done && limit > 1) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < limit; ++i) {
      if ((done = mbar_test(bar, parity))) break;
      if ((i & 63u) == 0 && global_ns() - t0 > ns) break;
    }
  }
  return __all_sync(kFullMask, done);
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Global -> shared bulk copy completing on `bar` (addresses 16-byte aligned,
// size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(__cvta_generic_to_global(src)), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// Orders this thread's earlier shared-memory accesses before later
// bulk-copy writes to the same stage.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- host side ----------------------------------------------------------------

// True for device memory (the only kind the bulk-copy engine is given).
inline bool device_memory(const void* ptr) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();  // a failed query is not sticky: clear it before the launch
    return false;
  }
  return attr.type == cudaMemoryTypeDevice;
}

// Opts `kernel` in to `smem` bytes of dynamic shared memory and counts its
// resident CTAs per SM, once per device (cached).
template <typename Kernel>
cudaError_t prepare(Kernel kernel, int threads, size_t smem, std::atomic<int>* cache,
                    int* per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *per_sm = v;
      return cudaSuccess;
    }
  }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  if (cached) cache[dev].store(n, std::memory_order_relaxed);
  *per_sm = n;
  return cudaSuccess;
}

}  // namespace tma
}  // namespace kvq
