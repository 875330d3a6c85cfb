// kvq_tma.cuh -- the bulk-copy (TMA) staging primitives of the staged launch
// shapes: mbarrier set-up and bounded waits, 1-D bulk copies and tiled
// tensor-map copies global -> shared with an L2 evict-first policy, the proxy
// fence, and the host-side helpers (pointer kind, tensor-map encoding,
// per-device shared-memory opt-in).  Inline PTX for sm_103a.
#pragma once

#include <atomic>
#include <mutex>

#include <cuda.h>
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

// Tiled copy of the box at (c0, c1, c2) of a 3-D tensor map -> shared,
// completing on `bar`.  `tmap` is the map's address in parameter space
// (a __grid_constant__ kernel parameter).
__device__ __forceinline__ void tile_load_3d(uint32_t dst, const CUtensorMap* tmap, int c0,
                                             int c1, int c2, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(pol)
      : "memory");
}

// Orders this thread's earlier shared-memory accesses before later
// bulk-copy writes to the same stage.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- host side ----------------------------------------------------------------

// True for memory of the current device (the only kind the bulk-copy engine
// is given: neither host memory nor another GPU's).  A failed query's error
// is taken off the runtime's last-error state only if no earlier error was
// pending there, so an error of other work is never consumed.
inline bool device_memory(const void* ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const bool clean = cudaPeekAtLastError() == cudaSuccess;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    if (clean) cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeDevice && attr.device == dev;
}

// cuTensorMapEncodeTiled, fetched once from the driver through the runtime
// (no link against the driver library); nullptr if unavailable.
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiled encode_tiled() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    const bool clean = cudaPeekAtLastError() == cudaSuccess;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
    else if (clean)
      cudaGetLastError();
  });
  return fn;
}

// A 3-D bf16 tensor map: dims[0] contiguous elements, strides (bytes) of
// dims 1 and 2, box `box`; no swizzle (the box lands densely, row after row),
// out-of-range elements read as zero.  False if it cannot be encoded.
inline bool encode_bf16_3d(CUtensorMap* map, const void* base, const cuuint64_t dims[3],
                           const cuuint64_t strides[2], const cuuint32_t box[3]) {
  const EncodeTiled fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
