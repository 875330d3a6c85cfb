// kvq_device.cuh -- device helpers shared by the sm_103a prologue kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

constexpr unsigned kFullMask = 0xffffffffu;

// Eight bf16 values packed in a 16-byte vector -> fp32.  A bf16 is the upper
// half of an IEEE binary32, so widening is a shift; word k holds elements
// 2k (low half) and 2k+1 (high half).
__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

// fp32 pair -> packed bf16x2, round to nearest even (low half = lo).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack_bf16x8(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                    pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

// Butterfly all-reduce over aligned groups of WIDTH lanes (WIDTH a power of 2).
template <int WIDTH>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
  return v;
}

template <int WIDTH>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
  return v;
}

// Programmatic dependent launch.  Every kernel starts by waiting until the
// grids it depends on have completed and their writes are visible (a no-op
// when it was launched the ordinary way).  One-shot grids then let the next
// grid on the stream be scheduled: it can start once their last wave runs.
// Persistent grids do not trigger: all their CTAs are resident from the
// start, and a dependent scheduled early would only take SM resources and
// wait (measured on GB300: a staged QK launch triggering once each warp had
// issued its last copy made the following DSV4 launch, and the step, 19 %
// slower; a DSV4 launch doing the same was neutral).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One-shot grids: wait as above, then let the next grid be scheduled -- but
// only from the CTAs of the grid's last wave (blockIdx.x >= trigger_from, the
// grid size minus the CTAs the GPU holds at once, computed on the host).  A
// dependent scheduled while earlier waves are still to come would take SM
// room from them (measured on GB300: a 32768-token one-shot QK launch
// followed by a persistent DSV4 launch ran 10 % slower when every CTA
// triggered at entry).  A grid of one wave triggers from every CTA.
__device__ __forceinline__ void grid_dependency_sync(int trigger_from) {
  grid_dependency_wait();
  if ((int)blockIdx.x >= trigger_from) launch_dependents();
}

// Streaming 16-byte accesses for data touched exactly once (evict-first).
__device__ __forceinline__ uint4 load_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void store_stream(void* p, const uint4& v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

}  // namespace kvq
