// kvq_launch.h -- internal host-side interface between the C ABI (kvq_api.cu)
// and the kernel launchers.  Not installed; callers use include/kvq.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace kvq {

struct QkArgs {
  void* qkv;
  const void* q_weight;
  const void* k_weight;
  const float* cos_sin;
  const int64_t* positions;
  int num_tokens;
  int num_heads_q, num_heads_k, num_heads_v;
  int head_dim, rotary_dim, is_neox;
  float eps;
  // bounds-checked launches (errors != nullptr): rows of cos_sin
  int64_t max_pos = 0;
  int* errors = nullptr;
};

struct Dsv4Args {
  const void* q;
  void* q_out;  // == q for the in-place operator
  const void* kv;
  const void* q_weight;
  const void* kv_weight;
  const float* cos_sin;
  const int64_t* positions;
  const int64_t* slot_mapping;
  uint8_t* kv_cache;
  int num_tokens;
  int num_heads;
  float eps;
  // bounds-checked launches (errors != nullptr): rows of cos_sin, cache slots
  int64_t max_pos = 0, num_slots = 0;
  int* errors = nullptr;
};

struct GatherArgs {
  const uint8_t* kv_cache;
  const int64_t* slots;
  void* out;
  int num_rows;
  // bounds-checked launches (errors != nullptr): cache slots
  int64_t num_slots = 0;
  int* errors = nullptr;
};

// A launch shape of one operator (an instantiation of one of its kernels).
struct LaunchConfig {
  const char* name;
};

extern const LaunchConfig kQkConfigs[];
extern const int kQkNumConfigs;
extern const LaunchConfig kDsv4Configs[];
extern const int kDsv4NumConfigs;

// Tuned kernel: head_dim 128, full-dimension NeoX rotation.
cudaError_t launch_qk_norm_rope(const QkArgs& a, int config, cudaStream_t stream);
// Every supported layout (head_dim 64/128/256, NeoX or GPT-J, partial), with
// fragments of frag = 4 or 8 dims per lane.
cudaError_t launch_qk_general(const QkArgs& a, bool small, int frag, cudaStream_t stream);
cudaError_t launch_dsv4(const Dsv4Args& a, int config, cudaStream_t stream);
cudaError_t launch_dsv4_gather(const GatherArgs& a, cudaStream_t stream);

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Programmatic dependent launch (kvq_set_programmatic_launch).  When on,
// kernels are launched with programmatic stream serialization: a kernel may
// be scheduled while the previous kernel on the stream is finishing, and
// every kernel of this library waits for that kernel's completion before its
// first memory access (grid_dependency_sync), so results and stream order are
// those of an ordinary launch.
bool programmatic_launch();

// Launches `kernel` with one by-value parameter block and returns the
// launch's own error.  A failed launch's error is taken off the runtime's
// last-error state (it is reported to the caller instead); after a successful
// launch that state is left alone, so an error still pending from earlier,
// unrelated work is not consumed here.
template <typename Params>
cudaError_t launch_kernel(void (*kernel)(Params), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic_launch() ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

constexpr int kMaxDevices = 64;

// CTAs of `kernel` that fit on one SM at `threads` threads per CTA (no
// dynamic shared memory), cached per device in `cache` -- one cache per
// kernel, kept by the launcher that owns it (the occupancy query is not free
// on every launch).
template <typename Kernel>
cudaError_t resident_ctas(Kernel kernel, int threads, std::atomic<int>* cache, int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *out = v;
      return cudaSuccess;
    }
  }
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0);
  if (e != cudaSuccess) return e;
  if (n < 1) n = 1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  *out = n;
  return cudaSuccess;
}

// First CTA of the last wave of a one-shot launch of `kernel` (grid CTAs of
// `threads` threads, no dynamic shared memory; occupancy cached in `cache`):
// the CTAs from there on let the next grid be scheduled
// (grid_dependency_sync).  0 if the whole grid is resident at once, or if the
// occupancy query fails.
template <typename Kernel>
int last_wave_start(Kernel kernel, int threads, int64_t grid, std::atomic<int>* cache) {
  int per_sm = 0;
  if (resident_ctas(kernel, threads, cache, &per_sm) != cudaSuccess) return 0;
  const int64_t start = grid - (int64_t)per_sm * device_sm_count();
  return start > 0 ? (int)start : 0;
}

}  // namespace kvq
