// kvq_launch.h -- internal host-side interface between the C ABI (kvq_api.cu)
// and the kernel launchers.  Not installed; callers use include/kvq.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

struct QkArgs {
  void* qkv;
  const void* q_weight;
  const void* k_weight;
  const float* cos_sin;
  const int64_t* positions;
  int num_tokens;
  int num_heads_q, num_heads_k, num_heads_v;
  float eps;
};

struct Dsv4Args {
  void* q;
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
};

// Launch shapes.  0 = small batch (one row per warp, narrow CTAs, widest
// spread over the SMs), 1 = token-tiled (several rows per warp, wide CTAs).
int qk_path(int64_t num_tokens, int num_rows_per_token);
cudaError_t launch_qk_norm_rope(const QkArgs& a, int path, cudaStream_t stream);
cudaError_t launch_dsv4(const Dsv4Args& a, int path, cudaStream_t stream);

}  // namespace kvq
