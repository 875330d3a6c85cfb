// kvq_api.cu -- the C ABI (include/kvq.h): host-side validation, launch-shape
// dispatch and launch on the caller's stream.  No allocation, no sync.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "kvq.h"
#include "kvq_launch.h"
#include "kvq_qk_bulk.h"
#include "kvq_tma.cuh"

namespace {

// Program-count crossover (T * (H + 1)) between the small-batch and the
// large-batch DSV4 launch shapes, measured on GB300 by the benchmark's
// dispatch sweep (the two shapes tie within 2% between 33K and 130K
// programs; below, the one-row-per-warp grid has the lower latency).
constexpr int64_t kDefaultDsv4Threshold = 65536;
// Launch shapes (indices into kDsv4Configs / kQkConfigs) the automatic
// dispatch uses below / above the threshold.
constexpr int kDsv4SmallConfig = 0;  // tiles<4w,1row>
constexpr int kDsv4LargeConfig = 4;  // stream<8w,85reg,pairs>
constexpr int kQkSmallConfig = 0;    // tiles<4w,1step>
constexpr int kQkLargeConfig = 2;    // tiles<4w,4step>
constexpr int kQkStagedConfig = 7;   // bulk<16w,2st,6KB>
constexpr int kQkMidStagedConfig = 8;  // bulk<24w,2st,3KB>
// Entries of kQkConfigs that name the general kernel (any layout) with 4- or
// 8-dim fragments; forcing one routes every layout through that kernel.
constexpr int kQkGeneralFrag4Config = 5;
constexpr int kQkGeneralFrag8Config = 6;
// Fragment width the general kernel takes for layouts outside the tuned one.
constexpr int kQkGeneralFrag = 4;
// Q+K head rows below which the QK operator takes its small-batch shape.
constexpr int64_t kQkSmallRows = 152 * 8;
// Bytes of Q+K head rows (rows x head_dim x 2) from which every layout takes
// the TMA-staged shape; below, the register-pipelined (head_dim 128, full
// NeoX) or one-shot general kernel.  Measured on GB300 with each launch
// following a 512 MB write (as the QKV projection precedes this operator):
// from 160 MB of rows the staged kernel is 5-13 % faster at every layout,
// and ties at 80 MB;
// it also holds its time after any preceding kernel (111-113 us at 32768
// tokens x 40 heads), while the one-shot kernels run 106-127 us depending
// on the L2 contents they start from.
constexpr int64_t kQkStagedBytes = (int64_t)1 << 27;
// Head_dim 128 with full NeoX rotation only: from 56 MiB of Q+K rows the
// 24-warp staged shape with 3 KB stages is 3-6 % faster than the
// register-pipelined kernel after a 512 MB write (GB300, two boxes, 32/8/8
// heads: T = 6144 29.4 vs 30.3-30.7 us, T = 8192 35.1 vs 37.1 us, T = 12288
// 49.4 vs 52.3-52.5 us; at T = 5120 the two tie within 2 % either way); the
// one-shot general kernel of the other layouts keeps its lead there.
constexpr int64_t kQkMidStagedBytes = (int64_t)56 << 20;

std::atomic<int64_t> g_threshold{-1};
std::atomic<int> g_dsv4_config{-1};
std::atomic<int> g_qk_config{-1};
std::atomic<int> g_sm_count[kvq::kMaxDevices];
std::once_flag g_env_once;
int64_t g_env_threshold = -1;
thread_local int t_last_cuda_error = 0;

int64_t env_threshold() {
  std::call_once(g_env_once, [] {
    const char* s = std::getenv("KVQ_DSV4_DISPATCH_THRESHOLD");
    if (s && *s) {
      char* end = nullptr;
      const long long v = std::strtoll(s, &end, 10);
      if (end && *end == '\0' && v >= 0) g_env_threshold = v;
    }
  });
  return g_env_threshold >= 0 ? g_env_threshold : kDefaultDsv4Threshold;
}

int64_t current_threshold() {
  const int64_t v = g_threshold.load(std::memory_order_relaxed);
  return v >= 0 ? v : env_threshold();
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kvq_status finish_launch(cudaError_t e) {
  if (e == cudaSuccess) return KVQ_OK;
  t_last_cuda_error = static_cast<int>(e);
  return KVQ_ERR_CUDA;
}

constexpr int64_t kIndexLimit = (int64_t)1 << 31;

int qk_config_for(int64_t num_tokens, int64_t rows, int head_dim, bool tuned) {
  const int forced = g_qk_config.load(std::memory_order_relaxed);
  if (forced >= 0) return forced;
  if (num_tokens >= kIndexLimit || rows >= kIndexLimit) return kQkStagedConfig;
  const int64_t n = num_tokens * rows;
  const int64_t bytes = n * head_dim * 2;
  if (n < kQkSmallRows) return kQkSmallConfig;
  if (bytes >= kQkStagedBytes) return kQkStagedConfig;
  return tuned && bytes >= kQkMidStagedBytes ? kQkMidStagedConfig : kQkLargeConfig;
}

int dsv4_config_for(int64_t num_tokens, int num_heads) {
  const int forced = g_dsv4_config.load(std::memory_order_relaxed);
  if (forced >= 0) return forced;
  return kvq_dsv4_dispatch_path(num_tokens, num_heads) == 0 ? kDsv4SmallConfig
                                                            : kDsv4LargeConfig;
}

int set_config(std::atomic<int>& slot, int id, int n) {
  const int prev = slot.load(std::memory_order_relaxed);
  if (id >= n) return -2;
  slot.store(id < 0 ? -1 : id, std::memory_order_relaxed);
  return prev;
}

}  // namespace

namespace kvq {

namespace {
std::atomic<uint32_t> g_stage_wait_limit{1u << 22};
std::atomic<bool> g_programmatic_launch{true};
}  // namespace

bool programmatic_launch() { return g_programmatic_launch.load(std::memory_order_relaxed); }

uint32_t stage_wait_limit() { return g_stage_wait_limit.load(std::memory_order_relaxed); }

uint32_t set_stage_wait_limit(uint32_t polls) {
  return g_stage_wait_limit.exchange(polls, std::memory_order_relaxed);
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < kMaxDevices) {
    const int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 1;
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace kvq

namespace {

kvq_status qk_impl(void* qkv, int64_t num_tokens, int num_heads_q, int num_heads_k,
                   int num_heads_v, int head_dim, float eps, const void* q_weight,
                   const void* k_weight, const float* cos_sin_cache, int rotary_dim,
                   int is_neox, const int64_t* positions, int64_t max_pos, int32_t* errors,
                   kvq_stream_t stream) {
  if (num_tokens < 0 || num_heads_q < 0 || num_heads_k < 0 || num_heads_v < 0)
    return KVQ_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  if (is_neox != 0 && is_neox != 1) return KVQ_ERR_UNSUPPORTED;
  if (rotary_dim < 16 || rotary_dim > head_dim || rotary_dim % 16 != 0)
    return KVQ_ERR_UNSUPPORTED;
  if (!std::isfinite(eps) || eps < 0.0f) return KVQ_ERR_VALUE;
  // head counts summed in 64 bits: each is at most INT_MAX
  const int64_t rows64 = (int64_t)num_heads_q + num_heads_k;
  if (rows64 + num_heads_v > (1 << 20) || num_tokens >= kIndexLimit ||
      num_tokens * (rows64 + 1) >= kIndexLimit)
    return KVQ_ERR_SHAPE;
  const int rows = (int)rows64;
  if (num_tokens == 0 || rows == 0) return KVQ_OK;
  if (!qkv || !q_weight || !k_weight || !cos_sin_cache || !positions) return KVQ_ERR_NULL;
  if (!aligned(qkv, 16) || !aligned(q_weight, 16) || !aligned(k_weight, 16) ||
      !aligned(cos_sin_cache, 16) || !aligned(positions, 8))
    return KVQ_ERR_ALIGN;
  kvq::QkArgs a;
  a.qkv = qkv;
  a.q_weight = q_weight;
  a.k_weight = k_weight;
  a.cos_sin = cos_sin_cache;
  a.positions = positions;
  a.num_tokens = (int)num_tokens;
  a.num_heads_q = num_heads_q;
  a.num_heads_k = num_heads_k;
  a.num_heads_v = num_heads_v;
  a.head_dim = head_dim;
  a.rotary_dim = rotary_dim;
  a.is_neox = is_neox;
  a.eps = eps;
  a.max_pos = max_pos;
  a.errors = reinterpret_cast<int*>(errors);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t n = num_tokens * (int64_t)rows;
  const bool small = n < kQkSmallRows;
  const bool tuned = head_dim == 128 && is_neox == 1 && rotary_dim == 128;
  const int config = qk_config_for(num_tokens, rows, head_dim, tuned);
  if (config == kQkGeneralFrag4Config || config == kQkGeneralFrag8Config)
    return finish_launch(
        kvq::launch_qk_general(a, small, config == kQkGeneralFrag8Config ? 8 : 4, st));
  // TMA-staged shapes serve every layout, unchecked calls on device memory.
  const int shape = config - kvq::kQkFirstBulk;
  if (errors == nullptr && shape >= 0 && kvq::qk_bulk_eligible(a, shape))
    return finish_launch(kvq::launch_qk_bulk(a, shape, st));
  if (tuned) return finish_launch(kvq::launch_qk_norm_rope(a, config, st));
  return finish_launch(kvq::launch_qk_general(a, small && shape < 0, kQkGeneralFrag, st));
}

kvq_status dsv4_impl(const void* q, void* q_out, const void* kv, int64_t num_tokens,
                     int num_heads, float eps, const void* q_weight, const void* kv_weight,
                     const float* cos_sin_cache, const int64_t* positions,
                     const int64_t* slot_mapping, uint8_t* kv_cache, int block_size,
                     int64_t max_pos, int64_t num_slots, int32_t* errors,
                     kvq_stream_t stream) {
  if (num_tokens < 0 || num_heads < 1 || block_size < 1) return KVQ_ERR_SHAPE;
  if (num_tokens >= kIndexLimit || num_tokens * ((int64_t)num_heads + 1) >= kIndexLimit)
    return KVQ_ERR_SHAPE;
  if (!std::isfinite(eps) || eps < 0.0f) return KVQ_ERR_VALUE;
  if (num_tokens == 0) return KVQ_OK;
  if (!q || !q_out || !kv || !q_weight || !kv_weight || !cos_sin_cache || !positions ||
      !slot_mapping || !kv_cache)
    return KVQ_ERR_NULL;
  if (!aligned(q, 16) || !aligned(q_out, 16) || !aligned(kv, 16) || !aligned(q_weight, 16) ||
      !aligned(kv_weight, 16) || !aligned(cos_sin_cache, 16) || !aligned(positions, 8) ||
      !aligned(slot_mapping, 8) || !aligned(kv_cache, 8))
    return KVQ_ERR_ALIGN;
  // q_out must be q itself or not overlap it: a partial overlap would let one
  // warp overwrite rows another warp has not read yet.
  const uintptr_t qa = reinterpret_cast<uintptr_t>(q), oa = reinterpret_cast<uintptr_t>(q_out);
  const uintptr_t qbytes = (uintptr_t)num_tokens * (uintptr_t)num_heads * 512u * 2u;
  if (qa != oa && qa < oa + qbytes && oa < qa + qbytes) return KVQ_ERR_VALUE;
  kvq::Dsv4Args a;
  a.q = q;
  a.q_out = q_out;
  a.kv = kv;
  a.q_weight = q_weight;
  a.kv_weight = kv_weight;
  a.cos_sin = cos_sin_cache;
  a.positions = positions;
  a.slot_mapping = slot_mapping;
  a.kv_cache = kv_cache;
  a.num_tokens = (int)num_tokens;
  a.num_heads = num_heads;
  a.eps = eps;
  a.max_pos = max_pos;
  a.num_slots = num_slots;
  a.errors = reinterpret_cast<int*>(errors);
  return finish_launch(kvq::launch_dsv4(a, dsv4_config_for(num_tokens, num_heads),
                                        reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status gather_impl(const uint8_t* kv_cache, int block_size, const int64_t* slots,
                       int64_t num_rows, void* out, int64_t num_slots, int32_t* errors,
                       kvq_stream_t stream) {
  if (num_rows < 0 || num_rows >= kIndexLimit || block_size < 1) return KVQ_ERR_SHAPE;
  if (num_rows == 0) return KVQ_OK;
  if (!kv_cache || !slots || !out) return KVQ_ERR_NULL;
  if (!aligned(kv_cache, 8) || !aligned(slots, 8) || !aligned(out, 16)) return KVQ_ERR_ALIGN;
  kvq::GatherArgs a;
  a.kv_cache = kv_cache;
  a.slots = slots;
  a.out = out;
  a.num_rows = (int)num_rows;
  a.num_slots = num_slots;
  a.errors = reinterpret_cast<int*>(errors);
  return finish_launch(kvq::launch_dsv4_gather(a, reinterpret_cast<cudaStream_t>(stream)));
}

// Extra arguments of the bounds-checked entry points.
kvq_status check_counter(const int32_t* errors, int64_t bound) {
  if (!errors) return KVQ_ERR_NULL;
  if (!aligned(errors, 4)) return KVQ_ERR_ALIGN;
  if (bound < 0) return KVQ_ERR_SHAPE;
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status fused_qk_norm_rope_ex(void* qkv, int64_t num_tokens, int num_heads_q,
                                 int num_heads_k, int num_heads_v, int head_dim,
                                 float eps, const void* q_weight,
                                 const void* k_weight, const float* cos_sin_cache,
                                 int rotary_dim, int is_neox,
                                 const int64_t* positions, kvq_stream_t stream) {
  return qk_impl(qkv, num_tokens, num_heads_q, num_heads_k, num_heads_v, head_dim, eps,
                 q_weight, k_weight, cos_sin_cache, rotary_dim, is_neox, positions, 0, nullptr,
                 stream);
}

kvq_status fused_qk_norm_rope(void* qkv, int64_t num_tokens, int num_heads_q,
                              int num_heads_k, int num_heads_v, int head_dim,
                              float eps, const void* q_weight,
                              const void* k_weight, const float* cos_sin_cache,
                              int is_neox, const int64_t* positions,
                              kvq_stream_t stream) {
  return qk_impl(qkv, num_tokens, num_heads_q, num_heads_k, num_heads_v, head_dim, eps,
                 q_weight, k_weight, cos_sin_cache, head_dim, is_neox, positions, 0, nullptr,
                 stream);
}

kvq_status fused_qk_norm_rope_checked(void* qkv, int64_t num_tokens, int num_heads_q,
                                      int num_heads_k, int num_heads_v, int head_dim,
                                      float eps, const void* q_weight,
                                      const void* k_weight, const float* cos_sin_cache,
                                      int64_t max_pos, int rotary_dim, int is_neox,
                                      const int64_t* positions, int32_t* error_count,
                                      kvq_stream_t stream) {
  const kvq_status c = check_counter(error_count, max_pos);
  if (c != KVQ_OK) return c;
  return qk_impl(qkv, num_tokens, num_heads_q, num_heads_k, num_heads_v, head_dim, eps,
                 q_weight, k_weight, cos_sin_cache, rotary_dim, is_neox, positions, max_pos,
                 error_count, stream);
}

kvq_status dsv4_qnorm_rope_kv_rope_quant_insert_out(
    const void* q, void* q_out, const void* kv, int64_t num_tokens, int num_heads, float eps,
    const void* q_weight, const void* kv_weight, const float* cos_sin_cache,
    const int64_t* positions, const int64_t* slot_mapping, uint8_t* kv_cache,
    int block_size, kvq_stream_t stream) {
  return dsv4_impl(q, q_out, kv, num_tokens, num_heads, eps, q_weight, kv_weight,
                   cos_sin_cache, positions, slot_mapping, kv_cache, block_size, 0, 0, nullptr,
                   stream);
}

kvq_status dsv4_qnorm_rope_kv_rope_quant_insert_checked(
    const void* q, void* q_out, const void* kv, int64_t num_tokens, int num_heads, float eps,
    const void* q_weight, const void* kv_weight, const float* cos_sin_cache, int64_t max_pos,
    const int64_t* positions, const int64_t* slot_mapping, uint8_t* kv_cache,
    int64_t num_blocks, int block_size, int32_t* error_count, kvq_stream_t stream) {
  kvq_status c = check_counter(error_count, max_pos);
  if (c == KVQ_OK && num_blocks < 0) c = KVQ_ERR_SHAPE;
  if (c != KVQ_OK) return c;
  const int64_t num_slots = block_size > 0 ? num_blocks * (int64_t)block_size : 0;
  return dsv4_impl(q, q_out, kv, num_tokens, num_heads, eps, q_weight, kv_weight,
                   cos_sin_cache, positions, slot_mapping, kv_cache, block_size, max_pos,
                   num_slots, error_count, stream);
}

kvq_status dsv4_qnorm_rope_kv_rope_quant_insert(
    void* q, const void* kv, int64_t num_tokens, int num_heads, float eps,
    const void* q_weight, const void* kv_weight, const float* cos_sin_cache,
    const int64_t* positions, const int64_t* slot_mapping, uint8_t* kv_cache,
    int block_size, kvq_stream_t stream) {
  return dsv4_qnorm_rope_kv_rope_quant_insert_out(q, q, kv, num_tokens, num_heads, eps,
                                                  q_weight, kv_weight, cos_sin_cache, positions,
                                                  slot_mapping, kv_cache, block_size, stream);
}

kvq_status dsv4_kv_cache_gather(const uint8_t* kv_cache, int block_size, const int64_t* slots,
                                int64_t num_rows, void* out, kvq_stream_t stream) {
  return gather_impl(kv_cache, block_size, slots, num_rows, out, 0, nullptr, stream);
}

kvq_status dsv4_kv_cache_gather_checked(const uint8_t* kv_cache, int64_t num_blocks,
                                        int block_size, const int64_t* slots, int64_t num_rows,
                                        void* out, int32_t* error_count, kvq_stream_t stream) {
  kvq_status c = check_counter(error_count, num_blocks);
  if (c != KVQ_OK) return c;
  const int64_t num_slots = block_size > 0 ? num_blocks * (int64_t)block_size : 0;
  return gather_impl(kv_cache, block_size, slots, num_rows, out, num_slots, error_count, stream);
}

const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_NULL: return "a required pointer is NULL";
    case KVQ_ERR_SHAPE: return "invalid count or size";
    case KVQ_ERR_UNSUPPORTED: return "unsupported head_dim / rotary_dim / is_neox";
    case KVQ_ERR_ALIGN: return "pointer not aligned as required";
    case KVQ_ERR_CUDA: return "CUDA launch failed (see kvq_last_cuda_error)";
    case KVQ_ERR_VALUE: return "eps not finite / negative, or q_out partly overlaps q";
  }
  return "unknown kvq_status";
}

int kvq_last_cuda_error(void) { return t_last_cuda_error; }

int64_t kvq_dsv4_dispatch_threshold(void) { return current_threshold(); }

int64_t kvq_set_dsv4_dispatch_threshold(int64_t value) {
  const int64_t prev = current_threshold();
  g_threshold.store(value >= 0 ? value : -1, std::memory_order_relaxed);
  return prev;
}

int kvq_dsv4_dispatch_path(int64_t num_tokens, int num_heads) {
  if (num_tokens >= kIndexLimit) return 1;  // keeps the product below from overflowing
  return num_tokens * ((int64_t)num_heads + 1) < current_threshold() ? 0 : 1;
}

uint32_t kvq_set_stage_wait_limit(uint32_t polls) { return kvq::set_stage_wait_limit(polls); }

kvq_status kvq_stage_events(uint64_t* fallbacks, uint64_t* drain_timeouts, int reset) {
  if (!fallbacks || !drain_timeouts) return KVQ_ERR_NULL;
  uint64_t v[2] = {0, 0};
  const cudaError_t e = kvq::stage_events(v, reset != 0);
  if (e != cudaSuccess) return finish_launch(e);
  *fallbacks = v[0];
  *drain_timeouts = v[1];
  return KVQ_OK;
}

int kvq_set_programmatic_launch(int enable) {
  return kvq::g_programmatic_launch.exchange(enable != 0, std::memory_order_relaxed) ? 1 : 0;
}

int kvq_qk_num_configs(void) { return kvq::kQkNumConfigs; }

const char* kvq_qk_config_name(int id) {
  return (id >= 0 && id < kvq::kQkNumConfigs) ? kvq::kQkConfigs[id].name : nullptr;
}

int kvq_set_qk_config(int id) { return set_config(g_qk_config, id, kvq::kQkNumConfigs); }

int kvq_qk_config_for(int64_t num_tokens, int num_heads_q, int num_heads_k) {
  return qk_config_for(num_tokens, (int64_t)num_heads_q + num_heads_k, 128, true);
}

int kvq_dsv4_num_configs(void) { return kvq::kDsv4NumConfigs; }

const char* kvq_dsv4_config_name(int id) {
  return (id >= 0 && id < kvq::kDsv4NumConfigs) ? kvq::kDsv4Configs[id].name : nullptr;
}

int kvq_set_dsv4_config(int id) { return set_config(g_dsv4_config, id, kvq::kDsv4NumConfigs); }

int kvq_dsv4_config_for(int64_t num_tokens, int num_heads) {
  return dsv4_config_for(num_tokens, num_heads);
}

}  // extern "C"
