// kvq_qk_bulk.cu -- the head_dim-128 full-NeoX QK operator with its inputs
// staged in shared memory by the bulk-copy (TMA) engine.
//
// Operator and row arithmetic: those of kvq_qk_norm_rope.cu (InfiniOps PR
// #1019, "Add the NineToothed NVIDIA implementation of FusedQkNormRope",
// section "Summary"), shared through kvq_qk_row.cuh, so the results are
// bit-identical to every other launch shape of the operator.
//
// Mapping on sm_103a.  A persistent grid (resident CTAs x SMs).  Each warp
// owns a ring of NS shared-memory stages with one mbarrier per stage and takes
// the work items gw, gw + W, gw + 2W, ... (W = warps in the grid), so at any
// moment the grid works on one contiguous window of qkv.  A work item is
// (token, chunk of at most RMAX consecutive Q/K head rows, the chunks of a
// token balanced in length).  Its rows are one contiguous span of qkv and
// arrive with one cp.async.bulk; the token's cos/sin row (512 bytes) arrives
// with a second; both complete on the stage's mbarrier, and both carry an L2
// evict-first policy (each byte is read once).  Lane 0 keeps NS items in
// flight: when the warp has consumed a stage it issues the item NS ahead
// into it.  The positions of the warp's next 32 items are fetched one per
// lane, a window ahead, so no copy waits on a position load.  All 32 lanes
// wait on the stage's barrier; then the half-warps take alternate rows, U row
// pairs at a time (independent rows, so their shuffles overlap), reading
// their 8-byte fragments and their cosines and sines from shared memory, and
// write the results straight to global memory with evict-first stores.  V
// columns are never addressed.
//
// Every wait is bounded.  A warp that has polled a stage barrier `wait_limit`
// times, or for 20 ms, stops staging: it first waits (bounded again) for the
// copies it still has in flight, then finishes its remaining items with
// direct global loads, which give the same bits.  A stalled copy costs time,
// never correctness.
#include <atomic>

#include "kvq_device.cuh"
#include "kvq_launch.h"
#include "kvq_qk_bulk.h"
#include "kvq_qk_row.cuh"

namespace kvq {
namespace {

using qk128::kHeadDim;
using qk128::row_math;
using qk128::Weights;

constexpr int kRowBytes = kHeadDim * 2;  // one bf16 head row
constexpr int kCsBytes = kHeadDim * 4;   // one fp32 cos/sin row
constexpr int kUnroll = 4;               // row pairs computed together
constexpr uint32_t kDefaultWaitLimit = 1u << 22;
constexpr uint64_t kWaitNs = 20000000;   // 20 ms: a stage wait then gives up
constexpr uint32_t kDrainPolls = 1u << 22;
constexpr uint64_t kDrainNs = 100000000; // 100 ms per copy still in flight

std::atomic<uint32_t> g_wait_limit{kDefaultWaitLimit};

struct BulkParams {
  __nv_bfloat16* qkv;
  const __nv_bfloat16* q_weight;
  const __nv_bfloat16* k_weight;
  const float* cos_sin;
  const int64_t* positions;
  int64_t row_elems;  // (Hq + Hk + Hv) * 128
  int num_q;          // Hq
  int num_rows;       // Hq + Hk
  int chunks;         // work items per token
  int chunk_rows;     // rows of every chunk but possibly the token's last
  int items;          // num_tokens * chunks
  float eps;
  uint32_t wait_limit;
};

// ---- inline PTX: mbarrier, bulk copy, cache policy, proxy fences ----------

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
// `limit` times and for at most `ns` nanoseconds; the result is the same on
// every lane of the warp.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint32_t limit,
                                               uint64_t ns) {
  bool done = false;
  const uint64_t t0 = limit ? global_ns() : 0;
  for (uint32_t i = 0; i < limit && !done; ++i) {
    done = mbar_test(bar, parity);
    if (!done && global_ns() - t0 > ns) break;
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

// ---- work items --------------------------------------------------------------

struct Item {
  int t, r0, nr;  // token, first row, rows
};

__device__ __forceinline__ Item item_at(const BulkParams& p, int item) {
  Item it;
  it.t = item / p.chunks;
  it.r0 = (item - it.t * p.chunks) * p.chunk_rows;
  it.nr = min(p.num_rows - it.r0, p.chunk_rows);
  return it;
}

// The rows of one item: fragments read by `fetch(j, lo, hi)` (row j of the
// item), normalised and rotated, and handed to `put(j, lo, hi)`.  Half-warp
// `half` takes rows half, half + 2, ...; the trip count is warp-uniform.
template <typename Fetch, typename Put>
__device__ __forceinline__ void item_rows(const BulkParams& p, const Item& it, int half,
                                          const Weights& w, const float4& c4, const float4& s4,
                                          Fetch fetch, Put put) {
  for (int j0 = 0; j0 < it.nr; j0 += 2 * kUnroll) {
    uint2 lo[kUnroll], hi[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = j0 + 2 * u + half;
      lo[u] = hi[u] = make_uint2(0u, 0u);
      if (j < it.nr) fetch(j, lo[u], hi[u]);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (j0 + 2 * u >= it.nr) break;  // warp-uniform: no row left for either half
      const int j = j0 + 2 * u + half;
      row_math(lo[u], hi[u], it.r0 + j < p.num_q, w, c4, s4, p.eps);
      if (j < it.nr) put(j, lo[u], hi[u]);
    }
  }
}

// Row j of an item in global memory.
__device__ __forceinline__ uint2* global_row(const BulkParams& p, const Item& it, int j) {
  return reinterpret_cast<uint2*>(p.qkv + (size_t)it.t * (size_t)p.row_elems +
                                  (size_t)(it.r0 + j) * kHeadDim);
}

// An item straight from global memory (the path after a wait ran out).
__device__ __forceinline__ void direct_item(const BulkParams& p, int item, int half, int l16,
                                            const Weights& w) {
  const Item it = item_at(p, item);
  const int64_t pos = __ldg(p.positions + it.t);
  const float4* cs = reinterpret_cast<const float4*>(p.cos_sin + pos * kHeadDim);
  const float4 c4 = __ldg(cs + l16);
  const float4 s4 = __ldg(cs + 16 + l16);
  item_rows(
      p, it, half, w, c4, s4,
      [&](int j, uint2& lo, uint2& hi) {
        const uint2* row = global_row(p, it, j);
        lo = __ldcs(row + l16);
        hi = __ldcs(row + 16 + l16);
      },
      [&](int j, const uint2& lo, const uint2& hi) {
        uint2* row = global_row(p, it, j);
        __stcs(row + l16, lo);
        __stcs(row + 16 + l16, hi);
      });
}

template <int WARPS, int NS, int RMAX>
__global__ void __launch_bounds__(WARPS * 32, 1)
qk_bulk_kernel(const BulkParams p) {
  constexpr int kCsAt = RMAX * kRowBytes;       // cos/sin row inside a stage
  constexpr int kStage = kCsAt + kCsBytes;      // a multiple of 128 bytes
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const int gw = blockIdx.x * WARPS + warp;
  const int nw = gridDim.x * WARPS;
  if (gw >= p.items) return;                    // whole warp leaves together
  const int n = (p.items - 1 - gw) / nw + 1;    // this warp's items: gw + k * nw, k < n

  uint8_t* ring = smem + (size_t)warp * NS * kStage;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar0 = smem_addr(smem + (size_t)WARPS * NS * kStage) + 8u * NS * warp;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8u * s, 1);
    mbar_init_fence();
  }
  __syncwarp();
  Weights w;
  qk128::load_weights(p.q_weight, p.k_weight, l16, w);
  const uint64_t pol = evict_first_policy();

  // Positions of issue window [wb, wb + 32) (one per lane) and of the next.
  auto position = [&](int k) -> int64_t {
    return k < n ? __ldg(p.positions + (gw + k * nw) / p.chunks) : 0;
  };
  int wb = 0;
  int64_t pos_cur = position(lane), pos_next = position(32 + lane);

  // Copies of item k into stage k % NS; every lane calls, lane 0 issues.
  // Issued in order k = 0, 1, 2, ...
  auto issue = [&](int k) {
    if (k >= n) return;  // warp-uniform
    if (k - wb == 32) {
      wb += 32;
      pos_cur = pos_next;
      pos_next = position(wb + 32 + lane);
    }
    const int64_t pos = __shfl_sync(kFullMask, pos_cur, k - wb);
    if (lane == 0) {
      const Item it = item_at(p, gw + k * nw);
      const uint32_t stage = ring_s + (uint32_t)(k % NS) * kStage;
      const uint32_t bar = bar0 + 8u * (k % NS);
      const uint32_t bytes = (uint32_t)it.nr * kRowBytes;
      fence_proxy_async();
      mbar_arrive_expect_tx(bar, bytes + kCsBytes);
      bulk_load(stage, global_row(p, it, 0), bytes, bar, pol);
      bulk_load(stage + kCsAt, p.cos_sin + pos * kHeadDim, kCsBytes, bar, pol);
    }
  };

#pragma unroll
  for (int k = 0; k < NS; ++k) issue(k);
  int k = 0;
  for (; k < n; ++k) {
    if (!mbar_wait_warp(bar0 + 8u * (k % NS), (uint32_t)(k / NS) & 1u, p.wait_limit, kWaitNs))
      break;
    const Item it = item_at(p, gw + k * nw);
    const uint8_t* stage = ring + (size_t)(k % NS) * kStage;
    const float4 c4 = *reinterpret_cast<const float4*>(stage + kCsAt + 16 * l16);
    const float4 s4 = *reinterpret_cast<const float4*>(stage + kCsAt + 256 + 16 * l16);
    item_rows(
        p, it, half, w, c4, s4,
        [&](int j, uint2& lo, uint2& hi) {
          const uint2* row = reinterpret_cast<const uint2*>(stage + j * kRowBytes);
          lo = row[l16];
          hi = row[16 + l16];
        },
        [&](int j, const uint2& lo, const uint2& hi) {
          uint2* row = global_row(p, it, j);
          __stcs(row + l16, lo);
          __stcs(row + 16 + l16, hi);
        });
    __syncwarp();
    issue(k + NS);
  }
  if (k < n) {
    // A wait ran out: let the copies still in flight (items k .. k+NS-1)
    // land before this warp's shared memory can be reused, then finish.
    for (int q = k; q < n && q < k + NS; ++q)
      mbar_wait_warp(bar0 + 8u * (q % NS), (uint32_t)(q / NS) & 1u, kDrainPolls, kDrainNs);
    for (; k < n; ++k) direct_item(p, gw + k * nw, half, l16, w);
  }
}

// ---- launch ---------------------------------------------------------------------

template <int WARPS, int NS, int RMAX>
constexpr size_t smem_bytes() {
  return (size_t)WARPS * NS * (RMAX * kRowBytes + kCsBytes) + (size_t)WARPS * NS * 8;
}

// Opts the kernel in to its shared memory and counts its resident CTAs per
// SM, once per device.
template <int WARPS, int NS, int RMAX>
cudaError_t prepare(int* per_sm) {
  static std::atomic<int> cache[kMaxDevices];
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
  auto kernel = qk_bulk_kernel<WARPS, NS, RMAX>;
  constexpr size_t bytes = smem_bytes<WARPS, NS, RMAX>();
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, WARPS * 32, bytes);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  if (cached) cache[dev].store(n, std::memory_order_relaxed);
  *per_sm = n;
  return cudaSuccess;
}

void chunking(const QkArgs& a, int rmax, int* chunks, int* chunk_rows) {
  const int rows = a.num_heads_q + a.num_heads_k;
  *chunks = (rows + rmax - 1) / rmax;
  *chunk_rows = (rows + *chunks - 1) / *chunks;
}

template <int WARPS, int NS, int RMAX>
cudaError_t launch_shape(const QkArgs& a, cudaStream_t stream) {
  static_assert((RMAX * kRowBytes + kCsBytes) % 128 == 0, "stage alignment");
  static_assert(smem_bytes<WARPS, NS, RMAX>() <= 227 * 1024, "shared memory per CTA");
  int per_sm = 0;
  cudaError_t e = prepare<WARPS, NS, RMAX>(&per_sm);
  if (e != cudaSuccess) return e;
  BulkParams p;
  p.qkv = static_cast<__nv_bfloat16*>(a.qkv);
  p.q_weight = static_cast<const __nv_bfloat16*>(a.q_weight);
  p.k_weight = static_cast<const __nv_bfloat16*>(a.k_weight);
  p.cos_sin = a.cos_sin;
  p.positions = a.positions;
  p.num_q = a.num_heads_q;
  p.num_rows = a.num_heads_q + a.num_heads_k;
  p.row_elems = (int64_t)(p.num_rows + a.num_heads_v) * kHeadDim;
  chunking(a, RMAX, &p.chunks, &p.chunk_rows);
  p.items = a.num_tokens * p.chunks;
  p.eps = a.eps;
  p.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  int64_t grid = (int64_t)per_sm * device_sm_count();
  const int64_t need = (p.items + WARPS - 1) / WARPS;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  qk_bulk_kernel<WARPS, NS, RMAX>
      <<<(unsigned)grid, WARPS * 32, smem_bytes<WARPS, NS, RMAX>(), stream>>>(p);
  return cudaGetLastError();
}

bool device_memory(const void* ptr) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();  // a failed query is not sticky: clear it before the launch
    return false;
  }
  return attr.type == cudaMemoryTypeDevice;
}

}  // namespace

bool qk_bulk_eligible(const QkArgs& a, int shape) {
  static constexpr int kRows[] = {
#define KVQ_ROWS(W, S, R) R,
      KVQ_QK_BULK_SHAPES(KVQ_ROWS)
#undef KVQ_ROWS
  };
  if (shape < 0 || shape >= kQkBulkShapes) return false;
  if (a.head_dim != kHeadDim || a.is_neox != 1 || a.rotary_dim != kHeadDim) return false;
  int chunks = 0, chunk_rows = 0;
  chunking(a, kRows[shape], &chunks, &chunk_rows);
  if ((int64_t)(chunks - 1) * chunk_rows >= a.num_heads_q + a.num_heads_k) return false;
  return device_memory(a.qkv) && device_memory(a.cos_sin);
}

cudaError_t launch_qk_bulk(const QkArgs& a, int shape, cudaStream_t stream) {
  using Launch = cudaError_t (*)(const QkArgs&, cudaStream_t);
  static constexpr Launch kLaunch[] = {
#define KVQ_LAUNCH(W, S, R) &launch_shape<W, S, R>,
      KVQ_QK_BULK_SHAPES(KVQ_LAUNCH)
#undef KVQ_LAUNCH
  };
  if (shape < 0 || shape >= kQkBulkShapes) return cudaErrorInvalidValue;
  return kLaunch[shape](a, stream);
}

uint32_t set_qk_stage_wait_limit(uint32_t polls) {
  return g_wait_limit.exchange(polls, std::memory_order_relaxed);
}

}  // namespace kvq
