// kvq_qk_bulk.cu -- the packed-QKV operator (every supported layout: head_dim
// 64 / 128 / 256, NeoX or GPT-J pairs, full or partial rotation) with its
// inputs staged in shared memory by the bulk-copy (TMA) engine.
//
// Operator and row arithmetic: those of InfiniOps PR #1019 ("Add the
// NineToothed NVIDIA implementation of FusedQkNormRope", section "Summary"),
// shared with the one-shot kernels through kvq_qk_general_row.cuh, so the
// results are the same bits.
//
// Mapping on sm_103a.  A persistent grid (resident CTAs x SMs).  Each warp
// owns a ring of NS shared-memory stages with one mbarrier per stage and takes
// the work items gw, gw + W, gw + 2W, ... (W = warps in the grid), so at any
// moment the grid works on one contiguous window of qkv.  A work item is
// (token, chunk of at most RMAX consecutive Q/K head rows, the chunks of a
// token balanced in length); a stage holds STAGE_BYTES of rows, so RMAX =
// STAGE_BYTES / (2 D).  The item's rows are one contiguous span of qkv and
// arrive with one cp.async.bulk (TILED: one cp.async.bulk.tensor box of a
// [T][Hq+Hk][D] tensor map, rows past the token's Q/K rows read as zero and
// never written -- measured slower, kept as a launch shape); the token's
// cos/sin row (4 rot bytes)
// arrives with a second; both complete on the stage's mbarrier, and both
// carry an L2 evict-first policy (each byte is read once).  Lane 0 keeps NS
// items in flight: when the warp has consumed a stage it issues the item NS
// ahead into it.  The positions of the warp's next 32 items are fetched one
// per lane, a window ahead, so no copy waits on a position load.  All 32
// lanes wait on the stage's barrier; then each group of D/8 lanes takes a
// row, four rows per group at a time (independent rows, so their shuffles
// overlap), reading its fragments and its cosines and sines from shared
// memory, and the results go straight to global memory with evict-first
// stores.  V columns are never addressed.
//
// Every wait is bounded.  A warp that has polled a stage barrier `wait_limit`
// times, or for 20 ms, stops staging: it first waits (bounded again) for the
// copies it still has in flight, then finishes its remaining items with
// direct global loads, which give the same bits.  A stalled copy costs time,
// never correctness.  Both events are counted in a per-device status word
// that the host reads (kvq_stage_events): a warp that stopped staging, and a
// warp whose copies in flight still had not landed when it stopped waiting
// for them -- its CTA may then exit with a copy still writing its shared
// memory, which the count makes visible instead of silent.
#include <atomic>
#include <cstring>

#include "kvq_device.cuh"
#include "kvq_launch.h"
#include "kvq_qk_bulk.h"
#include "kvq_qk_general_row.cuh"
#include "kvq_tma.cuh"

namespace kvq {
namespace {

using qkgen::Lane;
using Frag4 = qkgen::Frag<4>;
constexpr int kF = 4;                    // dims per fragment
constexpr int kUnroll = 4;               // row steps computed together
using namespace tma;

// Staging events on this device since the last reset: [0] warps that stopped
// staging because a stage wait ran out, [1] warps whose copies in flight then
// still had not landed within the drain limit.  Written only on those paths.
__device__ unsigned long long g_stage_events[2];

struct BulkParams {
  CUtensorMap rows_map;  // tiled launches: [T][Hq + Hk][D] view of the Q/K rows
  __nv_bfloat16* qkv;
  const __nv_bfloat16* q_weight;
  const __nv_bfloat16* k_weight;
  const float* cos_sin;
  const int64_t* positions;
  int64_t row_elems;  // (Hq + Hk + Hv) * D
  int num_q;          // Hq
  int num_rows;       // Hq + Hk
  int rot;            // rotary_dim
  int chunks;         // work items per token
  int chunk_rows;     // rows of every chunk but possibly the token's last
  int items;          // num_tokens * chunks
  float eps;
  uint32_t wait_limit;
};

// ---- work items -------------------------------------------------------------

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

// Row j of an item in global memory.
template <int D>
__device__ __forceinline__ __nv_bfloat16* global_row(const BulkParams& p, const Item& it, int j) {
  return p.qkv + (size_t)it.t * (size_t)p.row_elems + (size_t)(it.r0 + j) * D;
}

// The lane's packed Q and K weights at its two fragments.
struct Weights {
  uint2 qa, qb, ka, kb;
};

// The rows of one item: lane group g (of 32 / (D/8)) takes rows g, g + RPW,
// ...; `rows` points at the item's first row (shared or global memory),
// `angles` at the token's cos/sin row.  The trip count is warp-uniform.
template <int D, bool NEOX, bool SMEM>
__device__ __forceinline__ void item_rows(const BulkParams& p, const Item& it, int g, int l,
                                          const Lane<D, kF, NEOX>& ln, const Weights& w,
                                          const __nv_bfloat16* rows, const float* angles) {
  constexpr int RPW = 32 / (D / (2 * kF));  // rows per warp step
  float cs[kF], sn[kF];
  qkgen::lane_angles<D, kF, NEOX, !SMEM>(angles, l, p.rot, ln, cs, sn);
  for (int j0 = 0; j0 < it.nr; j0 += RPW * kUnroll) {
    uint2 xa[kUnroll], xb[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = j0 + RPW * u + g;
      xa[u] = xb[u] = Frag4::zero();
      if (j < it.nr) {
        const __nv_bfloat16* row = rows + (size_t)j * D;
        if (SMEM) {
          xa[u] = *reinterpret_cast<const uint2*>(row + ln.oa);
          xb[u] = *reinterpret_cast<const uint2*>(row + ln.ob);
        } else {
          xa[u] = __ldcs(reinterpret_cast<const uint2*>(row + ln.oa));
          xb[u] = __ldcs(reinterpret_cast<const uint2*>(row + ln.ob));
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (j0 + RPW * u >= it.nr) break;  // warp-uniform: no row left for any group
      const int j = j0 + RPW * u + g;
      const bool is_q = it.r0 + j < p.num_q;
      qkgen::row_math<D, kF, NEOX, true>(xa[u], xb[u], is_q ? w.qa : w.ka, is_q ? w.qb : w.kb, cs,
                                         sn, ln, p.eps);
      if (j < it.nr) {
        __nv_bfloat16* row = global_row<D>(p, it, j);
        __stcs(reinterpret_cast<uint2*>(row + ln.oa), xa[u]);
        __stcs(reinterpret_cast<uint2*>(row + ln.ob), xb[u]);
      }
    }
  }
}

template <int D, bool NEOX, int WARPS, int NS, int STAGE_BYTES, bool TILED>
__global__ void __launch_bounds__(WARPS * 32, 1)
qk_bulk_kernel(const __grid_constant__ BulkParams p) {
  grid_dependency_wait();
  constexpr int kCsAt = STAGE_BYTES;           // cos/sin row inside a stage
  constexpr int kStage = STAGE_BYTES + 4 * D;  // room for a full-width cos/sin row
  constexpr int LPR = D / (2 * kF);            // lanes per row
  static_assert(kStage % 128 == 0, "stage alignment");
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / LPR, l = lane % LPR;
  const int gw = blockIdx.x * WARPS + warp;
  const int nw = gridDim.x * WARPS;
  // This warp's items: gw + k nw, k < n.  (Giving each warp pairs or quads
  // of consecutive items instead, so that the items it has in flight are
  // adjacent, measured 1-5 % slower at every layout and size.)
  if (gw >= p.items) return;                    // whole warp leaves together
  const int n = (p.items - 1 - gw) / nw + 1;

  uint8_t* ring = smem + (size_t)warp * NS * kStage;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar0 = smem_addr(smem + (size_t)WARPS * NS * kStage) + 8u * NS * warp;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8u * s, 1);
    mbar_init_fence();
  }
  __syncwarp();
  const Lane<D, kF, NEOX> ln(l, p.rot);
  Weights w;
  w.qa = __ldg(reinterpret_cast<const uint2*>(p.q_weight + ln.oa));
  w.qb = __ldg(reinterpret_cast<const uint2*>(p.q_weight + ln.ob));
  w.ka = __ldg(reinterpret_cast<const uint2*>(p.k_weight + ln.oa));
  w.kb = __ldg(reinterpret_cast<const uint2*>(p.k_weight + ln.ob));
  const uint64_t pol = evict_first_policy();
  const uint32_t cs_bytes = 4u * (uint32_t)p.rot;

  // Positions of issue window [wb, wb + 32) (one per lane) and of the next.
  auto position = [&](int k) -> int64_t {
    return k < n ? __ldg(p.positions + (gw + k * nw) / p.chunks) : 0;
  };
  int wb = 0;
  int64_t pos_cur = position(lane), pos_next = position(32 + lane);

  // Copies of item k into stage k % NS, issued in order k = 0, 1, 2, ...;
  // every lane calls, lane 0 issues.
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
      fence_proxy_async();
      if (TILED) {
        // The whole box arrives: rows past the token's Q/K rows read as zero.
        mbar_arrive_expect_tx(bar, (uint32_t)p.chunk_rows * (2u * D) + cs_bytes);
        tile_load_3d(stage, &p.rows_map, 0, it.r0, it.t, bar, pol);
      } else {
        const uint32_t bytes = (uint32_t)it.nr * (2u * D);
        mbar_arrive_expect_tx(bar, bytes + cs_bytes);
        bulk_load(stage, global_row<D>(p, it, 0), bytes, bar, pol);
      }
      bulk_load(stage + kCsAt, p.cos_sin + pos * p.rot, cs_bytes, bar, pol);
    }
  };

#pragma unroll
  for (int k = 0; k < NS; ++k) issue(k);
  int k = 0;
  for (; k < n; ++k) {
    if (!mbar_wait_warp(bar0 + 8u * (k % NS), (uint32_t)(k / NS) & 1u, p.wait_limit, kWaitNs))
      break;
    const uint8_t* stage = ring + (size_t)(k % NS) * kStage;
    item_rows<D, NEOX, true>(p, item_at(p, gw + k * nw), g, l, ln, w,
                             reinterpret_cast<const __nv_bfloat16*>(stage),
                             reinterpret_cast<const float*>(stage + kCsAt));
    __syncwarp();
    issue(k + NS);
  }
  if (k < n) {
    // A wait ran out: let the copies still in flight (items k .. k+NS-1)
    // land before this warp's shared memory can be reused, then finish from
    // global memory.  Both events are counted for the host.
    bool drained = true;
    for (int q = k; q < n && q < k + NS; ++q)
      drained &= mbar_wait_warp(bar0 + 8u * (q % NS), (uint32_t)(q / NS) & 1u, kDrainPolls,
                                kDrainNs);
    if (lane == 0) {
      atomicAdd(&g_stage_events[0], 1ull);
      if (!drained) atomicAdd(&g_stage_events[1], 1ull);
    }
    for (; k < n; ++k) {
      const Item it = item_at(p, gw + k * nw);
      item_rows<D, NEOX, false>(p, it, g, l, ln, w, global_row<D>(p, it, 0),
                                p.cos_sin + __ldg(p.positions + it.t) * p.rot);
    }
  }
}

// ---- launch -------------------------------------------------------------------

template <int D, int WARPS, int NS, int STAGE_BYTES>
constexpr size_t smem_bytes() {
  return (size_t)WARPS * NS * (STAGE_BYTES + 4 * D) + (size_t)WARPS * NS * 8;
}

void chunking(const QkArgs& a, int rmax, int* chunks, int* chunk_rows) {
  const int rows = a.num_heads_q + a.num_heads_k;
  *chunks = (rows + rmax - 1) / rmax;
  *chunk_rows = (rows + *chunks - 1) / *chunks;
}

template <int D, bool NEOX, int WARPS, int NS, int STAGE_BYTES, bool TILED>
cudaError_t launch_layout(const QkArgs& a, cudaStream_t stream) {
  static_assert(smem_bytes<D, WARPS, NS, STAGE_BYTES>() <= 227 * 1024, "shared memory per CTA");
  static std::atomic<int> cache[kMaxDevices];
  int per_sm = 0;
  cudaError_t e = prepare(qk_bulk_kernel<D, NEOX, WARPS, NS, STAGE_BYTES, TILED>,
                          WARPS * 32, smem_bytes<D, WARPS, NS, STAGE_BYTES>(), cache, &per_sm);
  if (e != cudaSuccess) return e;
  BulkParams p;
  memset(&p.rows_map, 0, sizeof p.rows_map);
  p.qkv = static_cast<__nv_bfloat16*>(a.qkv);
  p.q_weight = static_cast<const __nv_bfloat16*>(a.q_weight);
  p.k_weight = static_cast<const __nv_bfloat16*>(a.k_weight);
  p.cos_sin = a.cos_sin;
  p.positions = a.positions;
  p.num_q = a.num_heads_q;
  p.num_rows = a.num_heads_q + a.num_heads_k;
  p.row_elems = (int64_t)(p.num_rows + a.num_heads_v) * D;
  p.rot = a.rotary_dim;
  chunking(a, STAGE_BYTES / (2 * D), &p.chunks, &p.chunk_rows);
  p.items = a.num_tokens * p.chunks;
  p.eps = a.eps;
  p.wait_limit = stage_wait_limit();
  if (TILED) {
    // [T][Hq + Hk][D] view: a token's V rows lie outside it.
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.num_rows, (cuuint64_t)a.num_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.row_elems * 2};
    const cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)p.chunk_rows, 1};
    if (!encode_bf16_3d(&p.rows_map, p.qkv, dims, strides, box))
      return launch_layout<D, NEOX, WARPS, NS, STAGE_BYTES, false>(a, stream);
  }
  int64_t grid = (int64_t)per_sm * device_sm_count();
  const int64_t need = (p.items + WARPS - 1) / WARPS;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  return launch_kernel(qk_bulk_kernel<D, NEOX, WARPS, NS, STAGE_BYTES, TILED>,
                       dim3((unsigned)grid), dim3(WARPS * 32),
                       smem_bytes<D, WARPS, NS, STAGE_BYTES>(), stream, p);
}

template <int WARPS, int NS, int STAGE_BYTES, bool TILED>
cudaError_t launch_shape(const QkArgs& a, cudaStream_t stream) {
  const bool neox = a.is_neox != 0;
  switch (a.head_dim) {
    case 64:
      return neox ? launch_layout<64, true, WARPS, NS, STAGE_BYTES, TILED>(a, stream)
                  : launch_layout<64, false, WARPS, NS, STAGE_BYTES, TILED>(a, stream);
    case 128:
      return neox ? launch_layout<128, true, WARPS, NS, STAGE_BYTES, TILED>(a, stream)
                  : launch_layout<128, false, WARPS, NS, STAGE_BYTES, TILED>(a, stream);
    case 256:
      return neox ? launch_layout<256, true, WARPS, NS, STAGE_BYTES, TILED>(a, stream)
                  : launch_layout<256, false, WARPS, NS, STAGE_BYTES, TILED>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool qk_bulk_eligible(const QkArgs& a, int shape) {
  static constexpr int kStageBytes[] = {
#define KVQ_STAGE(W, S, KB, T) KB * 1024,
      KVQ_QK_BULK_SHAPES(KVQ_STAGE)
#undef KVQ_STAGE
  };
  if (shape < 0 || shape >= kQkBulkShapes) return false;
  if (a.head_dim != 64 && a.head_dim != 128 && a.head_dim != 256) return false;
  int chunks = 0, chunk_rows = 0;
  chunking(a, kStageBytes[shape] / (2 * a.head_dim), &chunks, &chunk_rows);
  if ((int64_t)(chunks - 1) * chunk_rows >= a.num_heads_q + a.num_heads_k) return false;
  return device_memory(a.qkv) && device_memory(a.cos_sin);
}

cudaError_t stage_events(uint64_t out[2], bool reset) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned long long v[2] = {0, 0};
  e = cudaMemcpyFromSymbol(v, g_stage_events, sizeof v);
  if (e != cudaSuccess) return e;
  out[0] = v[0];
  out[1] = v[1];
  if (reset) {
    const unsigned long long zero[2] = {0, 0};
    e = cudaMemcpyToSymbol(g_stage_events, zero, sizeof zero);
  }
  return e;
}

cudaError_t launch_qk_bulk(const QkArgs& a, int shape, cudaStream_t stream) {
  using Launch = cudaError_t (*)(const QkArgs&, cudaStream_t);
  static constexpr Launch kLaunch[] = {
#define KVQ_LAUNCH(W, S, KB, T) &launch_shape<W, S, KB * 1024, T != 0>,
      KVQ_QK_BULK_SHAPES(KVQ_LAUNCH)
#undef KVQ_LAUNCH
  };
  if (shape < 0 || shape >= kQkBulkShapes) return cudaErrorInvalidValue;
  return kLaunch[shape](a, stream);
}

}  // namespace kvq
