// kvq_qk_norm_rope.cu -- packed-QKV per-head RMSNorm + NeoX RoPE, in place.
//
// Operator: InfiniOps PR #1019 ("Add the NineToothed NVIDIA implementation of
// FusedQkNormRope"), section "Summary": Q and K heads of a packed
// [T, (Hq+Hk+Hv)*D] bf16 tensor get per-head RMSNorm followed by NeoX RoPE in
// place, V untouched, separate [D] weights, and the NeoX partner read with
// its own dimension's weight.  This file covers the guarded case of "Notes
// for Reviewers": bf16, D = 128, full-dimension NeoX rotation.
//
// Mapping on sm_103a.  A 128-dim bf16 head row is 256 bytes; a half-warp
// takes one row, so a warp covers two rows per step (lanes 0-15 row h, lanes
// 16-31 row h+1).  Lane l (of 16) holds dims [4l, 4l+4) and their NeoX
// partners [64+4l, 64+4l+4) -- two 8-byte loads that each form, across the
// half-warp, one contiguous 128-byte segment -- so the rotation is local to
// the lane: no shuffle brings the partner in, and each element of a pair is
// weighted with its own dimension's weight before rotating.  The sum of
// squares is a 4-step butterfly inside the half-warp.  A work item is
// (token, chunk of consecutive Q/K head rows, at most 2*STEPS, chunks of a
// token balanced in length): the token's position and the lane's 4 cosines
// and 4 sines are fetched once per item and reused for every row, and all
// row loads of an item are issued before any arithmetic.  V columns are
// never addressed.  Two kernel shapes share the row arithmetic (so every
// launch shape gives bit-identical results):
//   * tiles:  one work item per warp, one-shot grid;
//   * stream: persistent grid sized to the resident-CTA capacity, each warp
//     taking grid-stride work items, weights loaded once per warp.
// (A persistent variant that keeps the next item's loads in flight, the
// shape that wins for the DSV4 operator, measured 45-71 % here and is not
// kept: at 74-86 registers it holds too few warps.)
#include "kvq_device.cuh"
#include "kvq_launch.h"
#include "kvq_qk_bulk.h"
#include "kvq_qk_general_row.cuh"

namespace kvq {
namespace {

constexpr int kHeadDim = 128;
constexpr int kHalf = kHeadDim / 2;

struct QkParams {
  __nv_bfloat16* qkv;
  const __nv_bfloat16* q_weight;
  const __nv_bfloat16* k_weight;
  const float* cos_sin;
  const int64_t* positions;
  int64_t row_elems;  // (Hq + Hk + Hv) * 128
  int num_tokens;
  int num_q;          // Hq
  int num_rows;       // Hq + Hk
  int chunks;         // work items per token
  int steps;          // row pairs per chunk (<= the kernel's STEPS)
  int items;          // num_tokens * chunks
  float eps;
  int64_t max_pos;    // bounds-checked launches: rows of cos_sin
  int* errors;        // bounds-checked launches: tokens rejected
  int trigger_from;   // one-shot launches: first CTA of the last wave
};

// Weight fragments of this lane (dims [4l, 4l+4) and [64+4l, 64+4l+4), Q and
// K), kept packed as bf16 and widened where they are used.
struct QkWeights {
  uint2 q_lo, q_hi, k_lo, k_hi;
};

__device__ __forceinline__ void load_weights(const QkParams& p, int l16, QkWeights& w) {
  const uint2* q = reinterpret_cast<const uint2*>(p.q_weight);
  const uint2* k = reinterpret_cast<const uint2*>(p.k_weight);
  w.q_lo = __ldg(q + l16);
  w.q_hi = __ldg(q + 16 + l16);
  w.k_lo = __ldg(k + l16);
  w.k_hi = __ldg(k + 16 + l16);
}

// Normalise + rotate one row fragment; all 32 lanes must call it together
// (the sum of squares is reduced across the half-warp).  The arithmetic is
// that of every layout (kvq_qk_general_row.cuh) at head_dim 128, NeoX, full
// rotation, whose lane geometry is this kernel's: every launch shape of the
// operator gives the same bits.
__device__ __forceinline__ void row_math(uint2& lo, uint2& hi, bool is_q, const QkWeights& w,
                                         const float4& c4, const float4& s4, float eps) {
  const float c[4] = {c4.x, c4.y, c4.z, c4.w};
  const float s[4] = {s4.x, s4.y, s4.z, s4.w};
  const qkgen::Lane<kHeadDim, 4, true> full(0, kHeadDim);  // both fragments rotated
  qkgen::row_math<kHeadDim, 4, true, false>(lo, hi, is_q ? w.q_lo : w.k_lo, is_q ? w.q_hi : w.k_hi, c, s,
                                     full, eps);
}

// The lane's 4 cosines and 4 sines of the token's row.
__device__ __forceinline__ void load_cos_sin(const QkParams& p, int t, int l16, float4& c,
                                             float4& s) {
  const int64_t pos = __ldg(p.positions + t);
  const float4* crow = reinterpret_cast<const float4*>(p.cos_sin + pos * kHeadDim);
  c = __ldg(crow + l16);
  s = __ldg(crow + kHalf / 4 + l16);
}

// One work item's rows as held by a lane: STEPS row fragments plus the
// token's cosines and sines for the lane's 4 frequencies.
template <int STEPS>
struct ItemRegs {
  uint2 lo[STEPS], hi[STEPS];
  float4 c, s;
  bool ok;  // bounds-checked launches: the position lies inside the table
};

// Work item `item` = (token t, chunk c of row pairs).  Lanes 0-15 take rows
// first, first+2, ..; lanes 16-31 the rows after them.
struct ItemPos {
  int t, first, last;  // token, this lane's first row, end of the chunk
};

__device__ __forceinline__ ItemPos item_pos(const QkParams& p, int item, int half) {
  ItemPos ip;
  ip.t = item / p.chunks;
  const int c = item - ip.t * p.chunks;
  ip.first = c * (2 * p.steps) + half;
  ip.last = min(p.num_rows, (c + 1) * (2 * p.steps));
  return ip;
}

template <int STEPS, bool CHECKED>
__device__ __forceinline__ void load_item(const QkParams& p, const ItemPos& ip, int l16,
                                          ItemRegs<STEPS>& r) {
  const __nv_bfloat16* tok = p.qkv + (size_t)ip.t * (size_t)p.row_elems;
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int h = ip.first + 2 * s;
    r.lo[s] = r.hi[s] = make_uint2(0u, 0u);
    if (h < ip.last) {
      const uint2* row = reinterpret_cast<const uint2*>(tok + (size_t)h * kHeadDim);
      r.lo[s] = __ldcs(row + l16);
      r.hi[s] = __ldcs(row + 16 + l16);
    }
  }
  r.ok = true;
  if (CHECKED) {  // no cos/sin row outside the table is read
    const int64_t pos = __ldg(p.positions + ip.t);
    r.ok = pos >= 0 && pos < p.max_pos;
    if (!r.ok) return;
  }
  load_cos_sin(p, ip.t, l16, r.c, r.s);
}

// A token whose position is outside the table (checked launches) keeps its
// rows unchanged and is counted once, by the item holding its first chunk.
template <int STEPS, bool CHECKED>
__device__ __forceinline__ void compute_item(const QkParams& p, const ItemPos& ip, int half,
                                             int l16, const QkWeights& w, ItemRegs<STEPS>& r) {
  if (CHECKED && !r.ok) {  // warp-uniform
    if (ip.first == 0 && l16 == 0) atomicAdd(p.errors, 1);
    return;
  }
  __nv_bfloat16* tok = p.qkv + (size_t)ip.t * (size_t)p.row_elems;
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    if (ip.first - half + 2 * s >= ip.last) break;  // warp-uniform: no row left in the chunk
    const int h = ip.first + 2 * s;
    row_math(r.lo[s], r.hi[s], h < p.num_q, w, r.c, r.s, p.eps);
    if (h < ip.last) {
      uint2* row = reinterpret_cast<uint2*>(tok + (size_t)h * kHeadDim);
      __stcs(row + l16, r.lo[s]);
      __stcs(row + 16 + l16, r.hi[s]);
    }
  }
}

template <int STEPS, bool CHECKED = false>
__device__ __forceinline__ void do_item(const QkParams& p, int item, int half, int l16,
                                        const QkWeights& w) {
  const ItemPos ip = item_pos(p, item, half);
  ItemRegs<STEPS> r;
  load_item<STEPS, CHECKED>(p, ip, l16, r);
  compute_item<STEPS, CHECKED>(p, ip, half, l16, w, r);
}

template <int WARPS, int STEPS, int MINB, bool CHECKED>
__global__ void __launch_bounds__(WARPS * 32, MINB)
qk_tiles_kernel(const QkParams p) {
  grid_dependency_sync(p.trigger_from);
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (item >= p.items) return;  // whole warp leaves together
  QkWeights w;
  load_weights(p, lane & 15, w);
  do_item<STEPS, CHECKED>(p, item, lane >> 4, lane & 15, w);
}

template <int WARPS, int STEPS, int MINB>
__global__ void __launch_bounds__(WARPS * 32, MINB)
qk_stream_kernel(const QkParams p) {
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = gridDim.x * WARPS;
  if (gw >= p.items) return;
  QkWeights w;
  load_weights(p, lane & 15, w);
  for (int item = gw; item < p.items; item += nw) do_item<STEPS>(p, item, lane >> 4, lane & 15, w);
}

QkParams make_params(const QkArgs& a, int steps) {
  QkParams p;
  p.qkv = static_cast<__nv_bfloat16*>(a.qkv);
  p.q_weight = static_cast<const __nv_bfloat16*>(a.q_weight);
  p.k_weight = static_cast<const __nv_bfloat16*>(a.k_weight);
  p.cos_sin = a.cos_sin;
  p.positions = a.positions;
  p.num_rows = a.num_heads_q + a.num_heads_k;
  p.row_elems = (int64_t)(p.num_rows + a.num_heads_v) * kHeadDim;
  p.num_tokens = a.num_tokens;
  p.num_q = a.num_heads_q;
  // Balanced chunks: as few as STEPS allows, then as short as possible.
  const int pairs = (p.num_rows + 1) / 2;
  p.chunks = (pairs + steps - 1) / steps;
  p.steps = (pairs + p.chunks - 1) / p.chunks;
  p.items = p.num_tokens * p.chunks;
  p.eps = a.eps;
  p.max_pos = a.max_pos;
  p.errors = a.errors;
  p.trigger_from = 0;
  return p;
}

template <int WARPS, int STEPS, int MINB, bool CHECKED = false>
cudaError_t launch_tiles(const QkArgs& a, cudaStream_t stream) {
  QkParams p = make_params(a, STEPS);
  const unsigned grid = (unsigned)((p.items + WARPS - 1) / WARPS);
  static std::atomic<int> cache[kMaxDevices];
  p.trigger_from =
      last_wave_start(qk_tiles_kernel<WARPS, STEPS, MINB, CHECKED>, WARPS * 32, grid, cache);
  return launch_kernel(qk_tiles_kernel<WARPS, STEPS, MINB, CHECKED>, dim3(grid), dim3(WARPS * 32),
                       0, stream, p);
}

template <typename Kernel>
cudaError_t launch_persistent(Kernel kernel, const QkParams& p, int warps,
                              std::atomic<int>* cache, cudaStream_t stream) {
  int per_sm = 0;
  cudaError_t e = resident_ctas(kernel, warps * 32, cache, &per_sm);
  if (e != cudaSuccess) return e;
  int64_t grid = (int64_t)per_sm * device_sm_count();
  const int64_t need = (p.items + warps - 1) / warps;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  return launch_kernel(kernel, dim3((unsigned)grid), dim3(warps * 32), 0, stream, p);
}

template <int WARPS, int STEPS, int MINB>
cudaError_t launch_stream(const QkArgs& a, cudaStream_t stream) {
  static std::atomic<int> cache[kMaxDevices];
  return launch_persistent(qk_stream_kernel<WARPS, STEPS, MINB>, make_params(a, STEPS), WARPS,
                           cache, stream);
}

}  // namespace

const LaunchConfig kQkConfigs[] = {
    {"tiles<4w,1step>"}, {"tiles<8w,2step>"}, {"tiles<4w,4step>"}, {"tiles<8w,4step>"},
    {"stream<8w,4step>"}, {"general<frag4>"}, {"general<frag8>"},
#define KVQ_BULK_NAME(W, S, KB, T) \
  {T ? "bulk<" #W "w," #S "st," #KB "KB,tile>" : "bulk<" #W "w," #S "st," #KB "KB>"},
    KVQ_QK_BULK_SHAPES(KVQ_BULK_NAME)
#undef KVQ_BULK_NAME
};
const int kQkNumConfigs = sizeof(kQkConfigs) / sizeof(kQkConfigs[0]);

cudaError_t launch_qk_norm_rope(const QkArgs& a, int config, cudaStream_t stream) {
  if (a.errors != nullptr) {  // bounds-checked: the two dispatch shapes
    return config == 2 || config >= kQkFirstBulk ? launch_tiles<4, 4, 1, true>(a, stream)
                                                 : launch_tiles<4, 1, 1, true>(a, stream);
  }
  // A staged shape that the call is not eligible for: the register-pipelined
  // large-batch shape (same bits).
  if (config >= kQkFirstBulk) return launch_tiles<4, 4, 1>(a, stream);
  switch (config) {
    case 0: return launch_tiles<4, 1, 1>(a, stream);
    case 1: return launch_tiles<8, 2, 1>(a, stream);
    case 2: return launch_tiles<4, 4, 1>(a, stream);
    case 3: return launch_tiles<8, 4, 1>(a, stream);
    case 4: return launch_stream<8, 4, 1>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
