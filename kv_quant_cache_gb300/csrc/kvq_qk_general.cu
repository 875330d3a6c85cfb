// kvq_qk_general.cu -- packed-QKV per-head RMSNorm + RoPE for every supported
// layout: head_dim 64 / 128 / 256, NeoX or GPT-J (interleaved) pairs, full or
// partial rotation.
//
// Operator: InfiniOps PR #1019 ("Add the NineToothed NVIDIA implementation of
// FusedQkNormRope"), section "Summary": the API aligned with vLLM's
// fused_qk_norm_rope carries is_neox; the InfiniOps fast path is guarded to
// head_dim 128, full-dimension NeoX ("Notes for Reviewers").  This kernel
// covers the rest of that API: partial rotation applies to the first
// rotary_dim dims of each head (cos/sin table [max_pos, rotary_dim]); NeoX
// pairs (i, i + rotary_dim/2), GPT-J pairs (2i, 2i+1), i < rotary_dim/2; the
// dims from rotary_dim on are normalised only.
//
// Mapping on sm_103a.  The lane geometry and the row arithmetic are those
// of kvq_qk_general_row.cuh: each lane holds two fragments of F dims, so a
// head row takes D/(2F) lanes and a warp covers 32*2F/D rows per step.  Work
// items are (token, chunk of rows): the position and the lane's cosines and
// sines are fetched once per item and every row load of the item is issued
// before any arithmetic.  rotary_dim is a multiple of 16, so every fragment,
// cosine and sine access is naturally aligned.
#include "kvq_device.cuh"
#include "kvq_launch.h"
#include "kvq_qk_general_row.cuh"

namespace kvq {
namespace {

struct GenParams {
  __nv_bfloat16* qkv;
  const __nv_bfloat16* q_weight;
  const __nv_bfloat16* k_weight;
  const float* cos_sin;
  const int64_t* positions;
  int64_t row_elems;  // (Hq + Hk + Hv) * D
  int num_q, num_rows;
  int rot;
  int chunks, steps, items;
  float eps;
  int64_t max_pos;  // bounds-checked launches: rows of cos_sin
  int* errors;      // bounds-checked launches: tokens rejected
  int trigger_from; // first CTA of the last wave
};

using qkgen::Frag;
using qkgen::Lane;

template <int D, int F, int STEPS, bool NEOX, bool CHECKED>
__global__ void __launch_bounds__(128)
qk_general_kernel(const GenParams p) {
  grid_dependency_sync(p.trigger_from);
  using V = typename Frag<F>::T;
  constexpr int LPR = D / (2 * F);  // lanes per row
  constexpr int RPW = 32 / LPR;     // rows per warp step
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (item >= p.items) return;  // whole warp leaves together
  const int g = lane / LPR, l = lane % LPR;

  const int t = item / p.chunks;
  const int c = item - t * p.chunks;
  const int first = c * p.steps * RPW + g;
  const int last = min(p.num_rows, (c + 1) * p.steps * RPW);
  __nv_bfloat16* tok = p.qkv + (size_t)t * (size_t)p.row_elems;
  const Lane<D, F, NEOX> ln(l, p.rot);
  const int oa = ln.oa, ob = ln.ob;

  V xa[STEPS], xb[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int h = first + RPW * s;
    xa[s] = xb[s] = Frag<F>::zero();
    if (s < p.steps && h < last) {
      const __nv_bfloat16* row = tok + (size_t)h * D;
      xa[s] = __ldcs(reinterpret_cast<const V*>(row + oa));
      xb[s] = __ldcs(reinterpret_cast<const V*>(row + ob));
    }
  }

  // Checked launches: a token whose position is outside the table keeps its
  // rows unchanged and is counted once, by the item holding its first chunk.
  if (CHECKED) {
    const int64_t pos = __ldg(p.positions + t);
    if (pos < 0 || pos >= p.max_pos) {  // warp-uniform
      if (c == 0 && lane == 0) atomicAdd(p.errors, 1);
      return;
    }
  }
  float cs[F], sn[F];
  qkgen::lane_angles<D, F, NEOX, true>(p.cos_sin + __ldg(p.positions + t) * p.rot, l, p.rot, ln,
                                       cs, sn);
  const V wqa = __ldg(reinterpret_cast<const V*>(p.q_weight + oa));
  const V wqb = __ldg(reinterpret_cast<const V*>(p.q_weight + ob));
  const V wka = __ldg(reinterpret_cast<const V*>(p.k_weight + oa));
  const V wkb = __ldg(reinterpret_cast<const V*>(p.k_weight + ob));

#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    if (s >= p.steps || first - g + RPW * s >= last) break;  // warp-uniform
    const int h = first + RPW * s;
    const bool is_q = h < p.num_q;
    qkgen::row_math<D, F, NEOX, false>(xa[s], xb[s], is_q ? wqa : wka, is_q ? wqb : wkb, cs, sn, ln,
                                p.eps);
    if (h < last) {
      __nv_bfloat16* row = tok + (size_t)h * D;
      __stcs(reinterpret_cast<V*>(row + oa), xa[s]);
      __stcs(reinterpret_cast<V*>(row + ob), xb[s]);
    }
  }
}

template <int D, int F, int STEPS, bool NEOX, bool CHECKED>
cudaError_t launch(const QkArgs& a, cudaStream_t stream) {
  constexpr int RPW = 32 / (D / (2 * F));
  GenParams p;
  p.qkv = static_cast<__nv_bfloat16*>(a.qkv);
  p.q_weight = static_cast<const __nv_bfloat16*>(a.q_weight);
  p.k_weight = static_cast<const __nv_bfloat16*>(a.k_weight);
  p.cos_sin = a.cos_sin;
  p.positions = a.positions;
  p.num_q = a.num_heads_q;
  p.num_rows = a.num_heads_q + a.num_heads_k;
  p.row_elems = (int64_t)(p.num_rows + a.num_heads_v) * D;
  p.rot = a.rotary_dim;
  p.eps = a.eps;
  p.max_pos = a.max_pos;
  p.errors = a.errors;
  const int groups = (p.num_rows + RPW - 1) / RPW;  // row groups of one warp step
  p.chunks = (groups + STEPS - 1) / STEPS;
  p.steps = (groups + p.chunks - 1) / p.chunks;
  p.items = a.num_tokens * p.chunks;
  const unsigned grid = (unsigned)((p.items + 3) / 4);
  static std::atomic<int> cache[kMaxDevices];
  p.trigger_from = last_wave_start(qk_general_kernel<D, F, STEPS, NEOX, CHECKED>, 128, grid, cache);
  return launch_kernel(qk_general_kernel<D, F, STEPS, NEOX, CHECKED>, dim3(grid), dim3(128), 0,
                       stream, p);
}

// Small batches: one warp step per item (widest spread); large batches: up to
// BIG warp steps per item (each item's loads in flight together), the chunks
// of a token balanced in length.
template <int D, int F, int BIG, bool CHECKED>
cudaError_t launch_c(const QkArgs& a, bool small, cudaStream_t stream) {
  if (a.is_neox)
    return small ? launch<D, F, 1, true, CHECKED>(a, stream)
                 : launch<D, F, BIG, true, CHECKED>(a, stream);
  return small ? launch<D, F, 1, false, CHECKED>(a, stream)
               : launch<D, F, BIG, false, CHECKED>(a, stream);
}

template <int D, int F, int BIG>
cudaError_t launch_d(const QkArgs& a, bool small, cudaStream_t stream) {
  return a.errors != nullptr ? launch_c<D, F, BIG, true>(a, small, stream)
                             : launch_c<D, F, BIG, false>(a, small, stream);
}

template <int F, int BIG>
cudaError_t launch_f(const QkArgs& a, bool small, cudaStream_t stream) {
  switch (a.head_dim) {
    case 64: return launch_d<64, F, BIG>(a, small, stream);
    case 128: return launch_d<128, F, BIG>(a, small, stream);
    case 256: return launch_d<256, F, BIG>(a, small, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_qk_general(const QkArgs& a, bool small, int frag, cudaStream_t stream) {
  return frag == 8 ? launch_f<8, 2>(a, small, stream) : launch_f<4, 4>(a, small, stream);
}

}  // namespace kvq
