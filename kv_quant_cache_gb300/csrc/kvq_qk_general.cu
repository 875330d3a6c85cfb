// kvq_qk_general.cu -- packed-QKV per-head RMSNorm + RoPE for the layouts
// outside the tuned full-NeoX head_dim-128 kernel: head_dim 64 / 128 / 256,
// NeoX or GPT-J (interleaved) pairs, full or partial rotation.
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
// Mapping on sm_103a.  D/8 lanes per head row, 8 dims per lane, so a warp
// covers 32*8/D rows per step (4 at D = 64, 2 at 128, 1 at 256); the sum of
// squares is a butterfly inside the row's lane group.  Every rotated pair is
// held by one lane, so the rotation needs no shuffle:
//   * NeoX: lane l < rot/8 holds dims [4l, 4l+4) and their partners
//     [rot/2 + 4l, rot/2 + 4l + 4) (two 8-byte loads, each contiguous across
//     those lanes); lanes from rot/8 on hold the unrotated tail [rot, D) in
//     8-dim pieces;
//   * GPT-J: lane l holds dims [8l, 8l+8) (one 16-byte load); its four pairs
//     (2i, 2i+1) are inside it.
// The pairing style is a template parameter, so each kernel carries only its
// own registers.  Work items are (token, chunk of rows) as in the tuned
// kernel: the position and the lane's 4 cosines and 4 sines are fetched once
// per item and every row load of the item is issued before any arithmetic.
#include "kvq_device.cuh"
#include "kvq_launch.h"

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
};

__device__ __forceinline__ void unpack4(const uint2& v, float* f) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xffff0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xffff0000u);
}

__device__ __forceinline__ uint2 pack4(const float* f) {
  return make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
}

// Element offsets (within a head row) of the lane's two 4-dim fragments.
template <bool NEOX>
__device__ __forceinline__ void fragment_offsets(int l, int rot, int& a, int& b) {
  if (NEOX) {
    if (4 * l < rot / 2) {
      a = 4 * l;
      b = rot / 2 + 4 * l;
    } else {
      a = rot + 8 * (l - rot / 8);
      b = a + 4;
    }
  } else {
    a = 8 * l;
    b = a + 4;
  }
}

template <int D, int STEPS, bool NEOX, bool CHECKED>
__global__ void __launch_bounds__(128)
qk_general_kernel(const GenParams p) {
  constexpr int LPR = D / 8;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp step
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (item >= p.items) return;  // whole warp leaves together
  const int g = lane / LPR, l = lane % LPR;

  const int t = item / p.chunks;
  const int c = item - t * p.chunks;
  const int first = c * p.steps * RPW + g;
  const int last = min(p.num_rows, (c + 1) * p.steps * RPW);
  __nv_bfloat16* tok = p.qkv + (size_t)t * (size_t)p.row_elems;
  int oa, ob;
  fragment_offsets<NEOX>(l, p.rot, oa, ob);
  const bool rot_lane = NEOX ? (4 * l < p.rot / 2) : (8 * l < p.rot);

  uint2 xa[STEPS], xb[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int h = first + RPW * s;
    xa[s] = xb[s] = make_uint2(0u, 0u);
    if (s < p.steps && h < last) {
      const __nv_bfloat16* row = tok + (size_t)h * D;
      xa[s] = __ldcs(reinterpret_cast<const uint2*>(row + oa));
      xb[s] = __ldcs(reinterpret_cast<const uint2*>(row + ob));
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
  // Cosines and sines of the lane's four pairs: frequency 4l + k.
  float cs[4] = {0.f, 0.f, 0.f, 0.f}, sn[4] = {0.f, 0.f, 0.f, 0.f};
  if (rot_lane) {
    const float* row = p.cos_sin + __ldg(p.positions + t) * p.rot;
    const float4 cv = __ldg(reinterpret_cast<const float4*>(row + 4 * l));
    const float4 sv = __ldg(reinterpret_cast<const float4*>(row + p.rot / 2 + 4 * l));
    cs[0] = cv.x; cs[1] = cv.y; cs[2] = cv.z; cs[3] = cv.w;
    sn[0] = sv.x; sn[1] = sv.y; sn[2] = sv.z; sn[3] = sv.w;
  }
  const uint2 wqa = __ldg(reinterpret_cast<const uint2*>(p.q_weight + oa));
  const uint2 wqb = __ldg(reinterpret_cast<const uint2*>(p.q_weight + ob));
  const uint2 wka = __ldg(reinterpret_cast<const uint2*>(p.k_weight + oa));
  const uint2 wkb = __ldg(reinterpret_cast<const uint2*>(p.k_weight + ob));

#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    if (s >= p.steps || first - g + RPW * s >= last) break;  // warp-uniform
    const int h = first + RPW * s;
    float a[4], b[4], wa[4], wb[4];
    unpack4(xa[s], a);
    unpack4(xb[s], b);
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) ss = fmaf(b[k], b[k], fmaf(a[k], a[k], ss));
    ss = group_sum<LPR>(ss);
    const float r = __frsqrt_rn(ss * (1.0f / D) + p.eps);
    const bool is_q = h < p.num_q;
    unpack4(is_q ? wqa : wka, wa);
    unpack4(is_q ? wqb : wkb, wb);
    float na[4], nb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      na[k] = a[k] * r * wa[k];
      nb[k] = b[k] * r * wb[k];
    }
    if (rot_lane) {
      if (NEOX) {  // pair (a[k], b[k]), frequency 4l + k
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x0 = na[k], x1 = nb[k];
          na[k] = fmaf(x0, cs[k], -x1 * sn[k]);
          nb[k] = fmaf(x1, cs[k], x0 * sn[k]);
        }
      } else {  // pairs (a0,a1), (a2,a3), (b0,b1), (b2,b3): frequencies 4l..4l+3
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float* v = j == 0 ? na : nb;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int k = 2 * j + q;
            const float e = v[2 * q], o = v[2 * q + 1];
            v[2 * q] = fmaf(e, cs[k], -o * sn[k]);
            v[2 * q + 1] = fmaf(o, cs[k], e * sn[k]);
          }
        }
      }
    }
    if (h < last) {
      __nv_bfloat16* row = tok + (size_t)h * D;
      __stcs(reinterpret_cast<uint2*>(row + oa), pack4(na));
      __stcs(reinterpret_cast<uint2*>(row + ob), pack4(nb));
    }
  }
}

template <int D, int STEPS, bool NEOX, bool CHECKED>
cudaError_t launch(const QkArgs& a, cudaStream_t stream) {
  constexpr int RPW = 32 / (D / 8);
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
  qk_general_kernel<D, STEPS, NEOX, CHECKED><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

// Large batches: up to BIG warp steps per item, chunks of a token balanced in
// length.  (Six steps for head_dim 64, which would split 40 rows into two
// equal chunks, measured no faster: the extra registers cost the occupancy
// the balancing gained.)
template <int D, int BIG, bool CHECKED>
cudaError_t launch_c(const QkArgs& a, bool small, cudaStream_t stream) {
  if (a.is_neox)
    return small ? launch<D, 1, true, CHECKED>(a, stream) : launch<D, BIG, true, CHECKED>(a, stream);
  return small ? launch<D, 1, false, CHECKED>(a, stream) : launch<D, BIG, false, CHECKED>(a, stream);
}

template <int D, int BIG>
cudaError_t launch_d(const QkArgs& a, bool small, cudaStream_t stream) {
  return a.errors != nullptr ? launch_c<D, BIG, true>(a, small, stream)
                             : launch_c<D, BIG, false>(a, small, stream);
}

}  // namespace

cudaError_t launch_qk_general(const QkArgs& a, bool small, cudaStream_t stream) {
  switch (a.head_dim) {
    case 64: return launch_d<64, 4>(a, small, stream);
    case 128: return launch_d<128, 4>(a, small, stream);
    case 256: return launch_d<256, 4>(a, small, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
