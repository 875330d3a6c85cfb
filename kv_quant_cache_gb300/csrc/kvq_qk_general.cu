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
// Mapping on sm_103a.  Each lane holds two fragments of F dims (F = 4: two
// 8-byte loads; F = 8: two 16-byte loads), so a head row takes D/(2F) lanes
// and a warp covers 32*2F/D rows per step; the sum of squares is a butterfly
// inside the row's lane group.  Every rotated pair is held by one lane, so the
// rotation needs no shuffle, and each of the two load instructions reads a
// contiguous span across the row's lanes (whole sectors):
//   * NeoX: lane l < rot/(2F) holds dims [F l, F l + F) and their partners
//     [rot/2 + F l, ...); the remaining lanes split the unrotated tail
//     [rot, D) the same way, its first half in one fragment, its second half
//     in the other;
//   * GPT-J: lane l holds dims [F l, F l + F) and [D/2 + F l, ...); a pair
//     (2i, 2i+1) never straddles a fragment, and a fragment lies wholly below
//     or wholly above rot (a multiple of 16).
// The fragment width and the pairing style are template parameters, so each
// instantiation carries only its own registers.  Work items are (token, chunk
// of rows): the position and the lane's cosines and sines are fetched once
// per item and every row load of the item is issued before any arithmetic.
// rotary_dim is a multiple of 16, so every fragment, cosine and sine access
// is naturally aligned.
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

// A fragment of F bf16 values.
template <int F> struct Frag;
template <> struct Frag<4> {
  using T = uint2;
  static __device__ __forceinline__ T zero() { return make_uint2(0u, 0u); }
  static __device__ __forceinline__ void unpack(const uint2& v, float* f) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
  }
  static __device__ __forceinline__ uint2 pack(const float* f) {
    return make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
  }
};
template <> struct Frag<8> {
  using T = uint4;
  static __device__ __forceinline__ T zero() { return make_uint4(0u, 0u, 0u, 0u); }
  static __device__ __forceinline__ void unpack(const uint4& v, float* f) { unpack_bf16x8(v, f); }
  static __device__ __forceinline__ uint4 pack(const float* f) { return pack_bf16x8(f); }
};

// N consecutive fp32 values, N = 2, 4 or 8 (the address is 8-byte aligned for
// N = 2, 16-byte aligned otherwise).
template <int N>
__device__ __forceinline__ void load_f32(const float* src, float* dst) {
  if constexpr (N == 2) {
    const float2 v = __ldg(reinterpret_cast<const float2*>(src));
    dst[0] = v.x;
    dst[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < N; k += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src + k));
      dst[k] = v.x;
      dst[k + 1] = v.y;
      dst[k + 2] = v.z;
      dst[k + 3] = v.w;
    }
  }
}

// Rotate pairs (v[2j], v[2j+1]) of one fragment by angles (c[j], s[j]).
template <int F>
__device__ __forceinline__ void rotate_interleaved(float* v, const float* c, const float* s) {
#pragma unroll
  for (int j = 0; j < F / 2; ++j) {
    const float e = v[2 * j], o = v[2 * j + 1];
    v[2 * j] = fmaf(e, c[j], -o * s[j]);
    v[2 * j + 1] = fmaf(o, c[j], e * s[j]);
  }
}

template <int D, int F, int STEPS, bool NEOX, bool CHECKED>
__global__ void __launch_bounds__(128)
qk_general_kernel(const GenParams p) {
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
  const int half = p.rot / 2;
  int oa, ob;          // element offsets of the lane's two fragments
  bool rot_a, rot_b;   // which of them are rotated
  if (NEOX) {
    const int lr = p.rot / (2 * F);  // lanes holding rotated pairs
    if (l < lr) {
      oa = F * l;
      ob = half + F * l;
    } else {
      oa = p.rot + F * (l - lr);
      ob = oa + (D - p.rot) / 2;
    }
    rot_a = rot_b = l < lr;
  } else {
    oa = F * l;
    ob = D / 2 + F * l;
    rot_a = oa < p.rot;
    rot_b = ob < p.rot;
  }

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
  // Cosines and sines.  NeoX: frequency F l + k for the pair (a[k], b[k]).
  // GPT-J: fragment a's pairs have frequencies F l/2 + j, fragment b's
  // D/4 + F l/2 + j (j < F/2), kept in slots j and F/2 + j.
  float cs[F], sn[F];
#pragma unroll
  for (int k = 0; k < F; ++k) cs[k] = sn[k] = 0.0f;
  if (rot_a || rot_b) {
    const float* row = p.cos_sin + __ldg(p.positions + t) * p.rot;
    if (NEOX) {
      load_f32<F>(row + F * l, cs);
      load_f32<F>(row + half + F * l, sn);
    } else {
      if (rot_a) {
        load_f32<F / 2>(row + F * l / 2, cs);
        load_f32<F / 2>(row + half + F * l / 2, sn);
      }
      if (rot_b) {
        load_f32<F / 2>(row + D / 4 + F * l / 2, cs + F / 2);
        load_f32<F / 2>(row + half + D / 4 + F * l / 2, sn + F / 2);
      }
    }
  }
  const V wqa = __ldg(reinterpret_cast<const V*>(p.q_weight + oa));
  const V wqb = __ldg(reinterpret_cast<const V*>(p.q_weight + ob));
  const V wka = __ldg(reinterpret_cast<const V*>(p.k_weight + oa));
  const V wkb = __ldg(reinterpret_cast<const V*>(p.k_weight + ob));

#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    if (s >= p.steps || first - g + RPW * s >= last) break;  // warp-uniform
    const int h = first + RPW * s;
    float a[F], b[F], wa[F], wb[F];
    Frag<F>::unpack(xa[s], a);
    Frag<F>::unpack(xb[s], b);
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < F; ++k) ss = fmaf(b[k], b[k], fmaf(a[k], a[k], ss));
    ss = group_sum<LPR>(ss);
    const float r = __frsqrt_rn(ss * (1.0f / D) + p.eps);
    const bool is_q = h < p.num_q;
    Frag<F>::unpack(is_q ? wqa : wka, wa);
    Frag<F>::unpack(is_q ? wqb : wkb, wb);
    float na[F], nb[F];
#pragma unroll
    for (int k = 0; k < F; ++k) {
      na[k] = a[k] * r * wa[k];
      nb[k] = b[k] * r * wb[k];
    }
    if (NEOX) {
      if (rot_a) {  // pair (a[k], b[k])
#pragma unroll
        for (int k = 0; k < F; ++k) {
          const float x0 = na[k], x1 = nb[k];
          na[k] = fmaf(x0, cs[k], -x1 * sn[k]);
          nb[k] = fmaf(x1, cs[k], x0 * sn[k]);
        }
      }
    } else {
      if (rot_a) rotate_interleaved<F>(na, cs, sn);
      if (rot_b) rotate_interleaved<F>(nb, cs + F / 2, sn + F / 2);
    }
    if (h < last) {
      __nv_bfloat16* row = tok + (size_t)h * D;
      __stcs(reinterpret_cast<V*>(row + oa), Frag<F>::pack(na));
      __stcs(reinterpret_cast<V*>(row + ob), Frag<F>::pack(nb));
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
  qk_general_kernel<D, F, STEPS, NEOX, CHECKED><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
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
