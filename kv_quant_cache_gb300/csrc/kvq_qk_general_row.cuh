// kvq_qk_general_row.cuh -- the per-row arithmetic of the packed-QKV
// operator for every supported layout: head_dim 64 / 128 / 256, NeoX or
// GPT-J (interleaved) pairs, full or partial rotation (InfiniOps PR #1019,
// "Add the NineToothed NVIDIA implementation of FusedQkNormRope", section
// "Summary": per-head RMSNorm, then RoPE on the first rotary_dim dims; NeoX
// pairs (i, i + rotary_dim/2), GPT-J pairs (2i, 2i+1), i < rotary_dim/2).
// Shared by the register-pipelined kernels (kvq_qk_norm_rope.cu), the
// one-shot general kernel (kvq_qk_general.cu) and the TMA-staged kernel
// (kvq_qk_bulk.cu).
//
// Lane geometry.  A lane holds two fragments of F dims of a row, so a row
// takes D/(2F) lanes; each of the two load instructions reads a contiguous
// span across the row's lanes, and every rotated pair is held by one lane:
//   * NeoX: lane l < rot/(2F) holds dims [F l, F l + F) (fragment a) and
//     their partners [rot/2 + F l, ...) (fragment b); the remaining lanes
//     split the unrotated tail [rot, D) into halves, fragment a in the
//     second half and b in the first.  That order makes one row's a
//     fragments (one load instruction) cover every shared-memory bank
//     equally at head_dim 128 and 256; with a in the first half, the
//     rotated and the tail lanes' a fragments share banks when rot < D
//     (measured on GB300, staged kernel, head_dim 128 with 64 rotated dims:
//     113 against 119 us at 32768 tokens);
//   * GPT-J: lane l holds dims [F l, F l + F) and [D/2 + F l, ...); a pair
//     (2i, 2i+1) never straddles a fragment, and a fragment lies wholly below
//     or wholly above rot (a multiple of 16).
#pragma once

#include "kvq_device.cuh"

namespace kvq {
namespace qkgen {

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
// N = 2, 16-byte aligned otherwise), read through the read-only path from
// global memory (GLOBAL) or with plain loads (shared memory).
template <int N, bool GLOBAL>
__device__ __forceinline__ void load_f32(const float* src, float* dst) {
  if constexpr (N == 2) {
    const float2 v = GLOBAL ? __ldg(reinterpret_cast<const float2*>(src))
                            : *reinterpret_cast<const float2*>(src);
    dst[0] = v.x;
    dst[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < N; k += 4) {
      const float4 v = GLOBAL ? __ldg(reinterpret_cast<const float4*>(src + k))
                              : *reinterpret_cast<const float4*>(src + k);
      dst[k] = v.x;
      dst[k + 1] = v.y;
      dst[k + 2] = v.z;
      dst[k + 3] = v.w;
    }
  }
}

// Element offsets of lane l's two fragments within a head row, and which of
// them are rotated.
template <int D, int F, bool NEOX>
struct Lane {
  int oa, ob;
  bool rot_a, rot_b;
  __device__ __forceinline__ Lane(int l, int rot) {
    if (NEOX) {
      const int lr = rot / (2 * F);  // lanes holding rotated pairs
      if (l < lr) {
        oa = F * l;
        ob = rot / 2 + F * l;
      } else {
        ob = rot + F * (l - lr);
        oa = ob + (D - rot) / 2;
      }
      rot_a = rot_b = l < lr;
    } else {
      oa = F * l;
      ob = D / 2 + F * l;
      rot_a = oa < rot;
      rot_b = ob < rot;
    }
  }
};

// Cosines and sines of lane l's pairs from one cos/sin row (rot/2 cosines,
// then rot/2 sines).  NeoX: frequency F l + k for the pair (a[k], b[k]).
// GPT-J: fragment a's pairs have frequencies F l/2 + j, fragment b's
// D/4 + F l/2 + j (j < F/2), kept in slots j and F/2 + j.  Slots of
// unrotated fragments are left at 0.
template <int D, int F, bool NEOX, bool GLOBAL>
__device__ __forceinline__ void lane_angles(const float* row, int l, int rot,
                                            const Lane<D, F, NEOX>& ln, float* cs, float* sn) {
#pragma unroll
  for (int k = 0; k < F; ++k) cs[k] = sn[k] = 0.0f;
  const int half = rot / 2;
  if (NEOX) {
    if (ln.rot_a) {
      load_f32<F, GLOBAL>(row + F * l, cs);
      load_f32<F, GLOBAL>(row + half + F * l, sn);
    }
  } else {
    if (ln.rot_a) {
      load_f32<F / 2, GLOBAL>(row + F * l / 2, cs);
      load_f32<F / 2, GLOBAL>(row + half + F * l / 2, sn);
    }
    if (ln.rot_b) {
      load_f32<F / 2, GLOBAL>(row + D / 4 + F * l / 2, cs + F / 2);
      load_f32<F / 2, GLOBAL>(row + half + D / 4 + F * l / 2, sn + F / 2);
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

// Normalise + rotate one row's fragments in place (xa, xb packed bf16; wa, wb
// the row's weights at the same dims, as fp32).  All 32 lanes must call it
// together: the sum of squares is reduced across each row's D/(2F) lanes.
// EXACT_RSQRT picks the reciprocal square root: the correctly rounded one,
// or the hardware approximation (rsqrtf, within 2 fp32 ulp; its error is far
// below one bf16 ulp of the outputs).  Measured on GB300: the approximation
// makes the one-shot and register-pipelined kernels 5-13 % faster (they issue
// an instruction on most cycles), but the TMA-staged kernel 8-12 % slower
// (its schedule around the copies changes), so each takes its faster form.
// Kernels on the same form give the same bits; across the two forms an
// output can differ in its last bit where the fp32 value lies next to a bf16
// rounding boundary.
template <int D, int F, bool NEOX, bool EXACT_RSQRT>
__device__ __forceinline__ void row_math_w(typename Frag<F>::T& xa, typename Frag<F>::T& xb,
                                           const float* wa, const float* wb, const float* cs,
                                           const float* sn, const Lane<D, F, NEOX>& ln,
                                           float eps) {
  constexpr int LPR = D / (2 * F);
  float a[F], b[F];
  Frag<F>::unpack(xa, a);
  Frag<F>::unpack(xb, b);
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < F; ++k) ss = fmaf(b[k], b[k], fmaf(a[k], a[k], ss));
  ss = group_sum<LPR>(ss);
  const float v = ss * (1.0f / D) + eps;
  const float r = EXACT_RSQRT ? __frsqrt_rn(v) : rsqrtf(v);
  float na[F], nb[F];
#pragma unroll
  for (int k = 0; k < F; ++k) {
    na[k] = a[k] * r * wa[k];
    nb[k] = b[k] * r * wb[k];
  }
  if (NEOX) {
    if (ln.rot_a) {  // pair (a[k], b[k])
#pragma unroll
      for (int k = 0; k < F; ++k) {
        const float x0 = na[k], x1 = nb[k];
        na[k] = fmaf(x0, cs[k], -x1 * sn[k]);
        nb[k] = fmaf(x1, cs[k], x0 * sn[k]);
      }
    }
  } else {
    if (ln.rot_a) rotate_interleaved<F>(na, cs, sn);
    if (ln.rot_b) rotate_interleaved<F>(nb, cs + F / 2, sn + F / 2);
  }
  xa = Frag<F>::pack(na);
  xb = Frag<F>::pack(nb);
}

// The same with the weights packed as bf16 (widened here).
template <int D, int F, bool NEOX, bool EXACT_RSQRT>
__device__ __forceinline__ void row_math(typename Frag<F>::T& xa, typename Frag<F>::T& xb,
                                         const typename Frag<F>::T& wpa,
                                         const typename Frag<F>::T& wpb, const float* cs,
                                         const float* sn, const Lane<D, F, NEOX>& ln, float eps) {
  float wa[F], wb[F];
  Frag<F>::unpack(wpa, wa);
  Frag<F>::unpack(wpb, wb);
  row_math_w<D, F, NEOX, EXACT_RSQRT>(xa, xb, wa, wb, cs, sn, ln, eps);
}

}  // namespace qkgen
}  // namespace kvq
