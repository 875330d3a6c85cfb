// kvq_qk_row.cuh -- the per-row arithmetic of the head_dim-128 full-NeoX QK
// operator (InfiniOps PR #1019, "Add the NineToothed NVIDIA implementation of
// FusedQkNormRope", section "Summary": per-head RMSNorm, then NeoX RoPE, each
// element of a pair weighted with its own dimension's weight).  Shared by the
// register-pipelined kernels (kvq_qk_norm_rope.cu) and the TMA-staged kernel
// (kvq_qk_bulk.cu), so every launch shape gives bit-identical results.
//
// Lane mapping: a half-warp holds one 128-dim row; lane l (of 16) holds dims
// [4l, 4l+4) ("lo") and their NeoX partners [64+4l, 64+4l+4) ("hi").
#pragma once

#include "kvq_device.cuh"

namespace kvq {
namespace qk128 {

constexpr int kHeadDim = 128;
constexpr int kHalf = kHeadDim / 2;

// Weight fragments of one lane (lo and hi dims, Q and K), kept packed as
// bf16 and widened where they are used.
struct Weights {
  uint2 q_lo, q_hi, k_lo, k_hi;
};

__device__ __forceinline__ void load_weights(const __nv_bfloat16* q_weight,
                                             const __nv_bfloat16* k_weight, int l16,
                                             Weights& w) {
  const uint2* q = reinterpret_cast<const uint2*>(q_weight);
  const uint2* k = reinterpret_cast<const uint2*>(k_weight);
  w.q_lo = __ldg(q + l16);
  w.q_hi = __ldg(q + 16 + l16);
  w.k_lo = __ldg(k + l16);
  w.k_hi = __ldg(k + 16 + l16);
}

__device__ __forceinline__ void unpack_bf16x4(const uint2& v, float* f) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xffff0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xffff0000u);
}

// Normalise + rotate one row fragment in place; all 32 lanes must call it
// together (the sum of squares is reduced across each half-warp).  c4 / s4
// are the cosines / sines of frequencies 4l .. 4l+3.
__device__ __forceinline__ void row_math(uint2& lo, uint2& hi, bool is_q, const Weights& w,
                                         const float4& c4, const float4& s4, float eps) {
  float a[4], b[4];
  unpack_bf16x4(lo, a);
  unpack_bf16x4(hi, b);
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) ss = fmaf(b[k], b[k], fmaf(a[k], a[k], ss));
  ss = group_sum<16>(ss);
  const float r = __frsqrt_rn(ss * (1.0f / kHeadDim) + eps);
  float wa[4], wb[4];
  unpack_bf16x4(is_q ? w.q_lo : w.k_lo, wa);
  unpack_bf16x4(is_q ? w.q_hi : w.k_hi, wb);
  const float c[4] = {c4.x, c4.y, c4.z, c4.w};
  const float s[4] = {s4.x, s4.y, s4.z, s4.w};
  float oa[4], ob[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float na = a[k] * r * wa[k];
    const float nb = b[k] * r * wb[k];
    oa[k] = fmaf(na, c[k], -nb * s[k]);
    ob[k] = fmaf(nb, c[k], na * s[k]);
  }
  lo = make_uint2(pack_bf16x2(oa[0], oa[1]), pack_bf16x2(oa[2], oa[3]));
  hi = make_uint2(pack_bf16x2(ob[0], ob[1]), pack_bf16x2(ob[2], ob[3]));
}

}  // namespace qk128
}  // namespace kvq
