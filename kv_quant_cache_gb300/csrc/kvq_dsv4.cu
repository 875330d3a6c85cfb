// kvq_dsv4.cu -- DeepSeek-V4-style Q norm + RoPE and KV norm + RoPE +
// UE8M0/e4m3 block quantisation + paged-cache insert, one launch.
//
// Operator: FlagGems PR #5449 ("[KMCompiler][Hygon] Token-tiled
// fused_deepseek_v4_qnorm_rope_kv_rope_quant_insert", section "Performance":
// slot_mapping/kv_cache inputs, seven per-block exponents per token) and
// FlagGems PR #5321 ("... plus test and benchmark fixes", section "What the
// optimisation does": H query-head slots and one KV slot per token, the KV
// slot doing seven quantisation blocks).  Slot split and cache entry as
// defined in include/kvq.h.
//
// Mapping on sm_103a.  A 512-dim bf16 row (1 KiB) is one warp: lane l holds
// dims [8l, 8l+8) ("chunk 0") and [256+8l, 256+8l+8) ("chunk 1"), each one
// coalesced 16-byte access, so a warp-wide access covers 512 contiguous bytes.
//   * RMSNorm: per-lane sum of 16 squares, 5-step butterfly.
//   * RoPE: dims 448..511 are chunk 1 of lanes 24..31; the interleaved pairs
//     (448+2i, 449+2i) sit inside one lane, so no shuffle is needed.  Those 8
//     lanes read 32 cosines/sines of the token's row (two 16-byte loads each).
//   * Quantisation block b (dims 64b..64b+63) is chunk 0 of lanes 8b..8b+7
//     for b < 4 and chunk 1 of lanes 8(b-4).. for b = 4..6, so each block
//     amax is a 3-step butterfly inside an aligned group of 8 lanes.
//   * Cache entry: chunk-0 codes are 32 x 8 contiguous bytes, chunk-1 codes
//     and the rotary bf16 values the next 320 bytes, and lane 0 writes the
//     seven exponent bytes plus the pad as one 8-byte store.  slot * 584 is a
//     multiple of 8, so every store is naturally aligned.
// CTAs are slot-type uniform: the first kv_ctas CTAs each take WARPS*KVROWS
// tokens' KV vectors, the rest take WARPS*QROWS consecutive q head rows, so
// no warp mixes the light Q work with the heavier KV work.  Within a warp all
// row loads are issued before any arithmetic.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kDim = 512;
constexpr int kEntry = 584;
constexpr int kRopeAt = 448;   // entry offset of the rotary bf16 values
constexpr int kScaleAt = 576;  // entry offset of the exponent bytes
constexpr int kRopeLane = 24;  // first lane whose chunk 1 is rotary

struct Dsv4Params {
  __nv_bfloat16* q;
  const __nv_bfloat16* kv;
  const __nv_bfloat16* q_weight;
  const __nv_bfloat16* kv_weight;
  const float* cos_sin;
  const int64_t* positions;
  const int64_t* slot_mapping;
  uint8_t* kv_cache;
  int num_tokens;
  int num_heads;
  int q_rows;   // num_tokens * num_heads
  int kv_ctas;  // leading CTAs that do KV work
  float eps;
};

// UE8M0 exponent byte (e + 127, clamped to [0, 254]) of the smallest power of
// two 2^e with 448 * 2^e >= amax, from amax's binary32 fields: amax =
// (1 + m) 2^E and 448 = 1.75 * 2^8, so e = E - 8 when 1 + m <= 1.75 and
// E - 7 otherwise; 1.75 is the mantissa field 0x600000.  Zero and subnormal
// amax clamp to byte 0.
__device__ __forceinline__ int ue8m0_byte(float amax) {
  const uint32_t u = __float_as_uint(amax);
  const int b = (int)(u >> 23) - 8 + ((u & 0x7fffffu) > 0x600000u ? 1 : 0);
  return min(max(b, 0), 254);
}

// 2^-(byte - 127) as a binary32 (always a normal number for byte <= 253).
__device__ __forceinline__ float ue8m0_inverse_scale(int byte) {
  return __uint_as_float((uint32_t)(254 - byte) << 23);
}

// Eight fp32 values times a power of two -> eight e4m3fn codes (RNE,
// saturating), element 0 in the lowest byte.
__device__ __forceinline__ uint2 e4m3x8(const float* v, float scale) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    w[k] = __nv_cvt_float2_to_fp8x2(make_float2(v[2 * k] * scale, v[2 * k + 1] * scale),
                                    __NV_SATFINITE, __NV_E4M3);
  }
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// Load a row's two 16-byte chunks for this lane.
__device__ __forceinline__ void load_row(const __nv_bfloat16* row, int lane, uint4& a, uint4& b) {
  a = load_stream(row + 8 * lane);
  b = load_stream(row + 256 + 8 * lane);
}

// Normalise a row held as 16 fp32 per lane: n = x * r * w, r from the
// warp-wide sum of squares.
__device__ __forceinline__ void rms_norm_row(float* x, const float* w, float eps) {
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) ss = fmaf(x[k], x[k], ss);
  ss = group_sum<32>(ss);
  const float r = __frsqrt_rn(ss * (1.0f / kDim) + eps);
#pragma unroll
  for (int k = 0; k < 16; ++k) x[k] = x[k] * r * w[k];
}

// Interleaved rotation of chunk 1 (x[8..15]) for the rotary lanes.
__device__ __forceinline__ void rope_chunk1(float* x, const float4& c, const float4& s) {
  const float cc[4] = {c.x, c.y, c.z, c.w};
  const float ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float e = x[8 + 2 * j], o = x[9 + 2 * j];
    x[8 + 2 * j] = fmaf(e, cc[j], -o * ss[j]);
    x[9 + 2 * j] = fmaf(o, cc[j], e * ss[j]);
  }
}

__device__ __forceinline__ void load_cos_sin(const Dsv4Params& p, int64_t token, int lane,
                                             float4& c, float4& s) {
  const int64_t pos = __ldg(p.positions + token);
  const float4* row = reinterpret_cast<const float4*>(p.cos_sin + pos * 64);
  c = __ldg(row + (lane - kRopeLane));
  s = __ldg(row + 8 + (lane - kRopeLane));
}

template <int R>
__device__ __forceinline__ void q_rows(const Dsv4Params& p, int row0, int lane) {
  uint4 a[R], b[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    a[i] = b[i] = make_uint4(0u, 0u, 0u, 0u);
    if (row0 + i < p.q_rows) load_row(p.q + (size_t)(row0 + i) * kDim, lane, a[i], b[i]);
  }
  float w[16];
  unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.q_weight) + lane), w);
  unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.q_weight) + 32 + lane), w + 8);
  float4 c[R], s[R];
  if (lane >= kRopeLane) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      c[i] = s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row0 + i < p.q_rows) load_cos_sin(p, (row0 + i) / p.num_heads, lane, c[i], s[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < R; ++i) {
    if (row0 + i >= p.q_rows) break;  // warp-uniform
    float x[16];
    unpack_bf16x8(a[i], x);
    unpack_bf16x8(b[i], x + 8);
    rms_norm_row(x, w, p.eps);
    if (lane >= kRopeLane) rope_chunk1(x, c[i], s[i]);
    __nv_bfloat16* row = p.q + (size_t)(row0 + i) * kDim;
    store_stream(row + 8 * lane, pack_bf16x8(x));
    store_stream(row + 256 + 8 * lane, pack_bf16x8(x + 8));
  }
}

template <int R>
__device__ __forceinline__ void kv_rows(const Dsv4Params& p, int t0, int lane) {
  uint4 a[R], b[R];
  int64_t slot[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    a[i] = b[i] = make_uint4(0u, 0u, 0u, 0u);
    slot[i] = -1;
    if (t0 + i < p.num_tokens) {
      load_row(p.kv + (size_t)(t0 + i) * kDim, lane, a[i], b[i]);
      slot[i] = __ldg(p.slot_mapping + t0 + i);
    }
  }
  float w[16];
  unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.kv_weight) + lane), w);
  unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.kv_weight) + 32 + lane), w + 8);
  float4 c[R], s[R];
  if (lane >= kRopeLane) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      c[i] = s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t0 + i < p.num_tokens) load_cos_sin(p, t0 + i, lane, c[i], s[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < R; ++i) {
    if (t0 + i >= p.num_tokens) break;  // warp-uniform
    float x[16];
    unpack_bf16x8(a[i], x);
    unpack_bf16x8(b[i], x + 8);
    rms_norm_row(x, w, p.eps);
    const bool rope_lane = lane >= kRopeLane;
    if (rope_lane) rope_chunk1(x, c[i], s[i]);

    // Block amax: chunk 0 -> blocks 0..3, chunk 1 -> blocks 4..6 (lanes < 24).
    float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      m0 = fmaxf(m0, fabsf(x[k]));
      m1 = fmaxf(m1, fabsf(x[8 + k]));
    }
    m0 = group_max<8>(m0);
    m1 = group_max<8>(m1);
    const int e0 = ue8m0_byte(m0);
    const int e1 = ue8m0_byte(m1);
    const uint2 codes0 = e4m3x8(x, ue8m0_inverse_scale(e0));
    const uint2 codes1 = e4m3x8(x + 8, ue8m0_inverse_scale(e1));
    const uint4 rope = pack_bf16x8(x + 8);
    // Exponent bytes of blocks 0..6 gathered to lane 0.
    const uint32_t g0 = __shfl_sync(kFullMask, e0, 0), g1 = __shfl_sync(kFullMask, e0, 8);
    const uint32_t g2 = __shfl_sync(kFullMask, e0, 16), g3 = __shfl_sync(kFullMask, e0, 24);
    const uint32_t g4 = __shfl_sync(kFullMask, e1, 0), g5 = __shfl_sync(kFullMask, e1, 8);
    const uint32_t g6 = __shfl_sync(kFullMask, e1, 16);

    if (slot[i] < 0) continue;  // warp-uniform: no cache slot for this token
    uint8_t* ent = p.kv_cache + slot[i] * kEntry;
    *reinterpret_cast<uint2*>(ent + 8 * lane) = codes0;
    if (!rope_lane) {
      *reinterpret_cast<uint2*>(ent + 256 + 8 * lane) = codes1;
    } else {
      uint2* dst = reinterpret_cast<uint2*>(ent + kRopeAt + 16 * (lane - kRopeLane));
      dst[0] = make_uint2(rope.x, rope.y);
      dst[1] = make_uint2(rope.z, rope.w);
    }
    if (lane == 0) {
      *reinterpret_cast<uint2*>(ent + kScaleAt) =
          make_uint2(g0 | (g1 << 8) | (g2 << 16) | (g3 << 24), g4 | (g5 << 8) | (g6 << 16));
    }
  }
}

template <int WARPS, int QROWS, int KVROWS>
__global__ void __launch_bounds__(WARPS * 32)
dsv4_kernel(const Dsv4Params p) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if ((int)blockIdx.x < p.kv_ctas) {
    kv_rows<KVROWS>(p, ((int)blockIdx.x * WARPS + warp) * KVROWS, lane);
  } else {
    q_rows<QROWS>(p, (((int)blockIdx.x - p.kv_ctas) * WARPS + warp) * QROWS, lane);
  }
}

template <int WARPS, int QROWS, int KVROWS>
cudaError_t launch(const Dsv4Args& a, cudaStream_t stream) {
  Dsv4Params p;
  p.q = static_cast<__nv_bfloat16*>(a.q);
  p.kv = static_cast<const __nv_bfloat16*>(a.kv);
  p.q_weight = static_cast<const __nv_bfloat16*>(a.q_weight);
  p.kv_weight = static_cast<const __nv_bfloat16*>(a.kv_weight);
  p.cos_sin = a.cos_sin;
  p.positions = a.positions;
  p.slot_mapping = a.slot_mapping;
  p.kv_cache = a.kv_cache;
  p.num_tokens = a.num_tokens;
  p.num_heads = a.num_heads;
  p.q_rows = a.num_tokens * a.num_heads;
  p.eps = a.eps;
  p.kv_ctas = (a.num_tokens + WARPS * KVROWS - 1) / (WARPS * KVROWS);
  const int q_ctas = (p.q_rows + WARPS * QROWS - 1) / (WARPS * QROWS);
  dsv4_kernel<WARPS, QROWS, KVROWS><<<p.kv_ctas + q_ctas, WARPS * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dsv4(const Dsv4Args& a, int path, cudaStream_t stream) {
  if (path == 0) return launch<4, 1, 1>(a, stream);
  return launch<8, 4, 1>(a, stream);
}

}  // namespace kvq
