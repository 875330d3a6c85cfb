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
//     multiple of 8, so every store is naturally aligned; all are streaming
//     (evict-first) stores.
// No warp mixes the light Q work with the heavier KV work (the pages'
// slot-type-uniform programs).  Two kernel shapes:
//   * tiles:  one-shot grid; the first CTAs take KV vectors (one token per
//     warp), the rest QROWS consecutive q rows per warp, all loads of a warp
//     issued before any arithmetic (KV first measured faster than KV CTAs
//     spread evenly through the grid);
//   * stream: persistent grid sized to the resident-CTA capacity of the GPU;
//     every warp first takes its grid-stride share of KV vectors, then its
//     q rows in groups of G adjacent rows (groups grid-strided), with the
//     next row's loads in flight while the current row is computed and
//     stored (two register buffers).
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
  const __nv_bfloat16* q;
  __nv_bfloat16* q_out;  // equal to q when the operator runs in place
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
  int kv_ctas;  // tiles kernel: leading CTAs that do KV work
  float eps;
  // bounds-checked launches only
  int64_t max_pos;    // rows of cos_sin
  int64_t num_slots;  // cache capacity
  int* errors;        // tokens rejected
  int trigger_from;   // tiles kernel: first CTA of the last wave
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

// One row's data as held by a lane: two 16-byte chunks plus, on the rotary
// lanes, the token's four cosines and four sines; `ok` (bounds-checked
// launches) says whether the token's position lies inside the cos/sin table.
struct RowRegs {
  uint4 a, b;
  float4 c, s;
  bool ok;
};

// CHECKED: every lane reads the position, so the whole warp agrees on `ok`,
// and no cos/sin row outside the table is read.
template <bool CHECKED>
__device__ __forceinline__ void load_row(const Dsv4Params& p, const __nv_bfloat16* row,
                                         int64_t token, int lane, RowRegs& r) {
  r.a = load_stream(row + 8 * lane);
  r.b = load_stream(row + 256 + 8 * lane);
  r.ok = true;
  if (CHECKED) {
    const int64_t pos = __ldg(p.positions + token);
    r.ok = pos >= 0 && pos < p.max_pos;
    if (lane >= kRopeLane && r.ok) {
      const float4* cs = reinterpret_cast<const float4*>(p.cos_sin + pos * 64);
      r.c = __ldg(cs + (lane - kRopeLane));
      r.s = __ldg(cs + 8 + (lane - kRopeLane));
    }
  } else if (lane >= kRopeLane) {
    const int64_t pos = __ldg(p.positions + token);
    const float4* cs = reinterpret_cast<const float4*>(p.cos_sin + pos * 64);
    r.c = __ldg(cs + (lane - kRopeLane));
    r.s = __ldg(cs + 8 + (lane - kRopeLane));
  }
}

// The lane's 16 weights, kept packed as bf16 (8 registers) and widened where
// they are used.
struct Weights {
  uint4 a, b;
};

__device__ __forceinline__ Weights load_weights(const __nv_bfloat16* w, int lane) {
  return {__ldg(reinterpret_cast<const uint4*>(w) + lane),
          __ldg(reinterpret_cast<const uint4*>(w) + 32 + lane)};
}

// n = x * r * w with r from the warp-wide sum of squares, then the
// interleaved rotation of chunk 1 on the rotary lanes.
__device__ __forceinline__ void norm_rope(const RowRegs& r, const Weights& wp, float eps,
                                          int lane, float* x) {
  unpack_bf16x8(r.a, x);
  unpack_bf16x8(r.b, x + 8);
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) ss = fmaf(x[k], x[k], ss);
  ss = group_sum<32>(ss);
  const float rs = __frsqrt_rn(ss * (1.0f / kDim) + eps);
  float w[16];
  unpack_bf16x8(wp.a, w);
  unpack_bf16x8(wp.b, w + 8);
#pragma unroll
  for (int k = 0; k < 16; ++k) x[k] = x[k] * rs * w[k];
  if (lane >= kRopeLane) {
    const float cc[4] = {r.c.x, r.c.y, r.c.z, r.c.w};
    const float sn[4] = {r.s.x, r.s.y, r.s.z, r.s.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float e = x[8 + 2 * j], o = x[9 + 2 * j];
      x[8 + 2 * j] = fmaf(e, cc[j], -o * sn[j]);
      x[9 + 2 * j] = fmaf(o, cc[j], e * sn[j]);
    }
  }
}

// A row whose token has no valid position (checked launches) is left as is.
template <bool CHECKED>
__device__ __forceinline__ void q_row(const Dsv4Params& p, int row, const RowRegs& r,
                                      const Weights& w, int lane) {
  if (CHECKED && !r.ok) return;  // warp-uniform
  float x[16];
  norm_rope(r, w, p.eps, lane, x);
  __nv_bfloat16* dst = p.q_out + (size_t)row * kDim;
  store_stream(dst + 8 * lane, pack_bf16x8(x));
  store_stream(dst + 256 + 8 * lane, pack_bf16x8(x + 8));
}

// Entry stores are streaming (evict-first), like the q stores.  Measured on
// GB300: with default write-back stores the entries of a large batch linger
// in L2 and cost the q stream up to 10% when the cache exceeds L2 (153 MB
// cache, 131072 tokens); evict-first stores bring the kernel within 2% of
// the same launch without any cache write.
__device__ __forceinline__ void store8(uint8_t* dst, uint2 v) {
  __stcs(reinterpret_cast<uint2*>(dst), v);
}

// Checked launches reject a token whose position is outside the table or
// whose slot is neither -1 nor inside the cache: no entry is written and the
// token is counted once (its q rows are skipped only for a bad position).
template <bool CHECKED>
__device__ __forceinline__ void kv_token(const Dsv4Params& p, int64_t slot, const RowRegs& r,
                                         const Weights& w, int lane) {
  if (CHECKED && (!r.ok || slot < -1 || slot >= p.num_slots)) {  // warp-uniform
    if (lane == 0) atomicAdd(p.errors, 1);
    return;
  }
  float x[16];
  norm_rope(r, w, p.eps, lane, x);
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
  if (slot < 0) return;  // warp-uniform: the token has no cache slot
  uint8_t* ent = p.kv_cache + slot * kEntry;
  store8(ent + 8 * lane, codes0);
  if (lane < kRopeLane) {
    store8(ent + 256 + 8 * lane, codes1);
  } else {
    uint8_t* dst = ent + kRopeAt + 16 * (lane - kRopeLane);
    store8(dst, make_uint2(rope.x, rope.y));
    store8(dst + 8, make_uint2(rope.z, rope.w));
  }
  if (lane == 0) {
    store8(ent + kScaleAt, make_uint2(g0 | (g1 << 8) | (g2 << 16) | (g3 << 24),
                                                   g4 | (g5 << 8) | (g6 << 16)));
  }
}

// ---- tiles: one-shot grid -------------------------------------------------

template <int WARPS, int QROWS, int MINB, bool CHECKED>
__global__ void __launch_bounds__(WARPS * 32, MINB)
dsv4_tiles_kernel(const Dsv4Params p) {
  grid_dependency_sync(p.trigger_from);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if ((int)blockIdx.x < p.kv_ctas) {
    const int t = (int)blockIdx.x * WARPS + warp;
    if (t >= p.num_tokens) return;
    RowRegs r;
    load_row<CHECKED>(p, p.kv + (size_t)t * kDim, t, lane, r);
    const int64_t slot = __ldg(p.slot_mapping + t);
    kv_token<CHECKED>(p, slot, r, load_weights(p.kv_weight, lane), lane);
    return;
  }
  const int row0 = (((int)blockIdx.x - p.kv_ctas) * WARPS + warp) * QROWS;
  RowRegs r[QROWS];
#pragma unroll
  for (int i = 0; i < QROWS; ++i)
    if (row0 + i < p.q_rows)
      load_row<CHECKED>(p, p.q + (size_t)(row0 + i) * kDim, (row0 + i) / p.num_heads, lane,
                        r[i]);
  const Weights w = load_weights(p.q_weight, lane);
#pragma unroll
  for (int i = 0; i < QROWS; ++i) {
    if (row0 + i >= p.q_rows) break;  // warp-uniform
    q_row<CHECKED>(p, row0 + i, r[i], w, lane);
  }
}

// ---- stream: persistent grid, two-deep register pipeline ------------------

template <bool CHECKED>
__device__ __forceinline__ void stream_kv(const Dsv4Params& p, int gw, int nw, int lane) {
  if (gw >= p.num_tokens) return;
  const Weights w = load_weights(p.kv_weight, lane);
  for (int t = gw; t < p.num_tokens; t += nw) {
    RowRegs r;
    load_row<CHECKED>(p, p.kv + (size_t)t * kDim, t, lane, r);
    kv_token<CHECKED>(p, __ldg(p.slot_mapping + t), r, w, lane);
  }
}

// The warp's q rows, two-deep: the next row's loads are in flight while the
// current row is computed and stored (two register buffers, compile-time
// indices).  Rows come in groups of G adjacent rows, group g of warp gw being
// rows (gw + g nw) G .. + G - 1, and the pipeline runs along that sequence:
// with G = 2 the row in flight is, every other time, the one right after the
// row being computed, and the grid as a whole reads one contiguous window of
// 2 nw rows.  Measured on GB300 against the plain grid-stride order (rows gw,
// gw + nw, ..., whose rows in flight lie nw rows apart): 2.5-5 % faster at
// every size from 2048 tokens on (99-102 % of the measured copy peak against
// 96-97 %); groups of 4 or 8 rows, and deeper pipelines (three or four
// buffers, hence fewer warps per SM), were slower.  The loop is kept in this
// form: an equivalent rewrite of the same row sequence (one loop over
// "sequence positions") compiled to a kernel that ran 2.7 % slower.
template <bool CHECKED, int G>
__device__ __forceinline__ void stream_q(const Dsv4Params& p, int gw, int nw, int lane) {
  constexpr int kDepth = 2;
  static_assert(G % kDepth == 0, "whole pipeline rounds per group");
  // Row numbers are unsigned 32-bit: q_rows < 2^31, and a row index computed
  // one group ahead stays below 2^31 + G nw.
  const uint32_t q_rows = (uint32_t)p.q_rows;
  const uint32_t step = (uint32_t)nw * G;
  uint32_t base = (uint32_t)gw * G;  // first row of the current group
  if (base >= q_rows) return;
  const Weights w = load_weights(p.q_weight, lane);
  RowRegs r[kDepth];
#pragma unroll
  for (int i = 0; i < kDepth - 1; ++i) {
    const uint32_t row = base + i;
    if (row < q_rows) load_row<CHECKED>(p, p.q + (size_t)row * kDim, row / p.num_heads, lane, r[i]);
  }
  for (;; base += step) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const uint32_t row = base + j;
      if (row >= q_rows) return;  // warp-uniform
      const uint32_t ahead =
          j + kDepth - 1 < G ? row + kDepth - 1 : base + step + j + kDepth - 1 - G;
      if (ahead < q_rows)
        load_row<CHECKED>(p, p.q + (size_t)ahead * kDim, ahead / p.num_heads, lane,
                          r[(j + kDepth - 1) % kDepth]);
      q_row<CHECKED>(p, (int)row, r[j % kDepth], w, lane);
    }
  }
}

// KV vectors first: each warp's share is small, and running them last was
// measured no faster.
template <int WARPS, int MINB, bool CHECKED, int G>
__global__ void __launch_bounds__(WARPS * 32, MINB)
dsv4_stream_kernel(const Dsv4Params p) {
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const int gw = (int)blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = (int)gridDim.x * WARPS;
  stream_kv<CHECKED>(p, gw, nw, lane);
  stream_q<CHECKED, G>(p, gw, nw, lane);
}

Dsv4Params make_params(const Dsv4Args& a) {
  Dsv4Params p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.q_out = static_cast<__nv_bfloat16*>(a.q_out);
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
  p.kv_ctas = 0;
  p.eps = a.eps;
  p.max_pos = a.max_pos;
  p.num_slots = a.num_slots;
  p.errors = a.errors;
  p.trigger_from = 0;
  return p;
}

template <int WARPS, int QROWS, int MINB, bool CHECKED = false>
cudaError_t launch_tiles(const Dsv4Args& a, cudaStream_t stream) {
  Dsv4Params p = make_params(a);
  p.kv_ctas = (p.num_tokens + WARPS - 1) / WARPS;
  const int q_ctas = (p.q_rows + WARPS * QROWS - 1) / (WARPS * QROWS);
  static std::atomic<int> cache[kMaxDevices];
  p.trigger_from = last_wave_start(dsv4_tiles_kernel<WARPS, QROWS, MINB, CHECKED>, WARPS * 32,
                                   p.kv_ctas + q_ctas, cache);
  return launch_kernel(dsv4_tiles_kernel<WARPS, QROWS, MINB, CHECKED>,
                       dim3((unsigned)(p.kv_ctas + q_ctas)), dim3(WARPS * 32), 0, stream, p);
}

template <int WARPS, int MINB, bool CHECKED, int G>
cudaError_t launch_stream(const Dsv4Args& a, cudaStream_t stream) {
  Dsv4Params p = make_params(a);
  int per_sm = 0;
  static std::atomic<int> cache[kMaxDevices];
  cudaError_t e =
      resident_ctas(dsv4_stream_kernel<WARPS, MINB, CHECKED, G>, WARPS * 32, cache, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t work_warps = p.q_rows > p.num_tokens ? p.q_rows : p.num_tokens;
  int64_t grid = (int64_t)per_sm * device_sm_count();
  const int64_t need = (work_warps + WARPS - 1) / WARPS;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  return launch_kernel(dsv4_stream_kernel<WARPS, MINB, CHECKED, G>, dim3((unsigned)grid),
                       dim3(WARPS * 32), 0, stream, p);
}

}  // namespace

const LaunchConfig kDsv4Configs[] = {
    {"tiles<4w,1row>"}, {"tiles<8w,1row>"}, {"tiles<8w,2row>"},
    {"tiles<8w,4row>"}, {"stream<8w,85reg,pairs>"},
};
const int kDsv4NumConfigs = sizeof(kDsv4Configs) / sizeof(kDsv4Configs[0]);

cudaError_t launch_dsv4(const Dsv4Args& a, int config, cudaStream_t stream) {
  if (a.errors != nullptr) {  // bounds-checked: the two dispatch shapes
    return config == 4 ? launch_stream<8, 3, true, 2>(a, stream)
                       : launch_tiles<4, 1, 1, true>(a, stream);
  }
  switch (config) {
    case 0: return launch_tiles<4, 1, 1>(a, stream);
    case 1: return launch_tiles<8, 1, 1>(a, stream);
    case 2: return launch_tiles<8, 2, 4>(a, stream);
    case 3: return launch_tiles<8, 4, 1>(a, stream);
    case 4: return launch_stream<8, 3, false, 2>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
