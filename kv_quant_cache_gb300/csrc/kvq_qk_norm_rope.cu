// kvq_qk_norm_rope.cu -- packed-QKV per-head RMSNorm + NeoX RoPE, in place.
//
// Operator: InfiniOps PR #1019 ("Add the NineToothed NVIDIA implementation of
// FusedQkNormRope"), section "Summary": Q and K heads of a packed
// [T, (Hq+Hk+Hv)*D] bf16 tensor get per-head RMSNorm followed by NeoX RoPE in
// place, V untouched, separate [D] weights, and the NeoX partner read with
// its own dimension's weight.  This build covers the guarded case of "Notes
// for Reviewers": bf16, D = 128, full-dimension NeoX rotation.
//
// Mapping on sm_103a.  A 128-dim bf16 head row is 256 bytes = 16 lanes x one
// 16-byte vector, so one warp covers two head rows per step: lanes 0-15 row
// h, lanes 16-31 row h+1.  Lane l (of 16) holds dims 8l..8l+7; the NeoX
// partner dims i +- 64 sit in lane l ^ 8 of the same half-warp, so one
// 4-word shuffle of the raw bf16 values brings the partner in, and the
// partner is then weighted with its own weight fragment.  The sum of squares
// is a 4-step butterfly inside the half-warp.  A warp task is (token, chunk of
// 2*STEPS consecutive Q/K head rows): the token's position and its 512-byte
// cos/sin row are fetched once per task and reused for every row, and all
// STEPS row loads are issued before any arithmetic so that each warp keeps
// STEPS x 512 bytes in flight.  V columns are never addressed.
#include "kvq_device.cuh"
#include "kvq_launch.h"

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
  int chunks;         // tasks per token
  float eps;
};

template <int WARPS, int STEPS>
__global__ void __launch_bounds__(WARPS * 32)
qk_norm_rope_kernel(const QkParams p) {
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int l16 = lane & 15;
  const int task = blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (task >= p.num_tokens * p.chunks) return;  // whole warp leaves together
  const int t = task / p.chunks;
  const int first = (task - t * p.chunks) * (2 * STEPS) + half;

  __nv_bfloat16* tok = p.qkv + (size_t)t * (size_t)p.row_elems;

  // 1. Issue every row load of this task first.
  uint4 x[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int h = first + 2 * s;
    x[s] = make_uint4(0u, 0u, 0u, 0u);
    if (h < p.num_rows) x[s] = load_stream(tok + (size_t)h * kHeadDim + 8 * l16);
  }

  // 2. Token position, its cos/sin for this lane's 8 frequencies, weights.
  const int64_t pos = __ldg(p.positions + t);
  const int f0 = 8 * (l16 & 7);  // frequency index of the lane's first dim
  const float4* crow = reinterpret_cast<const float4*>(p.cos_sin + pos * kHeadDim + f0);
  float c[8], sn[8];
  {
    const float4 c0 = __ldg(crow), c1 = __ldg(crow + 1);
    const float4 s0 = __ldg(crow + kHalf / 4), s1 = __ldg(crow + kHalf / 4 + 1);
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
    c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
    sn[0] = s0.x; sn[1] = s0.y; sn[2] = s0.z; sn[3] = s0.w;
    sn[4] = s1.x; sn[5] = s1.y; sn[6] = s1.z; sn[7] = s1.w;
  }
  // out = n*cos - n_partner*sin for dims < 64, n*cos + n_partner*sin above.
  const float sgn = (l16 < 8) ? -1.0f : 1.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) sn[k] *= sgn;

  float wq[8], wqp[8], wk[8], wkp[8];
  unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.q_weight) + l16), wq);
  unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.q_weight) + (l16 ^ 8)), wqp);
  unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.k_weight) + l16), wk);
  unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.k_weight) + (l16 ^ 8)), wkp);

  // 3. Normalise, rotate, store -- row by row.
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int h = first + 2 * s;
    uint4 y;  // partner lane's raw values (dims +- 64)
    y.x = __shfl_xor_sync(kFullMask, x[s].x, 8);
    y.y = __shfl_xor_sync(kFullMask, x[s].y, 8);
    y.z = __shfl_xor_sync(kFullMask, x[s].z, 8);
    y.w = __shfl_xor_sync(kFullMask, x[s].w, 8);
    float xf[8], yf[8];
    unpack_bf16x8(x[s], xf);
    unpack_bf16x8(y, yf);
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) ss = fmaf(xf[k], xf[k], ss);
    ss = group_sum<16>(ss);
    const float r = __frsqrt_rn(ss * (1.0f / kHeadDim) + p.eps);
    const bool is_q = h < p.num_q;
    float o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float n = xf[k] * r * (is_q ? wq[k] : wk[k]);
      const float np = yf[k] * r * (is_q ? wqp[k] : wkp[k]);
      o[k] = fmaf(n, c[k], np * sn[k]);
    }
    if (h < p.num_rows) store_stream(tok + (size_t)h * kHeadDim + 8 * l16, pack_bf16x8(o));
  }
}

template <int WARPS, int STEPS>
cudaError_t launch(const QkArgs& a, cudaStream_t stream) {
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
  p.chunks = (p.num_rows + 2 * STEPS - 1) / (2 * STEPS);
  p.eps = a.eps;
  const int64_t tasks = (int64_t)p.num_tokens * p.chunks;
  const unsigned grid = (unsigned)((tasks + WARPS - 1) / WARPS);
  qk_norm_rope_kernel<WARPS, STEPS><<<grid, WARPS * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

// Rows (Q+K heads x tokens) below which the one-row-pair-per-warp launch is
// used: it spreads a decode-sized batch over the most SMs.
constexpr int64_t kQkSmallRows = 152 * 4 * 2;

int qk_path(int64_t num_tokens, int num_rows_per_token) {
  return num_tokens * (int64_t)num_rows_per_token < kQkSmallRows ? 0 : 1;
}

cudaError_t launch_qk_norm_rope(const QkArgs& a, int path, cudaStream_t stream) {
  if (path == 0) return launch<4, 1>(a, stream);
  return launch<8, 4>(a, stream);
}

}  // namespace kvq
