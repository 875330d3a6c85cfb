// kvq_dsv4_gather.cu -- read DSV4 cache entries back as bf16 rows: the
// consumer side of dsv4_qnorm_rope_kv_rope_quant_insert.
//
// The blockwise UE8M0 layout (FlagGems PR #5449, "[KMCompiler][Hygon]
// Token-tiled fused_deepseek_v4_qnorm_rope_kv_rope_quant_insert", section
// "Performance": seven per-block exponents per token) exists to be read back
// by attention.  Row i of the output is the entry at slots[i]:
//   dims 64b + k (b < 7):  bf16(e4m3(code) * 2^(byte_b - 127)), one rounding
//   dims 448..511:         the stored bf16 rotary values
//   slots[i] < 0:          a row of +0.
//
// Mapping on sm_103a: a warp takes kRows consecutive rows.  Lanes 0..kRows-1
// load the rows' slots with one coalesced access; then, for every row, lane
// l reads the entry the way the insert kernel wrote it -- 8 code bytes of
// chunk 0 (dims 8l..8l+7), 8 of chunk 1 or, on lanes 24..31, 16 bytes of
// rotary bf16 -- plus the entry's 8-byte exponent word (one broadcast load).
// All entry loads of the warp's rows are in flight before any is used: a
// row costs two dependent memory latencies (slot, then entry), which one row
// per warp could not hide.  e4m3 -> f16 is exact in hardware; the f16 value
// times the power of two is exact in fp32; the result is rounded once to
// bf16.  Entries are 8-byte aligned, so every entry access is an 8-byte
// load; every output row is two 16-byte stores per lane.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kDim = 512;
constexpr int kEntry = 584;
constexpr int kRopeAt = 448;
constexpr int kScaleAt = 576;
constexpr int kRopeLane = 24;
constexpr int kWarps = 8;
constexpr int kRows = 4;  // rows per warp, all loads in flight together

struct GatherParams {
  const uint8_t* kv_cache;
  const int64_t* slots;
  __nv_bfloat16* out;
  int num_rows;
  int64_t num_slots;  // bounds-checked launches: cache capacity
  int* errors;        // bounds-checked launches: rows rejected
  int trigger_from;   // first CTA of the last wave
};

// 2^(byte - 127) as a binary32 (byte 0 gives the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_scale(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// Eight e4m3 codes (element 0 in the lowest byte) times a power of two ->
// eight bf16, packed.
__device__ __forceinline__ uint4 dequant8(const uint2 codes, float scale) {
  const uint32_t w[2] = {codes.x, codes.y};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)(w[k >> 1] >> (16 * (k & 1)));
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    o[k] = pack_bf16x2(f.x * scale, f.y * scale);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One row's entry as held by a lane.
struct EntryRegs {
  uint2 scales, c0, c1, r0;
};

// Checked launches turn a slot that is neither -1 nor inside the cache into a
// zero row and count it.
template <bool CHECKED>
__global__ void __launch_bounds__(kWarps * 32)
dsv4_gather_kernel(const GatherParams p) {
  grid_dependency_sync(p.trigger_from);
  const int lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRows;
  if (row0 >= p.num_rows) return;  // whole warp leaves together
  const int64_t my_slot = lane < kRows && row0 + lane < p.num_rows ? __ldg(p.slots + row0 + lane)
                                                                  : -1;
  int64_t slot[kRows];
  EntryRegs e[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    slot[r] = __shfl_sync(kFullMask, my_slot, r);
    const bool bad = CHECKED && (slot[r] < -1 || slot[r] >= p.num_slots);
    if (bad) {
      if (lane == 0 && row0 + r < p.num_rows) atomicAdd(p.errors, 1);
      slot[r] = -1;
    }
    if (slot[r] < 0) continue;  // warp-uniform
    const uint8_t* ent = p.kv_cache + slot[r] * kEntry;
    e[r].scales = __ldg(reinterpret_cast<const uint2*>(ent + kScaleAt));
    e[r].c0 = __ldg(reinterpret_cast<const uint2*>(ent + 8 * lane));
    if (lane < kRopeLane) {
      e[r].c1 = __ldg(reinterpret_cast<const uint2*>(ent + 256 + 8 * lane));
    } else {
      const uint2* rp = reinterpret_cast<const uint2*>(ent + kRopeAt + 16 * (lane - kRopeLane));
      e[r].c1 = __ldg(rp);
      e[r].r0 = __ldg(rp + 1);
    }
  }
  const uint32_t b0 = lane >> 3;        // block of chunk 0: 0..3
  const uint32_t b1 = 4 + (lane >> 3);  // block of chunk 1: 4..6 (lanes < 24)
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    if (row0 + r >= p.num_rows) break;  // warp-uniform
    __nv_bfloat16* dst = p.out + (size_t)(row0 + r) * kDim;
    if (slot[r] < 0) {
      store_stream(dst + 8 * lane, make_uint4(0u, 0u, 0u, 0u));
      store_stream(dst + 256 + 8 * lane, make_uint4(0u, 0u, 0u, 0u));
      continue;
    }
    const uint2 sc = e[r].scales;
    const uint32_t e0 = (sc.x >> (8 * b0)) & 0xffu;
    const uint32_t e1 = (b1 < 4 ? sc.x >> (8 * b1) : sc.y >> (8 * (b1 - 4))) & 0xffu;
    store_stream(dst + 8 * lane, dequant8(e[r].c0, ue8m0_scale(e0)));
    if (lane < kRopeLane) {
      store_stream(dst + 256 + 8 * lane, dequant8(e[r].c1, ue8m0_scale(e1)));
    } else {  // the rotary dims are stored as bf16 already
      store_stream(dst + 256 + 8 * lane, make_uint4(e[r].c1.x, e[r].c1.y, e[r].r0.x, e[r].r0.y));
    }
  }
}

}  // namespace

cudaError_t launch_dsv4_gather(const GatherArgs& a, cudaStream_t stream) {
  GatherParams p;
  p.kv_cache = a.kv_cache;
  p.slots = a.slots;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.num_rows = a.num_rows;
  p.num_slots = a.num_slots;
  p.errors = a.errors;
  const unsigned grid = (unsigned)((p.num_rows + kWarps * kRows - 1) / (kWarps * kRows));
  static std::atomic<int> cache[2][kMaxDevices];
  const bool checked = a.errors != nullptr;
  const auto kernel = checked ? dsv4_gather_kernel<true> : dsv4_gather_kernel<false>;
  p.trigger_from = last_wave_start(kernel, kWarps * 32, grid, cache[checked ? 1 : 0]);
  return launch_kernel(kernel, dim3(grid), dim3(kWarps * 32), 0, stream, p);
}

}  // namespace kvq
