/*
 * kvq_c_client.c -- a plain C99 caller of the C ABI (include/kvq.h), with no
 * Python and no torch: device buffers from the CUDA runtime's C API, one call
 * of every operator on cases whose results are exact by construction, and
 * the host-side error paths.
 *
 *   packed QKV:  x = +-1 everywhere, eps = 0, position 0 (cos = 1, sin = 0):
 *                r = 1 exactly and the rotation is the identity, so each
 *                output is the weight with the sign of x, bit for bit; V is
 *                untouched.  Run through the head_dim-128 NeoX path and the
 *                general path (GPT-J pairs, rotary_dim 64).
 *   DSV4:        q = kv = 1, eps = 0, position 0, kv_weight = 1, 2, 4, 8,
 *                0.5, 3, 5 on the seven 64-dim blocks and 1 on the rotary
 *                dims: the entry is codes 0x78 (blocks 0-4), 0x7c, 0x7a,
 *                the rotary bf16 1.0 values and exponent bytes
 *                119, 120, 121, 122, 118, 120, 121 (smallest 2^e with
 *                448 * 2^e >= block max), and q comes out as 1.0.
 *   gather:      reading that entry back gives the block weights exactly.
 *   errors:      a CUDA error pending in the caller's runtime survives a
 *                successful call of the library.
 *
 * Exit status 0 when every check holds.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "kvq.h"

static int failures = 0;

#define CHECK(cond, ...)                      \
  do {                                        \
    if (!(cond)) {                            \
      fprintf(stderr, "FAIL: " __VA_ARGS__);  \
      fprintf(stderr, "\n");                  \
      ++failures;                             \
    }                                         \
  } while (0)

#define CUDA(call)                                                              \
  do {                                                                          \
    cudaError_t e_ = (call);                                                    \
    if (e_ != cudaSuccess) {                                                    \
      fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_),       \
              __FILE__, __LINE__);                                              \
      exit(2);                                                                  \
    }                                                                           \
  } while (0)

static void* dev_copy(const void* host, size_t bytes) {
  void* d = NULL;
  CUDA(cudaMalloc(&d, bytes));
  CUDA(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice));
  return d;
}

/* cos/sin table of `rows` rows and width `rot`: row 0 = cos 1, sin 0; the
 * other rows hold arbitrary values that no call reads. */
static float* angle_table(int rows, int rot) {
  float* t = (float*)malloc(sizeof(float) * rows * rot);
  for (int p = 0; p < rows; ++p)
    for (int i = 0; i < rot; ++i) t[p * rot + i] = p == 0 ? (i < rot / 2 ? 1.0f : 0.0f) : 0.25f;
  return t;
}

/* Packed-QKV operator on x = +-1: each Q/K output is +-w, V unchanged. */
static void qk_case(int rotary_dim, int is_neox) {
  enum { T = 9, HQ = 2, HK = 2, HV = 1, D = 128, P = 4 };
  const int row = (HQ + HK + HV) * D;
  uint16_t* x = (uint16_t*)malloc(sizeof(uint16_t) * T * row);
  uint16_t qw[D], kw[D];
  int64_t pos[T];
  uint32_t state = 12345u;
  for (int i = 0; i < T * row; ++i) {
    state = state * 1664525u + 1013904223u;
    x[i] = (state >> 31) ? 0xBF80u : 0x3F80u; /* -1.0 or +1.0 in bf16 */
  }
  for (int i = 0; i < D; ++i) {
    qw[i] = (uint16_t)(0x3F80u + i);      /* 1 + i/128 */
    kw[i] = (uint16_t)(0x4000u + 2 * i);  /* 2 + i/32 */
  }
  for (int t = 0; t < T; ++t) pos[t] = 0;
  float* cs = angle_table(P, rotary_dim);
  void* d_x = dev_copy(x, sizeof(uint16_t) * T * row);
  void* d_qw = dev_copy(qw, sizeof qw);
  void* d_kw = dev_copy(kw, sizeof kw);
  float* d_cs = (float*)dev_copy(cs, sizeof(float) * P * rotary_dim);
  int64_t* d_pos = (int64_t*)dev_copy(pos, sizeof pos);

  kvq_status s = fused_qk_norm_rope_ex(d_x, T, HQ, HK, HV, D, 0.0f, d_qw, d_kw, d_cs,
                                       rotary_dim, is_neox, d_pos, NULL);
  CHECK(s == KVQ_OK, "fused_qk_norm_rope_ex(rot %d, neox %d): %s", rotary_dim, is_neox,
        kvq_status_string(s));
  CUDA(cudaDeviceSynchronize());
  uint16_t* y = (uint16_t*)malloc(sizeof(uint16_t) * T * row);
  CUDA(cudaMemcpy(y, d_x, sizeof(uint16_t) * T * row, cudaMemcpyDeviceToHost));
  int bad = 0;
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < HQ + HK + HV; ++h)
      for (int i = 0; i < D; ++i) {
        const int k = t * row + h * D + i;
        uint16_t want = x[k];
        if (h < HQ + HK) want = (uint16_t)((h < HQ ? qw[i] : kw[i]) | (x[k] & 0x8000u));
        bad += y[k] != want;
      }
  CHECK(bad == 0, "packed QKV (rot %d, neox %d): %d values differ", rotary_dim, is_neox, bad);

  /* host-side validation: nothing is launched on an error */
  CHECK(fused_qk_norm_rope(NULL, T, HQ, HK, HV, D, 1e-6f, d_qw, d_kw, d_cs, 1, d_pos, NULL) ==
            KVQ_ERR_NULL, "NULL qkv");
  CHECK(fused_qk_norm_rope(d_x, T, HQ, HK, HV, 96, 1e-6f, d_qw, d_kw, d_cs, 1, d_pos, NULL) ==
            KVQ_ERR_UNSUPPORTED, "head_dim 96");
  CHECK(fused_qk_norm_rope(d_x, 0, HQ, HK, HV, D, 1e-6f, d_qw, d_kw, d_cs, 1, d_pos, NULL) ==
            KVQ_OK, "zero tokens");

  CUDA(cudaFree(d_x));
  CUDA(cudaFree(d_qw));
  CUDA(cudaFree(d_kw));
  CUDA(cudaFree(d_cs));
  CUDA(cudaFree(d_pos));
  free(x);
  free(y);
  free(cs);
}

/* DSV4 operator and the read-back on the hand-derived entry. */
static void dsv4_case(void) {
  enum { T = 2, H = 3, DIM = 512, ENTRY = 584, BLOCKS = 2, BS = 4, P = 4 };
  static const uint16_t block_w[7] = {0x3F80u, 0x4000u, 0x4080u, 0x4100u,
                                      0x3F00u, 0x4040u, 0x40A0u}; /* 1 2 4 8 0.5 3 5 */
  static const uint8_t code[7] = {0x78, 0x78, 0x78, 0x78, 0x78, 0x7C, 0x7A};
  static const uint8_t expo[7] = {119, 120, 121, 122, 118, 120, 121};
  uint16_t q[T * H * DIM], kv[T * DIM], qw[DIM], kvw[DIM];
  int64_t pos[T] = {0, 0}, slots[T] = {5, -1}; /* token 1 has no cache slot */
  const size_t cache_bytes = (size_t)BLOCKS * BS * ENTRY;
  uint8_t* cache = (uint8_t*)malloc(cache_bytes);
  for (int i = 0; i < T * H * DIM; ++i) q[i] = 0x3F80u;
  for (int i = 0; i < T * DIM; ++i) kv[i] = 0x3F80u;
  for (int i = 0; i < DIM; ++i) {
    qw[i] = 0x3F80u;
    kvw[i] = i < 448 ? block_w[i / 64] : 0x3F80u;
  }
  memset(cache, 0xA5, cache_bytes);
  float* cs = angle_table(P, 64);
  void* d_q = dev_copy(q, sizeof q);
  void* d_kv = dev_copy(kv, sizeof kv);
  void* d_qw = dev_copy(qw, sizeof qw);
  void* d_kvw = dev_copy(kvw, sizeof kvw);
  float* d_cs = (float*)dev_copy(cs, sizeof(float) * P * 64);
  int64_t* d_pos = (int64_t*)dev_copy(pos, sizeof pos);
  int64_t* d_slots = (int64_t*)dev_copy(slots, sizeof slots);
  uint8_t* d_cache = (uint8_t*)dev_copy(cache, cache_bytes);

  kvq_status s = dsv4_qnorm_rope_kv_rope_quant_insert(d_q, d_kv, T, H, 0.0f, d_qw, d_kvw, d_cs,
                                                      d_pos, d_slots, d_cache, BS, NULL);
  CHECK(s == KVQ_OK, "dsv4 insert: %s", kvq_status_string(s));
  CUDA(cudaDeviceSynchronize());
  CUDA(cudaMemcpy(q, d_q, sizeof q, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(cache, d_cache, cache_bytes, cudaMemcpyDeviceToHost));
  int bad = 0;
  for (int i = 0; i < T * H * DIM; ++i) bad += q[i] != 0x3F80u;
  CHECK(bad == 0, "dsv4 q: %d values differ from 1.0", bad);
  bad = 0;
  for (size_t b = 0; b < cache_bytes; ++b) {
    const long rel = (long)b - 5L * ENTRY;
    uint8_t want = 0xA5;
    if (rel >= 0 && rel < ENTRY) {
      if (rel < 448) want = code[rel / 64];
      else if (rel < 576) want = (rel & 1) ? 0x3F : 0x80; /* bf16 1.0, little endian */
      else if (rel < 583) want = expo[rel - 576];
      else want = 0;
    }
    bad += cache[b] != want;
  }
  CHECK(bad == 0, "dsv4 cache: %d bytes differ from the hand-derived entry", bad);

  /* read back slots 5 and -1 */
  int64_t back[2] = {5, -1};
  int64_t* d_back = (int64_t*)dev_copy(back, sizeof back);
  uint16_t rows[2 * DIM];
  void* d_rows = NULL;
  CUDA(cudaMalloc(&d_rows, sizeof rows));
  s = dsv4_kv_cache_gather(d_cache, BS, d_back, 2, d_rows, NULL);
  CHECK(s == KVQ_OK, "gather: %s", kvq_status_string(s));
  CUDA(cudaDeviceSynchronize());
  CUDA(cudaMemcpy(rows, d_rows, sizeof rows, cudaMemcpyDeviceToHost));
  bad = 0;
  for (int i = 0; i < DIM; ++i) bad += rows[i] != (i < 448 ? block_w[i / 64] : 0x3F80u);
  for (int i = 0; i < DIM; ++i) bad += rows[DIM + i] != 0;
  CHECK(bad == 0, "gather: %d values differ", bad);

  CHECK(dsv4_qnorm_rope_kv_rope_quant_insert(d_q, d_kv, T, H, 0.0f, d_qw, d_kvw, d_cs, d_pos,
                                             d_slots, d_cache, 0, NULL) == KVQ_ERR_SHAPE,
        "block_size 0");
  CHECK(dsv4_qnorm_rope_kv_rope_quant_insert(d_q, d_kv, T, H, -1.0f, d_qw, d_kvw, d_cs, d_pos,
                                             d_slots, d_cache, BS, NULL) == KVQ_ERR_VALUE,
        "negative eps");

  void* bufs[] = {d_q, d_kv, d_qw, d_kvw, d_cs, d_pos, d_slots, d_cache, d_back, d_rows};
  for (size_t i = 0; i < sizeof bufs / sizeof bufs[0]; ++i) CUDA(cudaFree(bufs[i]));
  free(cache);
  free(cs);
}

/* An error the caller has pending in its CUDA runtime (here a refused
 * allocation, which is not sticky) is still there after a successful call of
 * the library: the library never consumes another party's error. */
static void pending_error_case(void) {
  void* huge = NULL;
  CHECK(cudaMalloc(&huge, (size_t)1 << 62) == cudaErrorMemoryAllocation, "huge allocation");
  qk_case(128, 1);
  CHECK(cudaPeekAtLastError() == cudaErrorMemoryAllocation,
        "the caller's pending error was consumed by a library call");
  CHECK(cudaGetLastError() == cudaErrorMemoryAllocation, "pending error");
  CHECK(cudaGetLastError() == cudaSuccess, "error state cleared");
}

int main(void) {
  for (int st = 0; st <= 6; ++st) CHECK(kvq_status_string((kvq_status)st) != NULL, "status %d", st);
  qk_case(128, 1);  /* head_dim-128 NeoX kernel */
  qk_case(64, 0);   /* general kernel: GPT-J pairs, partial rotation */
  dsv4_case();
  pending_error_case();
  if (failures) {
    fprintf(stderr, "%d check(s) failed\n", failures);
    return 1;
  }
  printf("c client ok\n");
  return 0;
}
