/*
 * oracle.c -- plain CPU fp64 reference of the attention-prologue operators.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): used by the tests, the package
 * smoke check and the benchmark's CPU baseline, never by the product path.
 *
 * Everything here is the definition written out, one token at a time, one
 * head row at a time, in the order the pages describe the operators: RMSNorm,
 * weight, rotary embedding, then (DSV4 KV vector only) the UE8M0 exponent per
 * 64-element block, the e4m3 codes and the 584-byte cache entry.  Threads only
 * split the token range; every token is computed the same way regardless.
 *
 * Compiled with -ffp-contract=off so that no fused multiply-add changes the
 * fp64 rounding between hosts.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* Scalar codecs                                                             */
/* ------------------------------------------------------------------------ */

/* A bf16 value is, by definition of the format, the upper 16 bits of an
 * IEEE binary32 pattern. */
double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* bf16 keeps 8 significant bits (1 implicit + 7 stored) and binary32's
 * exponent range, so the spacing in the binade [2^e, 2^(e+1)) is 2^(e-7), and
 * 2^-133 below 2^-126.  Divide by the spacing (exact: a power of two), round
 * the quotient to the nearest integer with ties to even, multiply back. */
uint16_t orc_bf16_round(double v) {
  if (isnan(v)) return 0x7fc0u;
  uint16_t sign = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7f80u);
  int k;
  (void)frexp(a, &k); /* a in [2^(k-1), 2^k) */
  int e = k - 1;
  if (e < -126) e = -126;
  double spacing = ldexp(1.0, e - 7);
  double r = nearbyint(a / spacing) * spacing; /* default mode: ties to even */
  if (r > ldexp(255.0, 120)) return (uint16_t)(sign | 0x7f80u); /* > max finite */
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities, only S.1111.111 is NaN.  Normal: (1 + m/8) 2^(E-7); subnormal
 * (E = 0): (m/8) 2^-6. */
double orc_e4m3_value(uint8_t code) {
  int mag = code & 0x7f;
  if (mag == 0x7f) return NAN;
  int ef = mag >> 3, mf = mag & 7;
  double v = (ef == 0) ? ldexp((double)mf, -9) : ldexp(8.0 + mf, ef - 10);
  return (code & 0x80) ? -v : v;
}

/* Nearest representable magnitude, ties to the even code.  The magnitudes of
 * codes 0..126 increase strictly, so a binary search finds the largest code
 * whose value does not exceed |v|; Sterbenz's lemma makes both distances
 * below exact. */
uint8_t orc_e4m3_encode(double v) {
  if (isnan(v)) return 0x7f;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7e);
  int lo = 0, hi = 126; /* value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (orc_e4m3_value((uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  double dl = a - orc_e4m3_value((uint8_t)lo);
  double dh = orc_e4m3_value((uint8_t)hi) - a;
  int c;
  if (dl < dh) c = lo;
  else if (dh < dl) c = hi;
  else c = (lo % 2 == 0) ? lo : hi;
  return (uint8_t)(sign | c);
}

/* UE8M0 scale of a block [FG5449 "Performance": one power-of-two exponent per
 * block]: the smallest power of two 2^e with 448 * 2^e >= amax, so that every
 * element of the block scaled by 2^-e lies within e4m3's +-448.  ldexp is exact,
 * so both comparisons are exact. */
int orc_ue8m0_exponent(double amax) {
  if (!(amax > 0.0)) return -100000;
  int k;
  (void)frexp(amax, &k);
  int e = k - 9; /* 448 = 0.875 * 2^9: a guess within one of the answer */
  while (ldexp(448.0, e) < amax) ++e;
  while (ldexp(448.0, e - 1) >= amax) --e;
  return e;
}

uint8_t orc_ue8m0_byte(double amax) {
  int e = orc_ue8m0_exponent(amax);
  int b = e + 127;
  if (b < 0) b = 0;
  if (b > 254) b = 254;
  return (uint8_t)b;
}

/* Relative distance of amax to the nearer of the two boundaries 448 * 2^(e-1)
 * < amax <= 448 * 2^e that bracket its exponent decision e; HUGE_VAL for
 * amax = 0 (no boundary).  A computation of amax that is off by less than
 * this relative amount reaches the same exponent. */
double orc_exponent_margin(double amax) {
  if (!(amax > 0.0)) return HUGE_VAL;
  const int e = orc_ue8m0_exponent(amax);
  const double up = ldexp(448.0, e) / amax - 1.0;        /* >= 0 */
  const double dn = 1.0 - ldexp(448.0, e - 1) / amax;    /* > 0 */
  return up < dn ? up : dn;
}

void orc_bf16_round_n(const double* v, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round(v[i]);
}

void orc_e4m3_encode_n(const double* v, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

void orc_ue8m0_byte_n(const double* amax, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_ue8m0_byte(amax[i]);
}

/* ------------------------------------------------------------------------ */
/* Row operations                                                            */
/* ------------------------------------------------------------------------ */

/* Per-head RMSNorm followed by the per-dimension weight [IO1019 "Summary"]:
 * n_i = x_i / sqrt(mean(x^2) + eps) * w_i, the mean over all D dimensions. */
static void rms_norm_weight(const uint16_t* x, const uint16_t* w, int D,
                            double eps, double* n) {
  double ss = 0.0;
  for (int i = 0; i < D; ++i) {
    double xi = orc_bf16_value(x[i]);
    ss += xi * xi;
  }
  double r = 1.0 / sqrt(ss / (double)D + eps);
  for (int i = 0; i < D; ++i)
    n[i] = orc_bf16_value(x[i]) * r * orc_bf16_value(w[i]);
}

/* Rotary embedding of dims [off, off + rot) of the normalised row n.  The
 * cos/sin row holds rot/2 cosines then rot/2 sines.  NeoX pairs dim i with
 * dim i + rot/2; the interleaved form pairs 2i with 2i+1.  Each element of a
 * pair is rotated from the already weighted values, so the partner enters
 * with its own dimension's weight [IO1019 "Summary"]. */
static void rope_rotate(double* n, double* mag, int off, int rot, int neox,
                        const float* cs) {
  int half = rot / 2;
  for (int i = 0; i < half; ++i) {
    int a = neox ? off + i : off + 2 * i;
    int b = neox ? off + i + half : off + 2 * i + 1;
    double c = (double)cs[i], s = (double)cs[half + i];
    double na = n[a], nb = n[b];
    n[a] = na * c - nb * s;
    n[b] = nb * c + na * s;
    if (mag) {
      mag[a] = fabs(na * c) + fabs(nb * s);
      mag[b] = fabs(nb * c) + fabs(na * s);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Threading: contiguous token ranges, one per worker                        */
/* ------------------------------------------------------------------------ */

int orc_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

typedef int (*token_fn)(const void* args, int64_t t, double* scratch);

typedef struct {
  token_fn fn;
  const void* args;
  int64_t t0, t1;
  int err;
} range_job;

static void* run_range(void* p) {
  range_job* j = (range_job*)p;
  double scratch[1024];
  for (int64_t t = j->t0; t < j->t1; ++t) {
    int e = j->fn(j->args, t, scratch);
    if (e != 0 && j->err == 0) j->err = e;
  }
  return NULL;
}

static int run_tokens(token_fn fn, const void* args, int64_t T, int nthreads) {
  if (T <= 0) return 0;
  if (nthreads <= 0) nthreads = orc_default_threads();
  if ((int64_t)nthreads > T) nthreads = (int)T;
  range_job* jobs = (range_job*)calloc((size_t)nthreads, sizeof(range_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  char* live = (char*)calloc((size_t)nthreads, 1);
  if (!jobs || !th || !live) { free(jobs); free(th); free(live); return -5; }
  int64_t per = (T + nthreads - 1) / nthreads;
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].fn = fn;
    jobs[i].args = args;
    jobs[i].t0 = (int64_t)i * per;
    jobs[i].t1 = jobs[i].t0 + per < T ? jobs[i].t0 + per : T;
    if (jobs[i].t0 >= jobs[i].t1) continue;
    if (nthreads > 1 && pthread_create(&th[i], NULL, run_range, &jobs[i]) == 0)
      live[i] = 1;
    else
      run_range(&jobs[i]); /* serial: the per-token result is the same */
  }
  int err = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (live[i]) pthread_join(th[i], NULL);
    if (jobs[i].err != 0 && err == 0) err = jobs[i].err;
  }
  free(jobs);
  free(th);
  free(live);
  return err;
}

/* ------------------------------------------------------------------------ */
/* Packed-QKV norm + RoPE [IO1019]                                           */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint16_t* in;
  uint16_t* out;
  int Hq, Hk, Hv, D, rot, neox;
  double eps;
  const uint16_t *qw, *kw;
  const float* cs;
  int64_t max_pos;
  const int64_t* pos;
  double *ref, *mag;
} qk_args;

static int qk_token(const void* p, int64_t t, double* n) {
  const qk_args* A = (const qk_args*)p;
  const int NR = A->Hq + A->Hk, D = A->D;
  const int64_t width = (int64_t)(NR + A->Hv) * D;
  const uint16_t* in = A->in + t * width;
  uint16_t* out = A->out + t * width;
  const int64_t pos = A->pos[t];
  if (pos < 0 || pos >= A->max_pos) return -3;
  const float* cs = A->cs + pos * A->rot;
  for (int h = 0; h < NR; ++h) {
    rms_norm_weight(in + (int64_t)h * D, h < A->Hq ? A->qw : A->kw, D, A->eps, n);
    double* mg = A->mag ? A->mag + (t * NR + h) * (int64_t)D : NULL;
    if (mg)
      for (int i = 0; i < D; ++i) mg[i] = fabs(n[i]);
    rope_rotate(n, mg, 0, A->rot, A->neox, cs);
    for (int i = 0; i < D; ++i) {
      out[(int64_t)h * D + i] = orc_bf16_round(n[i]);
      if (A->ref) A->ref[(t * NR + h) * (int64_t)D + i] = n[i];
    }
  }
  /* V is never modified [IO1019 "Summary": "preserving the V section"]. */
  if (out != in)
    memcpy(out + (int64_t)NR * D, in + (int64_t)NR * D,
           (size_t)A->Hv * (size_t)D * sizeof(uint16_t));
  return 0;
}

int orc_qk_norm_rope(const uint16_t* qkv_in, uint16_t* qkv_out, int64_t T,
                     int Hq, int Hk, int Hv, int D, float eps,
                     const uint16_t* q_weight, const uint16_t* k_weight,
                     const float* cos_sin, int64_t max_pos, int rot_dim,
                     int is_neox, const int64_t* positions,
                     double* ref, double* mag, int nthreads) {
  if (T < 0 || Hq < 0 || Hk < 0 || Hv < 0 || D <= 0 || D > 1024) return -2;
  if (rot_dim < 0 || rot_dim > D || rot_dim % 2 != 0) return -2;
  if (T == 0) return 0;
  if (!qkv_in || !qkv_out || !q_weight || !k_weight || !cos_sin || !positions)
    return -1;
  qk_args A = {qkv_in, qkv_out, Hq, Hk, Hv, D, rot_dim, is_neox ? 1 : 0,
               (double)eps, q_weight, k_weight, cos_sin, max_pos, positions,
               ref, mag};
  return run_tokens(qk_token, &A, T, nthreads);
}

/* ------------------------------------------------------------------------ */
/* DSV4 Q norm + RoPE, KV norm + RoPE + quantise + insert [FG5449, FG5321]   */
/* ------------------------------------------------------------------------ */

enum {
  DSV4_DIM = 512,      /* q head and shared kv width (reading R3) */
  DSV4_ROPE_OFF = 448, /* RoPE on the last 64 dims */
  DSV4_ROPE = 64,
  DSV4_BLOCK = 64,     /* quantisation block */
  DSV4_NBLOCK = 7,     /* "seven per-block exponents per token" */
  DSV4_ENTRY = 584,    /* 448 + 128 + 7 + 1 (reading R6) */
  DSV4_ROPE_AT = 448,
  DSV4_SCALE_AT = 576
};

typedef struct {
  const uint16_t* qin;
  uint16_t* qout;
  const uint16_t* kv;
  int H;
  double eps;
  const uint16_t *qw, *kvw;
  const float* cs;
  int64_t max_pos;
  const int64_t *pos, *slot;
  uint8_t* cache;
  int64_t num_slots;
  int block_size;
  double *q_ref, *q_mag, *kv_ref, *kv_mag, *margin;
} dsv4_args;

static int dsv4_token(const void* p, int64_t t, double* n) {
  const dsv4_args* A = (const dsv4_args*)p;
  const int64_t pos = A->pos[t];
  if (pos < 0 || pos >= A->max_pos) return -3;
  const float* cs = A->cs + pos * DSV4_ROPE;

  /* Q heads: normalise, weight, rotate the tail, round once (in place). */
  for (int h = 0; h < A->H; ++h) {
    const int64_t row = (t * A->H + h) * (int64_t)DSV4_DIM;
    rms_norm_weight(A->qin + row, A->qw, DSV4_DIM, A->eps, n);
    double* mg = A->q_mag ? A->q_mag + row : NULL;
    if (mg)
      for (int i = 0; i < DSV4_DIM; ++i) mg[i] = fabs(n[i]);
    rope_rotate(n, mg, DSV4_ROPE_OFF, DSV4_ROPE, 0, cs);
    for (int i = 0; i < DSV4_DIM; ++i) {
      A->qout[row + i] = orc_bf16_round(n[i]);
      if (A->q_ref) A->q_ref[row + i] = n[i];
    }
  }

  /* Shared KV vector: the same normalisation with its own weight. */
  const int64_t krow = t * (int64_t)DSV4_DIM;
  rms_norm_weight(A->kv + krow, A->kvw, DSV4_DIM, A->eps, n);
  double* kmg = A->kv_mag ? A->kv_mag + krow : NULL;
  if (kmg)
    for (int i = 0; i < DSV4_DIM; ++i) kmg[i] = fabs(n[i]);
  rope_rotate(n, kmg, DSV4_ROPE_OFF, DSV4_ROPE, 0, cs);
  if (A->kv_ref)
    for (int i = 0; i < DSV4_DIM; ++i) A->kv_ref[krow + i] = n[i];

  /* Exponent and codes per block, decided on the unrounded normalised values
   * (reading R5).  Blocks cover dims 0..447, which the rotation does not
   * touch. */
  uint8_t entry[DSV4_ENTRY];
  for (int b = 0; b < DSV4_NBLOCK; ++b) {
    const double* blk = n + b * DSV4_BLOCK;
    double amax = 0.0;
    for (int j = 0; j < DSV4_BLOCK; ++j)
      if (fabs(blk[j]) > amax) amax = fabs(blk[j]);
    const uint8_t byte = orc_ue8m0_byte(amax);
    const int e = (int)byte - 127;
    for (int j = 0; j < DSV4_BLOCK; ++j)
      entry[b * DSV4_BLOCK + j] = orc_e4m3_encode(ldexp(blk[j], -e));
    entry[DSV4_SCALE_AT + b] = byte;
    if (A->margin) A->margin[t * DSV4_NBLOCK + b] = orc_exponent_margin(amax);
  }
  for (int i = 0; i < DSV4_ROPE; ++i) {
    uint16_t bits = orc_bf16_round(n[DSV4_ROPE_OFF + i]);
    entry[DSV4_ROPE_AT + 2 * i] = (uint8_t)(bits & 0xff);
    entry[DSV4_ROPE_AT + 2 * i + 1] = (uint8_t)(bits >> 8);
  }
  entry[DSV4_ENTRY - 1] = 0;

  /* Paged insert through slot_mapping; -1 means the token has no slot. */
  const int64_t s = A->slot[t];
  if (s < 0) return 0;
  if (s >= A->num_slots) return -4;
  const int64_t blk = s / A->block_size, off = s % A->block_size;
  memcpy(A->cache + (blk * A->block_size + off) * (int64_t)DSV4_ENTRY, entry,
         DSV4_ENTRY);
  return 0;
}

int orc_dsv4(const uint16_t* q_in, uint16_t* q_out, const uint16_t* kv,
             int64_t T, int H, float eps,
             const uint16_t* q_weight, const uint16_t* kv_weight,
             const float* cos_sin, int64_t max_pos, const int64_t* positions,
             const int64_t* slot_mapping, uint8_t* kv_cache,
             int64_t num_blocks, int block_size,
             double* q_ref, double* q_mag, double* kv_ref, double* kv_mag,
             double* exp_margin, int nthreads) {
  if (T < 0 || H < 0 || block_size <= 0 || num_blocks < 0) return -2;
  if (T == 0) return 0;
  if ((H > 0 && (!q_in || !q_out || !q_weight)) || !kv || !kv_weight ||
      !cos_sin || !positions || !slot_mapping || !kv_cache)
    return -1;
  dsv4_args A = {q_in, q_out, kv, H, (double)eps, q_weight, kv_weight,
                 cos_sin, max_pos, positions, slot_mapping, kv_cache,
                 num_blocks * (int64_t)block_size, block_size,
                 q_ref, q_mag, kv_ref, kv_mag, exp_margin};
  return run_tokens(dsv4_token, &A, T, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Reading entries back                                                      */
/* ------------------------------------------------------------------------ */

int orc_dsv4_gather(const uint8_t* kv_cache, int64_t num_blocks, int block_size,
                    const int64_t* slots, int64_t n, uint16_t* out) {
  if (n < 0 || block_size <= 0 || num_blocks < 0) return -2;
  if (n == 0) return 0;
  if (!kv_cache || !slots || !out) return -1;
  const int64_t num_slots = num_blocks * (int64_t)block_size;
  for (int64_t i = 0; i < n; ++i) {
    uint16_t* row = out + i * DSV4_DIM;
    const int64_t s = slots[i];
    if (s < 0) {
      memset(row, 0, DSV4_DIM * sizeof(uint16_t));
      continue;
    }
    if (s >= num_slots) return -4;
    const int64_t blk = s / block_size, off = s % block_size;
    const uint8_t* e = kv_cache + (blk * block_size + off) * (int64_t)DSV4_ENTRY;
    for (int b = 0; b < DSV4_NBLOCK; ++b) {
      const int ex = (int)e[DSV4_SCALE_AT + b] - 127;
      for (int j = 0; j < DSV4_BLOCK; ++j)
        row[b * DSV4_BLOCK + j] = orc_bf16_round(ldexp(orc_e4m3_value(e[b * DSV4_BLOCK + j]), ex));
    }
    for (int i2 = 0; i2 < DSV4_ROPE; ++i2)
      row[DSV4_ROPE_OFF + i2] =
          (uint16_t)(e[DSV4_ROPE_AT + 2 * i2] | ((uint16_t)e[DSV4_ROPE_AT + 2 * i2 + 1] << 8));
  }
  return 0;
}
