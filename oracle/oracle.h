/*
 * oracle.h -- CPU reference ("oracle") for the two attention-prologue operators.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this code: only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA library; the only thing both sides see is the same
 * seeded input bytes.
 *
 * Sources (web pages; cited by title and section):
 *   [IO1019]  InfiniOps PR #1019, "Add the NineToothed NVIDIA implementation of
 *             FusedQkNormRope" -- sections "Summary" and "Notes for Reviewers":
 *             per-head Q/K RMSNorm followed by NeoX RoPE, in place on a packed
 *             [tokens, (Hq+Hk+Hv)*D] tensor, V unchanged, separate [D] weights,
 *             and the paired dimension's weight applied to the NeoX partner.
 *   [FG5449]  FlagGems PR #5449, "[KMCompiler][Hygon] Token-tiled
 *             fused_deepseek_v4_qnorm_rope_kv_rope_quant_insert" -- section
 *             "Performance" (seven per-block exponents per token, slot_mapping
 *             and kv_cache inputs, UE8M0 blockwise layout).
 *   [FG5321]  FlagGems PR #5321, "[KMCompiler][MetaX][Hygon] Token-tiled
 *             fused_deepseek_v4_qnorm_rope_kv_rope_quant_insert, plus test and
 *             benchmark fixes" -- section "What the optimisation does" (one KV
 *             slot per token next to the Q heads; seven quantisation blocks)
 *             and "The four test and benchmark fixes" (per-token independence,
 *             so token slices are exact).
 *
 * Where the pages are silent the oracle takes the readings below (each is also
 * listed with its justification in the design notes of the repository):
 *   R1 cos_sin_cache row p = [cos(p f_0) .. cos(p f_{R/2-1}), sin(p f_0) .. ],
 *      R = rotary width; the table is an input, consumed as fp32.
 *   R2 order: RMSNorm (mean over the whole head, eps inside the sqrt), then the
 *      weight, then RoPE; a single rounding of every output.
 *   R3 DSV4 head = 512 dims; RoPE on the last 64, interleaved pairs
 *      (448+2i, 449+2i); dims 0..447 form 7 quantisation blocks of 64.
 *   R4 UE8M0 exponent e = smallest integer with 448 * 2^e >= amax; stored byte
 *      clamp(e + 127, 0, 254); codes = e4m3fn round-to-nearest-even of
 *      n * 2^-e with e = byte - 127.
 *   R5 the exponent and code decisions are taken on the unrounded (fp64)
 *      normalised value n itself: amax, the exponent and n * 2^-e are exact
 *      functions of n and the codes are rounded once from n * 2^-e.  The
 *      pages fix no precision for these decisions; an implementation that
 *      computes n in fp32 can land on the other side of an exponent boundary
 *      or an e4m3 rounding midpoint, which the comparison tolerates (margin
 *      below) rather than the oracle copying that precision.
 *   R6 cache entry (584 bytes) at byte offset slot * 584 of a contiguous
 *      [num_blocks, block_size, 584] uint8 cache: [0,448) e4m3 codes,
 *      [448,576) 64 bf16 RoPE'd values (little endian), [576,583) the seven
 *      exponent bytes, [583] = 0.  slot < 0 means "skip"; other bytes of the
 *      cache are never written.
 *   R7 the DSV4 q tensor is updated in place; kv is read only; q is processed
 *      even when the token's slot is -1.
 */
#ifndef KVQ_ORACLE_H
#define KVQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar codecs (exposed so that tests can pin them) ---------------- */

/* bf16 bit pattern -> exact value. */
double orc_bf16_value(uint16_t bits);
/* Exact value -> bf16 bits, one round-to-nearest-even step (no detour through
 * fp32).  Overflow gives +-inf, NaN gives 0x7fc0. */
uint16_t orc_bf16_round(double v);
/* e4m3fn code -> exact value (NaN for 0x7f / 0xff). */
double orc_e4m3_value(uint8_t code);
/* Exact value -> e4m3fn code: nearest representable value, ties to the even
 * code, magnitudes above 448 saturate to 448, the sign is kept (so negative
 * values that round to zero give 0x80).  NaN gives 0x7f. */
uint8_t orc_e4m3_encode(double v);
/* Smallest integer e with 448 * 2^e >= amax (amax > 0); returns -100000 for
 * amax <= 0. */
int orc_ue8m0_exponent(double amax);
/* clamp(orc_ue8m0_exponent(amax) + 127, 0, 254). */
uint8_t orc_ue8m0_byte(double amax);
/* Relative distance (|amax - B| / amax) from amax to the nearer of the two
 * boundaries B = 448 * 2^(e-1) and 448 * 2^e that bracket its exponent
 * decision e; HUGE_VAL for amax <= 0. */
double orc_exponent_margin(double amax);

/* Element-wise array forms of the three encoders above (for the tests). */
void orc_bf16_round_n(const double* v, uint16_t* out, int64_t n);
void orc_e4m3_encode_n(const double* v, uint8_t* out, int64_t n);
void orc_ue8m0_byte_n(const double* amax, uint8_t* out, int64_t n);

/* ---- operators ----------------------------------------------------------- */

/* Number of worker threads used when nthreads <= 0 (all online host cores). */
int orc_default_threads(void);

/*
 * Packed-QKV per-head RMSNorm + RoPE [IO1019].
 *   qkv_in   bf16 bits [T, (Hq+Hk+Hv)*D]
 *   qkv_out  bf16 bits [T, (Hq+Hk+Hv)*D]; may equal qkv_in.  V columns are
 *            copied through unchanged.
 *   cos_sin  fp32 [max_pos, rot_dim]; positions int64 [T], each in [0,max_pos)
 *   rot_dim  rotary width (== D for full rotation), even, <= D
 *   is_neox  1: pairs (i, i+rot_dim/2); 0: pairs (2i, 2i+1)
 *   ref      optional fp64 [T, Hq+Hk, D]: exact (unrounded) results
 *   mag      optional fp64 [T, Hq+Hk, D]: sum of the magnitudes of the terms
 *            that form each result (|n_i| unrotated, |n_a c| + |n_b s| rotated)
 * Returns 0, or a negative code for bad arguments (-1 null, -2 shape,
 * -3 position out of range).
 */
int orc_qk_norm_rope(const uint16_t* qkv_in, uint16_t* qkv_out, int64_t T,
                     int Hq, int Hk, int Hv, int D, float eps,
                     const uint16_t* q_weight, const uint16_t* k_weight,
                     const float* cos_sin, int64_t max_pos, int rot_dim,
                     int is_neox, const int64_t* positions,
                     double* ref, double* mag, int nthreads);

/*
 * DeepSeek-V4-style Q norm + RoPE and KV norm + RoPE + UE8M0/e4m3 quantise +
 * paged insert [FG5449, FG5321], readings R3-R7.
 *   q_in/q_out bf16 bits [T, H, 512] (may alias)
 *   kv         bf16 bits [T, 512]
 *   cos_sin    fp32 [max_pos, 64]
 *   slot_mapping int64 [T]; -1 = skip; else < num_blocks*block_size
 *   kv_cache   uint8 [num_blocks, block_size, 584], written in place
 *   q_ref, q_mag   optional fp64 [T, H, 512]
 *   kv_ref, kv_mag optional fp64 [T, 512] (n after RoPE, before any rounding)
 *   exp_margin     optional fp64 [T, 7]: orc_exponent_margin of each block's
 *                  amax (HUGE_VAL for an all-zero block)
 * Returns 0 or a negative code (-1 null, -2 shape, -3 position out of range,
 * -4 slot out of range).
 */
int orc_dsv4(const uint16_t* q_in, uint16_t* q_out, const uint16_t* kv,
             int64_t T, int H, float eps,
             const uint16_t* q_weight, const uint16_t* kv_weight,
             const float* cos_sin, int64_t max_pos, const int64_t* positions,
             const int64_t* slot_mapping, uint8_t* kv_cache,
             int64_t num_blocks, int block_size,
             double* q_ref, double* q_mag, double* kv_ref, double* kv_mag,
             double* exp_margin, int nthreads);

/*
 * Read cache entries back (the consumer side of the DSV4 insert): row i of
 * `out` (bf16 bits [n, 512]) is the entry at slot slots[i]: dims 64b+k
 * (b < 7) = bf16(e4m3_value(code) * 2^(byte_b - 127)), one rounding; dims
 * 448..511 = the stored bf16 values; slots[i] < 0 gives a row of +0.
 * Returns 0, -1 null, -2 shape, -4 slot out of range.
 */
int orc_dsv4_gather(const uint8_t* kv_cache, int64_t num_blocks, int block_size,
                    const int64_t* slots, int64_t n, uint16_t* out);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_ORACLE_H */
