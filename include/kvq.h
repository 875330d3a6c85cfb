/*
 * kvq.h -- C ABI of the GB300 (sm_103a) attention-prologue kernels.
 *
 * Two operators of the memory-bound per-token prologue that runs between the
 * QKV projection and attention in LLM serving:
 *
 *   fused_qk_norm_rope
 *       per-head RMSNorm + NeoX rotary embedding, in place, on the Q and K
 *       heads of a packed bf16 QKV tensor; V is neither read nor written.
 *       Source: InfiniOps PR #1019, "Add the NineToothed NVIDIA implementation
 *       of FusedQkNormRope", sections "Summary" (semantics, parameter order
 *       aligned with vLLM's fused_qk_norm_rope, separate [D] weights, the
 *       paired dimension's weight applied to the NeoX partner) and "Notes for
 *       Reviewers" (the guarded fast path: bf16, head_dim 128, full-dimension
 *       NeoX rotation, contiguous packed QKV, contiguous int64 positions).
 *
 *   dsv4_qnorm_rope_kv_rope_quant_insert
 *       DeepSeek-V4-style prologue: per-head RMSNorm + RoPE of q in place, and
 *       RMSNorm + RoPE of the one shared KV vector per token, whose non-rotary
 *       part is quantised to FP8 e4m3 with one UE8M0 (power-of-two) scale per
 *       64-element block and written, with its rotary part, into a paged cache
 *       through slot_mapping.
 *       Sources: FlagGems PR #5449, "[KMCompiler][Hygon] Token-tiled
 *       fused_deepseek_v4_qnorm_rope_kv_rope_quant_insert", section
 *       "Performance" (the operator takes slot_mapping and kv_cache and carries
 *       seven per-block exponents per token), and FlagGems PR #5321,
 *       "[KMCompiler][MetaX][Hygon] Token-tiled ... plus test and benchmark
 *       fixes", section "What the optimisation does" (H query-head slots plus
 *       one KV slot per token; the KV slot does seven quantisation blocks).
 *       The pages fix neither the split of the 512-wide slot nor the cache
 *       entry; this library defines them as listed below.
 *
 * General contract (both operators)
 *   - Every pointer must be dereferenceable by the current CUDA device at
 *     the address given: device memory, or host memory mapped into the
 *     device's address space at the same address (pinned with cudaHostAlloc
 *     or cudaHostRegister on a unified-addressing system).  On an
 *     NVLink-C2C coherent system (Grace-Blackwell) the kernels then read and
 *     write such host buffers directly over the interconnect, one pass, with
 *     no staging copy -- V of the packed QKV tensor never crosses it.  Only
 *     the packed-QKV operator's large batches look at the kind: their
 *     TMA-staged launch shapes copy qkv and cos_sin_cache with the bulk-copy
 *     engine, so they are used only when both are device memory
 *     (cudaPointerGetAttributes, one query per pointer and call); other
 *     buffers take the register-pipelined shape, with the same results.
 *   - All buffers are owned by the caller.  The library allocates no memory,
 *     keeps no per-call state, and never synchronises the stream, so every
 *     entry point can be recorded into a CUDA graph (stream capture); call
 *     each operator once on the device before capturing, so that the
 *     per-device set-up of the large-batch shapes (occupancy query, the
 *     staged shapes' shared-memory opt-in) is done and cached.
 *   - Work is enqueued on `stream` (NULL = legacy default stream).  A KVQ_OK
 *     return means "validated and enqueued"; kernel faults surface on the
 *     stream like any other kernel's.
 *   - Arguments are validated on the host before anything is launched.  On
 *     any error status nothing was launched and no memory was touched.
 *   - num_tokens == 0 returns KVQ_OK without a launch (pointers may be NULL).
 *   - A launch that fails is reported as KVQ_ERR_CUDA (its error is taken
 *     off the CUDA runtime's last-error state); the raw code is available
 *     from kvq_last_cuda_error().  A successful call leaves that state
 *     alone: an error still pending from earlier, unrelated work stays
 *     pending for its owner.  (The library carries its own copy of the CUDA
 *     runtime, linked statically, so its last-error state is not the
 *     caller's in any case.)
 *   - Not checked by the plain entry points (no sizes cross them; the caller
 *     guarantees): 0 <= positions[t] < rows of cos_sin_cache; slot_mapping[t]
 *     == -1 or a slot inside the cache.  Violations are undefined behaviour;
 *     the *_checked entry points below take the sizes and reject them.  Never
 *     checked: no two tokens map to the same slot; q/qkv do not overlap the
 *     cache.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Layout-compatible with cudaStream_t of the CUDA runtime. */
typedef struct CUstream_st* kvq_stream_t;

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_NULL = 1,        /* a required pointer is NULL */
  KVQ_ERR_SHAPE = 2,       /* negative or too-large count, bad block_size */
  KVQ_ERR_UNSUPPORTED = 3, /* head_dim / rotary_dim / is_neox outside the set above */
  KVQ_ERR_ALIGN = 4,       /* a pointer is not aligned as required below */
  KVQ_ERR_CUDA = 5,        /* the kernel launch itself failed */
  KVQ_ERR_VALUE = 6        /* eps negative or not finite; q_out partly overlaps q */
} kvq_status;

/*
 * fused_qk_norm_rope -- in place on qkv; full-dimension rotation
 * (rotary_dim = head_dim).  Same as fused_qk_norm_rope_ex below.
 */
kvq_status fused_qk_norm_rope(void* qkv, int64_t num_tokens, int num_heads_q,
                              int num_heads_k, int num_heads_v, int head_dim,
                              float eps, const void* q_weight,
                              const void* k_weight, const float* cos_sin_cache,
                              int is_neox, const int64_t* positions,
                              kvq_stream_t stream);

/*
 * fused_qk_norm_rope_ex -- in place on qkv, with a rotary width.
 *
 *   qkv            bf16 [num_tokens, (Hq + Hk + Hv) * head_dim], row-major,
 *                  contiguous, 16-byte aligned.  Per token: Hq query heads,
 *                  then Hk key heads, then Hv value heads, head_dim each.
 *                  Q and K heads are replaced by their normalised, rotated
 *                  values; V heads are not accessed.
 *   num_tokens     T >= 0 (T * (Hq + Hk + 1) must stay below 2^31).
 *   num_heads_q/k/v  >= 0 each.
 *   head_dim       64, 128 or 256 (else KVQ_ERR_UNSUPPORTED).
 *   eps            added to the mean square inside the square root; finite,
 *                  >= 0.  With eps = 0 an all-zero head row has no norm
 *                  (0/0): its outputs are NaN.
 *   q_weight, k_weight  bf16 [head_dim] RMSNorm weights, 16-byte aligned.
 *   cos_sin_cache  fp32 [max_pos, rotary_dim]; row p holds cos(p * f_i) for
 *                  i < rotary_dim/2 followed by sin(p * f_i); 16-byte aligned.
 *   rotary_dim     rotated width: a multiple of 16 in [16, head_dim] (else
 *                  KVQ_ERR_UNSUPPORTED); the first rotary_dim dims of each
 *                  head rotate, the rest are normalised only.
 *   is_neox        1: dim i pairs with dim i + rotary_dim/2 (NeoX);
 *                  0: dim 2i pairs with dim 2i+1 (GPT-J); else
 *                  KVQ_ERR_UNSUPPORTED.
 *   positions      int64 [num_tokens], 8-byte aligned, each < max_pos.
 *
 * Per head row x (fp32 arithmetic, one bf16 round-to-nearest-even at the end):
 *   r = 1 / sqrt(sum(x^2) / head_dim + eps);  n_i = x_i * r * w_i
 *   for each rotated pair (a, b) with frequency index i:
 *     out_a = n_a * cos_i - n_b * sin_i,   out_b = n_b * cos_i + n_a * sin_i
 * so the partner enters with its own dimension's weight.  head_dim 128 with
 * full NeoX rotation runs tuned register-pipelined kernels, the other
 * layouts a general one; batches of 128 MiB of Q+K rows and more, in every
 * layout (and from 56 MiB at head_dim 128 with full NeoX rotation), take a
 * kernel that stages rows through shared memory with the bulk-copy (TMA)
 * engine (launch shapes below).  The staged kernel computes
 * 1/sqrt correctly rounded, the others with the hardware approximation
 * (within 2 fp32 ulp), each the form it runs fastest with; outputs of the two
 * are equal but for rare values (about 1 in 10^5), each within the stated
 * tolerance of the exact result.
 * Source: InfiniOps PR #1019, "Summary" (the API carries is_neox, following
 * vLLM's fused_qk_norm_rope) and "Notes for Reviewers" (the fast path the
 * page guards to: bf16, head_dim 128, full-dimension NeoX).
 */
kvq_status fused_qk_norm_rope_ex(void* qkv, int64_t num_tokens, int num_heads_q,
                                 int num_heads_k, int num_heads_v, int head_dim,
                                 float eps, const void* q_weight,
                                 const void* k_weight, const float* cos_sin_cache,
                                 int rotary_dim, int is_neox,
                                 const int64_t* positions, kvq_stream_t stream);

/*
 * dsv4_qnorm_rope_kv_rope_quant_insert -- q in place, cache entries written.
 *
 *   q              bf16 [num_tokens, num_heads, 512], contiguous, 16-byte
 *                  aligned; every head row is normalised with q_weight and
 *                  its last 64 dims rotated, in place, whether or not the
 *                  token has a cache slot.
 *   kv             bf16 [num_tokens, 512], contiguous, 16-byte aligned; read
 *                  only.
 *   num_tokens     T >= 0; num_heads H >= 1 (T * (H + 1) below 2^31).
 *   eps            finite, >= 0.  With eps = 0 an all-zero q row comes out
 *                  NaN, and the cache entry of an all-zero kv vector is
 *                  unspecified (0/0 has no norm).
 *   q_weight, kv_weight  bf16 [512], 16-byte aligned.
 *   cos_sin_cache  fp32 [max_pos, 64]: 32 cosines then 32 sines per row;
 *                  16-byte aligned.
 *   positions      int64 [num_tokens], 8-byte aligned.
 *   slot_mapping   int64 [num_tokens], 8-byte aligned; -1 = no cache write.
 *   kv_cache       uint8 [num_blocks, block_size, 584], contiguous, 8-byte
 *                  aligned; slot s is the 584 bytes at offset s * 584.
 *   block_size     >= 1 (the cache's second dimension).
 *
 * RoPE (both q and kv): interleaved pairs (448 + 2i, 449 + 2i), i < 32, with
 * cos/sin column i of row positions[t].
 * Cache entry of a token with slot s >= 0 (n = normalised, rotated kv, fp32):
 *   bytes [0, 448)    e4m3fn codes of n_j * 2^-e_b, round to nearest even,
 *                     j = 64 b + k for blocks b = 0..6
 *   bytes [448, 576)  n_448 .. n_511 as bf16, little endian
 *   bytes [576, 583)  UE8M0 exponent bytes e_b + 127, b = 0..6, where e_b is
 *                     the smallest integer with 448 * 2^e_b >= max_k |n_64b+k|,
 *                     clamped to [0, 254]
 *   byte  583         0
 * Other cache bytes are never written.
 *
 * Launch shape: a program count T * (H + 1) below the dispatch threshold
 * (kvq_dsv4_dispatch_threshold) takes the small-batch launch shape, otherwise
 * the large-batch one.  Results do not depend on the choice.
 */
kvq_status dsv4_qnorm_rope_kv_rope_quant_insert(
    void* q, const void* kv, int64_t num_tokens, int num_heads, float eps,
    const void* q_weight, const void* kv_weight, const float* cos_sin_cache,
    const int64_t* positions, const int64_t* slot_mapping, uint8_t* kv_cache,
    int block_size, kvq_stream_t stream);

/*
 * dsv4_qnorm_rope_kv_rope_quant_insert_out -- the same operator with a
 * separate q output: q is read only and the normalised, rotated rows go to
 * q_out (bf16 [num_tokens, num_heads, 512], 16-byte aligned).  q_out == q is
 * the in-place operator above; a q_out that partly overlaps q is rejected
 * with KVQ_ERR_VALUE.  Everything else as above.
 */
kvq_status dsv4_qnorm_rope_kv_rope_quant_insert_out(
    const void* q, void* q_out, const void* kv, int64_t num_tokens, int num_heads, float eps,
    const void* q_weight, const void* kv_weight, const float* cos_sin_cache,
    const int64_t* positions, const int64_t* slot_mapping, uint8_t* kv_cache,
    int block_size, kvq_stream_t stream);

/*
 * dsv4_kv_cache_gather -- read cache entries back as bf16 rows (the consumer
 * side of dsv4_qnorm_rope_kv_rope_quant_insert, e.g. for attention).
 *
 *   kv_cache   uint8 [num_blocks, block_size, 584], 8-byte aligned (layout as
 *              written by the insert above); read only.
 *   block_size >= 1.
 *   slots      int64 [num_rows], 8-byte aligned; each -1 or a slot inside
 *              the cache (not checked).
 *   num_rows   >= 0 and below 2^31.
 *   out        bf16 [num_rows, 512], 16-byte aligned, written:
 *                dims 64b + k (b < 7): e4m3(code) * 2^(byte_b - 127), rounded
 *                once to bf16 (exact unless below bf16's range);
 *                dims 448..511: the stored bf16 rotary values;
 *                slots[i] == -1: a row of +0.
 * Source: FlagGems PR #5449, "Performance" (the blockwise UE8M0 layout with
 * seven per-block exponents per token is the cache format to be read back).
 */
kvq_status dsv4_kv_cache_gather(const uint8_t* kv_cache, int block_size, const int64_t* slots,
                                int64_t num_rows, void* out, kvq_stream_t stream);

/*
 * Bounds-checked variants.  The entry points above cannot check positions or
 * slots (no table or cache size crosses them); these take the sizes and a
 * device counter, and the kernels reject what lies outside instead of
 * reading or writing out of range:
 *   max_pos      rows of cos_sin_cache (>= 0); a token whose position is
 *                outside [0, max_pos) is left entirely unchanged (its q/qkv
 *                rows are not written, no cache entry is written);
 *   num_blocks   cache blocks (>= 0); a slot that is neither -1 nor inside
 *                [0, num_blocks * block_size) gets no cache write (the token's
 *                q rows are still processed) -- in the gather, a zero row;
 *   error_count  int32 device counter, 4-byte aligned: the kernels add the
 *                number of rejected tokens (rows, for the gather); the caller
 *                zeroes it and reads it after the stream has run.
 * Accepted tokens give exactly the results of the unchecked entry points.
 * NULL or misaligned error_count, negative sizes: KVQ_ERR_NULL / _ALIGN /
 * _SHAPE, nothing launched.  Otherwise as the unchecked entry points.
 */
kvq_status fused_qk_norm_rope_checked(void* qkv, int64_t num_tokens, int num_heads_q,
                                      int num_heads_k, int num_heads_v, int head_dim,
                                      float eps, const void* q_weight,
                                      const void* k_weight, const float* cos_sin_cache,
                                      int64_t max_pos, int rotary_dim, int is_neox,
                                      const int64_t* positions, int32_t* error_count,
                                      kvq_stream_t stream);
kvq_status dsv4_qnorm_rope_kv_rope_quant_insert_checked(
    const void* q, void* q_out, const void* kv, int64_t num_tokens, int num_heads, float eps,
    const void* q_weight, const void* kv_weight, const float* cos_sin_cache, int64_t max_pos,
    const int64_t* positions, const int64_t* slot_mapping, uint8_t* kv_cache,
    int64_t num_blocks, int block_size, int32_t* error_count, kvq_stream_t stream);
kvq_status dsv4_kv_cache_gather_checked(const uint8_t* kv_cache, int64_t num_blocks,
                                        int block_size, const int64_t* slots, int64_t num_rows,
                                        void* out, int32_t* error_count, kvq_stream_t stream);

/* Static description of a status code (never NULL). */
const char* kvq_status_string(kvq_status status);

/* The cudaError_t value behind the most recent KVQ_ERR_CUDA returned on the
 * calling thread (0 if none). */
int kvq_last_cuda_error(void);

/* Program-count threshold of the DSV4 launch-shape dispatch.  The default is
 * the crossover measured on GB300; the environment variable
 * KVQ_DSV4_DISPATCH_THRESHOLD, read once at the first call that needs it,
 * overrides it (0 = always the token-tiled launch). */
int64_t kvq_dsv4_dispatch_threshold(void);
/* Set the threshold (value >= 0) or restore the default/environment value
 * (value < 0).  Returns the previous threshold.  Not synchronised with
 * concurrent launches on other threads. */
int64_t kvq_set_dsv4_dispatch_threshold(int64_t value);
/* Which side of the threshold a call with these sizes falls on: 0 small-batch
 * launch shape, 1 large-batch launch shape. */
int kvq_dsv4_dispatch_path(int64_t num_tokens, int num_heads);

/*
 * Launch shapes (diagnostics and tuning).  Each operator has a fixed table of
 * launch configurations (kernel shape, warps per CTA, rows per warp).  The
 * automatic dispatch picks one by problem size; the override forces one for
 * every later call of the process (benchmark sweeps, tests).  Every DSV4
 * configuration computes bit-identical results.  QK configurations 0-4
 * (register-pipelined shapes of the head_dim-128 full-NeoX kernel) and 5
 * (the general kernel with 4-dim fragments, any layout) agree bit for bit;
 * so do configurations 7-10 (TMA-staged, bulk<...>, any layout) among
 * themselves.  The two groups differ only in the reciprocal square root
 * (approximate vs correctly rounded; see fused_qk_norm_rope_ex).
 * Configuration 6 (general, 8-dim fragments) also adds the sum of squares in
 * another order.  Automatic choice: below 1216 Q+K rows the small-batch
 * shape; below 128 MiB of Q+K rows (rows x head_dim x 2) the
 * register-pipelined shape (head_dim 128, full NeoX; from 56 MiB on the
 * 24-warp staged shape bulk<24w,2st,3KB> instead) or the general kernel
 * (other layouts); from there on the staged shape bulk<16w,2st,6KB>
 * (kvq_qk_config_for describes head_dim 128, full NeoX).
 *   *_num_configs   number of configurations
 *   *_config_name   static name of configuration id (NULL if out of range)
 *   kvq_set_*_config  force id (0 <= id < num) or restore automatic (id < 0);
 *                   returns the previous override (-1 = automatic), or -2 and
 *                   changes nothing if id >= num.  Not synchronised with
 *                   launches on other threads.
 *   *_config_for    the configuration a call with these sizes would use now
 */
/*
 * Staged launch shapes (the packed-QKV operator's configurations named
 * bulk<...>): each warp keeps its next items in flight in shared memory
 * through the bulk-copy (TMA) engine and waits on an mbarrier per stage.
 * Every such wait polls at most `polls` times (default 1 << 22) and for at
 * most 20 ms.  A warp whose wait runs out lets its copies in flight land
 * (each wait bounded again), then finishes its remaining rows from global
 * memory, with the same results: the limit bounds how long a stalled copy can
 * hold a warp and never changes an output.  0 sends every staged launch
 * straight to that path (diagnostics and tests).  Applies to launches
 * enqueued after the call; returns the previous limit.  Not synchronised
 * with launches on other threads.  The staged shapes copy only from device
 * memory (qkv and the cos/sin table); other buffers take the
 * register-pipelined large-batch shape.
 */
uint32_t kvq_set_stage_wait_limit(uint32_t polls);

/*
 * Staging events of the staged launch shapes on the current device, counted
 * by the kernels in a status word of the library (one per device) since the
 * last reset:
 *   *fallbacks       warps that stopped staging because a stage wait ran out
 *                    (or the limit above is 0) and finished from global
 *                    memory -- results unchanged;
 *   *drain_timeouts  of those, warps whose copies in flight still had not
 *                    landed after the drain wait (2^22 polls or 100 ms per
 *                    copy).  Such a warp still writes correct rows, but its
 *                    CTA may exit while a bulk copy is writing into its
 *                    shared memory, which the hardware leaves undefined; a
 *                    non-zero count means results of work that ran on the
 *                    device at the same time should not be trusted.
 * reset != 0 zeroes both counters after reading them.  The call first waits
 * for all work on the current device to finish (cudaDeviceSynchronize), so
 * it is a diagnostic, not for the launch path.  NULL pointers:
 * KVQ_ERR_NULL; a CUDA error (including one left by earlier asynchronous
 * work): KVQ_ERR_CUDA.  No counterpart in the source pages: a health check
 * of this library's bulk-copy staging.
 */
kvq_status kvq_stage_events(uint64_t* fallbacks, uint64_t* drain_timeouts, int reset);

/*
 * Programmatic dependent launch.  enable != 0 (the default): launches of
 * this library carry CUDA's programmatic stream serialization attribute, so a
 * kernel may be scheduled while the kernel before it on the stream is still
 * finishing.  Every kernel of this library first waits until the kernels it
 * depends on have completed and their writes are visible
 * (griddepcontrol.wait); its one-shot launch shapes then let the next kernel
 * be scheduled (griddepcontrol.launch_dependents), its persistent shapes do
 * not.  Results and stream order are those of ordinary launches; only the
 * launch gaps shrink: on GB300 a 32-layer decode step captured in a CUDA
 * graph goes from 2.47 to 1.79 us per launch, a mid-size step gains 3 %, and
 * the 32768-token step is unchanged.  A kernel of the caller's that follows
 * one of ours and was itself launched with the attribute must wait
 * (griddepcontrol.wait or cudaGridDependencySynchronize) before reading our
 * outputs, as with any programmatic launch.  Returns the previous setting
 * (0 or 1).  Not synchronised with launches on other threads.  No
 * counterpart in the source pages: a launch option of this library.
 */
int kvq_set_programmatic_launch(int enable);

int kvq_qk_num_configs(void);
const char* kvq_qk_config_name(int id);
int kvq_set_qk_config(int id);
int kvq_qk_config_for(int64_t num_tokens, int num_heads_q, int num_heads_k);
int kvq_dsv4_num_configs(void);
const char* kvq_dsv4_config_name(int id);
int kvq_set_dsv4_config(int id);
int kvq_dsv4_config_for(int64_t num_tokens, int num_heads);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
