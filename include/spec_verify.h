/*
 * spec_verify.h -- C ABI of the batched speculative-decoding verify step
 * (sm_103a).
 *
 * One verify step, for B sequences with their own KV lengths L_i and their own
 * draft counts K_i (no padding anywhere), does three things:
 *   1. verify attention: every query head of the K_i + 1 block rows of
 *      sequence i attends over that sequence's KV cache plus the block itself,
 *      causally inside the block ("Accelerating Large Language Model Decoding
 *      with Speculative Sampling", section "Conditional scoring"; batch without
 *      padding: BASS and EMS-SD abstracts); optionally over a prefill KV block
 *      shared by a group of sequences (bifurcated attention abstract);
 *   2. modified rejection sampling over the vocabulary (same SpS paper,
 *      section "Modified rejection sampling"): temperature and nucleus applied
 *      to both q and p first, accept draft x~ while u < min(1, q(x~)/p(x~)),
 *      on the first rejection draw from max(0, q - p) normalized, after K_i
 *      acceptances draw a bonus token from the last target row;
 *   3. append of the accepted rows' K/V only (EMS-SD abstract), giving every
 *      sequence its own new length.
 *
 * Conventions shared by every entry point
 *   - Pointers marked [dev] are device pointers, [host] are host pointers.
 *     Every buffer is owned by the caller; the library keeps no pointer after
 *     a call returns and allocates nothing.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and never synchronize.
 *   - Row bookkeeping: cu_q[B+1] is the prefix sum of R_i = K_i + 1 (block
 *     rows of sequence i are cu_q[i] .. cu_q[i+1]-1, R = cu_q[B]); draft rows
 *     (draft logits, draft tokens) of sequence i are cu_q[i]-i .. cu_q[i+1]-i-2
 *     (R - B rows in total).  Block row 0 is the pending token (its K/V not yet
 *     cached), rows 1..K_i the drafts; block row j sits at token index L_i + j
 *     and its logits decide token index L_i + j + 1.
 *   - KV pool layout: token-major [pool_rows, Hkv, D]; sequence i's committed
 *     rows are kv_start[i] .. kv_start[i] + kv_len[i] - 1.  The regions
 *     [kv_start[i], kv_start[i] + kv_cap[i]) must not overlap each other or a
 *     shared prefix.
 *   - Host-checkable errors return a status != SV_OK synchronously and launch
 *     nothing; sv_last_error() then describes it.  Data-dependent problems set
 *     bits in *dev_status (atomic OR, never cleared by the library) and skip
 *     only the affected sequence.  Kernels never trap.
 *   - Workspace: sv_workspace_bytes() gives the size; the buffer must be
 *     16-byte aligned and zeroed once (sv_workspace_init) before its first
 *     use; every call leaves it ready for the next.  Calls that share one
 *     workspace must not overlap in time (same stream, or ordered).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SV_API __attribute__((visibility("default")))
#define SV_ABI_VERSION 5

typedef enum sv_status {
  SV_OK = 0,
  SV_ERR_INVALID = 1,      /* bad argument (null pointer, size out of range) */
  SV_ERR_WORKSPACE = 2,    /* workspace missing, misaligned or too small */
  SV_ERR_CUDA = 3,         /* a CUDA runtime call failed (launch, attribute) */
  SV_ERR_UNSUPPORTED = 4   /* valid but not built: e.g. head_dim not 64/128 */
} sv_status;

/* SV_E4M3: 8-bit floating point K/V codes (sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, subnormals at exponent 0, no infinities, S.1111.111 NaN;
 * the OCP FP8 "E4M3" layout), read as code value times a per-tensor scale.
 * Only as sv_attn_args.kv_dtype and as the dtype of kv_append_ragged. */
typedef enum sv_dtype { SV_F32 = 0, SV_BF16 = 1, SV_E4M3 = 2 } sv_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
enum {
  SV_DEV_CAPACITY = 1u,        /* append would pass kv_cap[i]: append skipped,
                                  new_kv_len[i] = kv_len[i] */
  SV_DEV_BAD_TOKEN = 2u,       /* a draft token outside [0, V): treated as a
                                  rejection at that row */
  SV_DEV_NONFINITE = 4u,       /* a logits row holds NaN/+inf or only -inf:
                                  the sequence fails (num_accepted = -1, its
                                  out_tokens stay -1, no append) */
  SV_DEV_EMPTY_RESIDUAL = 8u,  /* rejected but max(0, q-p) sums to 0: the
                                  token is drawn from the target row instead */
  SV_DEV_BAD_LENGTH = 16u,     /* cu_q / kv_len / kv_start / prefix values
                                  inconsistent with the host bounds or the
                                  pool: that sequence is skipped */
  SV_DEV_TIMEOUT = 32u,        /* an internal wait of the attention pipeline
                                  gave up (not expected at the built-in bound,
                                  see sv_set_wait_limit; outputs of the
                                  affected CTA are left unwritten) */
  SV_DEV_BAD_PARAM = 64u       /* a per-sequence temperature < 0 or NaN, top_p
                                  <= 0 or NaN, or top_k < 0: that sequence
                                  fails (with SV_DEV_NONFINITE) */
};

/* Verify attention (a1, a1b).  scale * q.k softmax over keys
 *   [prefix rows of group[i] (if num_groups > 0)] ++ [kv rows of i] ++
 *   [block rows 0..j of i]
 * with KV head h / (Hq / Hkv); fp32 accumulation.  Split over KV chunks
 * (partials in the workspace) and merged by the last chunk to finish. */
typedef struct sv_attn_args {
  int32_t batch;            /* B >= 0 */
  int32_t num_q_heads;      /* Hq >= 1 */
  int32_t num_kv_heads;     /* Hkv >= 1, Hq % Hkv == 0 */
  int32_t head_dim;         /* D: 64 or 128 */
  int32_t dtype;            /* sv_dtype of q, k_new, v_new, caches and out */
  int32_t max_q_rows;       /* host bound on R_i, 1..16; (Hq/Hkv)*max_q_rows <= 64 */
  int64_t num_rows;         /* R = cu_q[B] (host copy) */
  int64_t kv_rows_bound;    /* host bound on sum_i kv_len[i] (sizes the split) */
  int64_t pool_rows;        /* rows of k_cache / v_cache */
  float scale;              /* softmax scale; 0 -> 1/sqrt(D) */
  int32_t num_groups;       /* G; 0 = no shared prefix */
  int64_t prefix_rows_bound;/* host bound on sum_g prefix_len[g] (0 if G = 0) */
  const int32_t *cu_q;      /* [dev] [B+1] */
  const void *q;            /* [dev] [R, Hq, D] */
  const void *k_new;        /* [dev] [R, Hkv, D] block K rows */
  const void *v_new;        /* [dev] [R, Hkv, D] block V rows */
  const void *k_cache;      /* [dev] [pool_rows, Hkv, D] */
  const void *v_cache;      /* [dev] [pool_rows, Hkv, D] */
  const int64_t *kv_start;  /* [dev] [B] first pool row of sequence i */
  const int32_t *kv_len;    /* [dev] [B] L_i >= 0 */
  const int32_t *group;     /* [dev] [B] group of sequence i (NULL if G = 0) */
  const int64_t *prefix_start; /* [dev] [G] first pool row of the prefix */
  const int32_t *prefix_len;   /* [dev] [G] */
  void *out;                /* [dev] [R, Hq, D] */
  uint32_t *dev_status;     /* [dev] one word */
  /* Added in ABI 4: an 8-bit KV cache.  The speculative-sampling paper (end
   * of section "Modified rejection sampling") notes the method composes with
   * memory-saving techniques such as quantization, since it leaves the
   * transformer body alone.  kv_dtype SV_E4M3: k_new, v_new, k_cache and
   * v_cache hold E4M3 codes (one byte per element, same [rows, Hkv, D]
   * layout; the step's own rows come in the cache's format), read as
   * code * k_scale and code * v_scale; q and out stay bf16.  Built for dtype
   * SV_BF16, head_dim 128, no shared prefix and (Hq/Hkv)*max_q_rows <= 16;
   * other combinations return SV_ERR_UNSUPPORTED.  The tensor-core operands
   * are f16, so q is rounded to f16: q must lie within the f16 range
   * (|q| <= 65504).  A larger q element becomes infinite and makes the
   * outputs of its own (row, head) non-finite (other rows and heads are
   * unaffected); no status bit reports it. */
  int32_t kv_dtype;         /* 0 (K/V in dtype) or SV_E4M3 */
  float k_scale;            /* E4M3 K scale; 0 -> 1 */
  float v_scale;            /* E4M3 V scale; 0 -> 1 */
} sv_attn_args;

/* Rejection sampling (a2-a5, a7).  Per sequence: processes its target rows
 * (K_i + 1) and draft rows (K_i) with temperature then nucleus, accepts
 * drafts left to right with Philox4x32-10 uniforms keyed by (seed,
 * seq_ids[i], position, stream 0), draws the residual or bonus token by
 * inverse CDF in vocabulary order.  Outputs: num_accepted[i] = n_i in
 * [0, K_i] (-1 on failure); out_tokens[cu_q[i] + j] = draft j+1 for j < n_i,
 * the drawn token at j = n_i, -1 after. */
typedef struct sv_sample_args {
  int32_t batch;            /* B >= 0 (must equal the attention's B in a step) */
  int32_t vocab;            /* V >= 1 */
  int32_t dtype;            /* sv_dtype of both logits tensors */
  int32_t max_q_rows;       /* host bound on R_i, 1..16 */
  int64_t num_rows;         /* R = cu_q[B] (host copy) */
  float temperature;        /* >= 0; 0 = greedy */
  float top_p;              /* (0, 1]; >= 1 disables the nucleus */
  uint64_t seed;            /* Philox key */
  const int32_t *cu_q;      /* [dev] [B+1] */
  const void *target_logits;/* [dev] [R, V] */
  const void *draft_logits; /* [dev] [R - B, V] */
  const int32_t *draft_tokens; /* [dev] [R - B] */
  const int32_t *kv_len;    /* [dev] [B] L_i: row j decides token L_i + j + 1 */
  const int64_t *seq_ids;   /* [dev] [B] Philox sequence ids; NULL -> i */
  int32_t *num_accepted;    /* [dev] [B] out */
  int32_t *out_tokens;      /* [dev] [R] out */
  uint32_t *dev_status;     /* [dev] one word */
  /* Added in ABI 2.  Processing order: temperature, top-k, top-p (the
   * speculative-sampling paper, section "Modified rejection sampling": such
   * transforms change q and p before the scheme).  temperature 0 is greedy:
   * q and p become one-hot at the first (lowest-index) maximum, so a draft is
   * kept iff it is the target row's argmax.  top_k > 0 keeps the tokens whose
   * logit is at least the k-th largest (ties at the boundary kept); top-p then
   * applies to the renormalized top-k distribution. */
  int32_t top_k;            /* >= 0; 0 disables */
  const float *temperatures;/* [dev] [B] per-sequence temperature or NULL */
  const float *top_ps;      /* [dev] [B] per-sequence top_p or NULL */
  const int32_t *top_ks;    /* [dev] [B] per-sequence top_k or NULL */
} sv_sample_args;

/* Workspace bytes for an attention call, a sampling call, or (both
 * non-NULL) a fused step.  Returns 0 if the arguments are invalid. */
SV_API size_t sv_workspace_bytes(const sv_attn_args *attn, const sv_sample_args *sample);

/* Zero a workspace once before its first use (cudaMemsetAsync on stream). */
SV_API sv_status sv_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Verify attention only: writes attn->out. */
SV_API sv_status spec_verify_attn(const sv_attn_args *attn, void *ws, size_t ws_bytes,
                                  void *stream);

/* Bytes of the static scratch array behind spec_verify_attn_static. */
#define SV_STATIC_SCRATCH_BYTES (16u << 20)

/* spec_verify_attn without a caller workspace, allocating nothing.  The
 * speculative-sampling and verify-attention papers have no counterpart of
 * this call: it serves callers that may not allocate device memory when they
 * call (an embedder whose device memory belongs to another allocator, a
 * serving runtime that forbids allocation once it has started) and so cannot
 * supply the workspace spec_verify_attn takes.  The split-KV partials and
 * merge counters live instead in a fixed SV_STATIC_SCRATCH_BYTES array inside
 * the library's device image, one per device, held until the process exits.
 *   - Setup: the first call in a CUDA context (the current one: normally a
 *     device's primary context) looks the array up and clears it to zero,
 *     synchronizing the device; make that first call before any stream
 *     capture and outside code that must not synchronize.  Later calls in
 *     that context only launch kernels on `stream`.  The looked-up address is
 *     kept per context, so a context made after cudaDeviceReset (or one that
 *     a driver-API caller created) gets its own lookup and clearing.
 *   - Limits: the first 64 KiB hold only the merge counters (batch *
 *     num_kv_heads <= 16384); the scratch of the call
 *     (sv_workspace_bytes(attn, NULL)) plus those 64 KiB must fit in
 *     SV_STATIC_SCRATCH_BYTES.  A call beyond either limit returns
 *     SV_ERR_WORKSPACE and launches nothing.
 *   - Zero state: the merge counters must be zero when a call starts; setup
 *     zeroes them and every call that runs to completion leaves them zero.
 *     A call that ends with SV_DEV_TIMEOUT in *dev_status can leave counts
 *     behind: call sv_static_scratch_reset before the next static call.
 *   - Concurrency: all calls in one context share the array, so calls that
 *     can overlap on the GPU (other streams, other host threads without
 *     ordering) race and corrupt each other's partials; order them on one
 *     stream.
 * Results are those of spec_verify_attn on the same arguments (same kernels,
 * same merge order: equal bits). */
SV_API sv_status spec_verify_attn_static(const sv_attn_args *attn, void *stream);

/* Zero the merge counters of the static array (64 KiB, cudaMemsetAsync on
 * `stream`; allocates nothing; the first call in a context also runs the setup
 * described above).  Needed only after a static call reported SV_DEV_TIMEOUT;
 * like spec_verify_attn_static it has no counterpart in the papers. */
SV_API sv_status sv_static_scratch_reset(void *stream);

/* Rejection sampling only: writes num_accepted and out_tokens. */
SV_API sv_status spec_reject_sample(const sv_sample_args *sample, void *ws, size_t ws_bytes,
                                    void *stream);

/* Ragged append of accepted rows (a6).  dtype SV_F32, SV_BF16 or SV_E4M3
 * (one byte per element: an 8-bit cache).  For every sequence with
 * num_accepted[i] = n >= 0 and kv_len[i] + n + 1 <= kv_cap[i]: copies block
 * rows cu_q[i] .. cu_q[i] + n of k_new / v_new to pool rows kv_start[i] +
 * kv_len[i] .. + n, and writes new_kv_len[i] = kv_len[i] + n + 1; otherwise
 * new_kv_len[i] = kv_len[i] (with SV_DEV_CAPACITY on overflow).  Layouts as
 * in sv_attn_args.  new_kv_len must not alias kv_len. */
SV_API sv_status kv_append_ragged(int32_t batch, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t dtype, int32_t max_q_rows, int64_t num_rows,
                                  const int32_t *cu_q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, int64_t pool_rows,
                                  const int64_t *kv_start, const int32_t *kv_len,
                                  const int32_t *kv_cap, const int32_t *num_accepted,
                                  int32_t *new_kv_len, uint32_t *dev_status, void *stream);

/* The fused verify step: attention, rejection sampling and the append of the
 * accepted rows, on one stream with no host synchronization.  attn and sample
 * must describe the same batch (same cu_q and kv_len pointers).  kv_cap [dev]
 * [B]; new_kv_len [dev] [B] out (must not alias kv_len).  The append writes
 * only pool rows at or beyond kv_len[i], which the attention does not read. */
SV_API sv_status spec_verify_step(const sv_attn_args *attn, const sv_sample_args *sample,
                                  const int32_t *kv_cap, int32_t *new_kv_len, void *ws,
                                  size_t ws_bytes, void *stream);

/* Draft-token draw (added in ABI 3): the sampling half of one draft
 * position of the speculative-sampling loop.  The speculative-sampling
 * paper's algorithm has the draft model propose its K tokens one at a time,
 * each drawn from the draft distribution given the context and the drafts so
 * far; by section "Modified rejection sampling" (compatibility with standard
 * sampling methods) the draw is from the processed draft row p_hat
 * (temperature, top-k, top-p as in sv_sample_args), the same p_hat the verify
 * step's accept rule uses.  The draft model's single-row attention and the
 * append of its row are spec_verify_attn and kv_append_ragged with one block
 * row per sequence (cu_q = 0..B, num_accepted all 0).
 *
 * For sequence i the token drawn from row i sits at index kv_len[i] + 1
 * (kv_len[i] = the draft cache's length before this position's append): the
 * inverse CDF of p_hat in vocabulary order (first x whose cumulative weight
 * exceeds u * Z) with u = word 1 of Philox4x32-10 at counter (kv_len[i] + 1,
 * seq_ids[i], stream 1) under key seed, so draft draws never reuse a verify
 * step uniform (stream 0).  A sequence whose row holds NaN or +inf, or only
 * -inf, or whose per-sequence parameter is invalid gets draft_tokens[i] = -1
 * with SV_DEV_NONFINITE (plus SV_DEV_BAD_PARAM for a parameter). */
typedef struct sv_draft_args {
  int32_t batch;            /* B >= 0 */
  int32_t vocab;            /* V >= 1 */
  int32_t dtype;            /* sv_dtype of draft_logits */
  int32_t top_k;            /* >= 0; 0 disables */
  float temperature;        /* >= 0; 0 = greedy (first argmax) */
  float top_p;              /* (0, 1]; >= 1 disables the nucleus */
  uint64_t seed;            /* Philox key (the verify step's seed) */
  const void *draft_logits; /* [dev] [B, V] one row per sequence */
  const int32_t *kv_len;    /* [dev] [B] cache length before this position's append */
  const int64_t *seq_ids;   /* [dev] [B] Philox sequence ids; NULL -> i */
  const float *temperatures;/* [dev] [B] per-sequence temperature or NULL */
  const float *top_ps;      /* [dev] [B] per-sequence top_p or NULL */
  const int32_t *top_ks;    /* [dev] [B] per-sequence top_k or NULL */
  int32_t *draft_tokens;    /* [dev] [B] out */
  uint32_t *dev_status;     /* [dev] one word */
} sv_draft_args;

/* Workspace bytes of spec_draft_sample (0 if the arguments are invalid).  The
 * workspace follows the same rule as the others: zeroed once before first use
 * (sv_workspace_init), left zero by every call that runs to completion. */
SV_API size_t sv_draft_workspace_bytes(const sv_draft_args *draft);

/* Draws draft_tokens (asynchronous on stream; host-checkable problems return
 * SV_ERR_* and launch nothing). */
SV_API sv_status spec_draft_sample(const sv_draft_args *draft, void *ws, size_t ws_bytes,
                                   void *stream);

/* Bound on the polls of one internal wait of the attention pipeline (an
 * mbarrier of the copy ring, of a Q slot, of the consumer group or of the
 * merge hand-off), for every attention launch that starts after the call in
 * this process; 0 restores the built-in bound (2^22 polls).  A wait that runs
 * out sets SV_DEV_TIMEOUT in *dev_status; its CTA stops, drains the copies
 * it started (that drain always keeps the built-in bound) and leaves, so the
 * outputs it owned stay unwritten and the workspace's merge counters may be
 * left nonzero: zero the workspace again (sv_workspace_init, or
 * sv_static_scratch_reset for spec_verify_attn_static) before its next use.
 * A small bound makes waits run out on purpose; this exists to exercise that
 * path (the papers have no counterpart).  Not synchronized with launches in
 * flight on other host threads. */
SV_API sv_status sv_set_wait_limit(uint32_t polls);

/* One whole draft position (added in ABI 5): the draft model's single-row
 * attention (spec_verify_attn with one block row per sequence: cu_q = 0..B,
 * max_q_rows 1, num_rows B), the append of the position's own K/V row, and
 * the draft-token draw of spec_draft_sample, as one call.  The speculative-
 * sampling paper's algorithm draws the K drafts one position at a time; the
 * draw reads only the draft logits (inputs here), so it and the append start
 * beside the attention (programmatic dependent launch) instead of after it.
 * attn and draft must describe the same batch (same B, kv_len pointer and
 * dtype).  Writes attn->out, draft->draft_tokens, the pool row kv_start[i] +
 * kv_len[i] and new_kv_len[i] = kv_len[i] + 1 (kv_len[i] with
 * SV_DEV_CAPACITY when kv_len[i] + 1 > kv_cap[i]; new_kv_len must not alias
 * kv_len).  Same results as the three separate calls.  Workspace:
 * sv_draft_step_workspace_bytes, zeroed once like the others. */
SV_API size_t sv_draft_step_workspace_bytes(const sv_attn_args *attn, const sv_draft_args *draft);
SV_API sv_status spec_draft_step(const sv_attn_args *attn, const sv_draft_args *draft,
                                 const int32_t *kv_cap, int32_t *new_kv_len, void *ws,
                                 size_t ws_bytes, void *stream);

/* Thread-local description of the last non-OK status returned on this
 * thread ("" if none). */
SV_API const char *sv_last_error(void);

/* SV_ABI_VERSION of the loaded library. */
SV_API int32_t sv_abi_version(void);

/* sizeof(sv_attn_args) for which = 0, sizeof(sv_sample_args) for which = 1,
 * sizeof(sv_draft_args) for which = 2 (lets a binding check its struct
 * mirrors). */
SV_API size_t sv_struct_size(int32_t which);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
