/*
 * peagle.h -- C ABI of the GB300 (sm_103a) P-EAGLE parallel draft pass.
 *
 * One library call runs one step of the speculative round described in
 *   "P-EAGLE: A Technical Deep Dive into Parallel Speculative Decoding",
 *   section "2. The P-EAGLE Parallel Drafter", and
 *   "P-EAGLE: Parallel-Drafting EAGLE with Scalable Training", A2 section 2:
 * from the target's captured hidden states and the newly generated token, ONE forward
 * pass of an N-layer Llama-3 drafter produces all K draft tokens; the target then
 * verifies them and keeps the longest agreeing prefix plus a bonus token
 * ("EAGLE-4", section "EAGLE-4 overview").
 *
 * Conventions shared by every call
 *   - Sizes are int32; pointers are plain pointers.  "device" means a CUDA device
 *     pointer on the current device; "host or device" means any pointer that
 *     cudaMemcpy with cudaMemcpyDefault accepts (pageable/pinned host or device).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Every call except peagle_create, peagle_status and peagle_destroy is
 *     asynchronous on `stream`, performs no allocation and no host synchronisation,
 *     and may be captured into a CUDA graph.
 *   - Return value: PEAGLE_OK or a negative error code.  Host-detectable argument
 *     errors are returned immediately and nothing is launched.  Errors that depend on
 *     device-resident values (token ids, seq_lens) are latched in the context's
 *     device error word by the kernels, which then skip the offending access; the
 *     next peagle_status() reports them.  No call aborts, exits or traps.
 *   - dtype: PEAGLE_F32 keeps every tensor (weights, caches, activations) in fp32
 *     and computes with fp32 FMA; PEAGLE_BF16 stores weights, caches and
 *     activations in bf16 and accumulates in fp32 on the tensor cores.
 */
#ifndef PEAGLE_H
#define PEAGLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PEAGLE_OK 0
#define PEAGLE_ERR_INVALID (-1)      /* bad pointer / size / argument combination  */
#define PEAGLE_ERR_UNSUPPORTED (-2)  /* dims outside what the kernels implement     */
#define PEAGLE_ERR_CAPACITY (-3)     /* batch, K, rows or KV capacity beyond limits */
#define PEAGLE_ERR_CUDA (-4)         /* a CUDA runtime/driver call failed           */
#define PEAGLE_ERR_DEVICE (-5)       /* a device-side check tripped (see status)    */

/* Device error word bits (peagle_status() returns PEAGLE_ERR_DEVICE if any is set;
 * peagle_device_error_bits() returns the raw bits of the last status call). */
#define PEAGLE_DEV_BAD_TOKEN 0x1     /* token id outside [0, target_vocab)          */
#define PEAGLE_DEV_KV_OVERFLOW 0x2   /* seq_lens[b] + K (or + n_commit) > capacity  */
#define PEAGLE_DEV_BAD_COMMIT 0x4    /* n_commit[b] outside [0, n_max]              */
#define PEAGLE_DEV_BAD_ROW 0x8       /* forward_parallel row (p, d) invalid         */
#define PEAGLE_DEV_TIMEOUT 0x10      /* a bounded on-chip wait gave up              */

typedef enum { PEAGLE_F32 = 0, PEAGLE_BF16 = 1 } peagle_dtype;

typedef struct peagle_ctx peagle_ctx;

/* Drafter dimensions.  Constraints (else PEAGLE_ERR_UNSUPPORTED):
 *   head_dim in {64, 128}; n_q_heads % n_kv_heads == 0; hidden % 64 == 0, <= 16384;
 *   intermediate % 64 == 0; (n_q_heads + 2 n_kv_heads) * head_dim % 128 == 0;
 *   max_batch * max_K <= 256; max_K <= 16; max_K * (n_q_heads / n_kv_heads) <= 128;
 *   n_q_heads / n_kv_heads <= 64 when max_rows > 0. */
typedef struct peagle_dims {
  int32_t hidden;        /* H                                                     */
  int32_t n_layers;      /* N decoder layers                                      */
  int32_t n_q_heads;     /* nq                                                    */
  int32_t n_kv_heads;    /* nkv (GQA: q head h reads kv head h / (nq / nkv))       */
  int32_t head_dim;      /* hd                                                    */
  int32_t intermediate;  /* I (SwiGLU)                                            */
  int32_t draft_vocab;   /* Vd rows of the LM head                                */
  int32_t target_vocab;  /* Vt rows of the embedding table; d2t maps into it      */
  int32_t max_batch;     /* largest `batch` any draft call will use               */
  int32_t max_K;         /* largest K any draft call will use                     */
  int32_t max_rows;      /* largest M of peagle_forward_parallel (0: not used)    */
  int32_t max_seq;       /* largest n of peagle_forward_parallel (0: not used)    */
  int32_t max_positions; /* RoPE table size: every position used must be below it */
  int32_t dtype;         /* peagle_dtype                                          */
  float rope_theta;      /* RoPE base                                             */
  float rms_eps;         /* RMSNorm epsilon                                       */
  int32_t attn_window;   /* sliding-window drafter attention ("EAGLE-4", section
                            "EAGLE-4 overview"): a draft-block row at position pos
                            sees only the keys at positions pos - attn_window + 1
                            .. pos.  0 = the whole context.  Draft and catch-up
                            passes only; peagle_forward_parallel rejects a window
                            with PEAGLE_ERR_UNSUPPORTED.                         */
  int32_t lm_rank;       /* efficient LM head ("EAGLE-4", "EAGLE-4 overview": a
                            rank-128 projection scores the whole vocabulary, the
                            full head scores only the best candidates): 0 = the
                            full head; else 64, 128, 256 or 512, with weights
                            lm_proj / lm_score, hidden <= 12288 and a draft
                            vocabulary of at most 2^24 entries.  Draft and
                            catch-up passes only (peagle_forward_parallel:
                            UNSUPPORTED).                                         */
  int32_t lm_topk;       /* candidates the full head scores (1 .. 1024; more than
                            the draft vocabulary means all of it).  With the
                            efficient head, out_logits holds the exact logits of
                            the candidates and -inf elsewhere.                   */
  int32_t train;         /* 1: peagle_create also makes the training step's
                            workspaces for max_rows rows and max_seq positions
                            (needs max_rows > 0, neither attn_window nor lm_rank);
                            0: peagle_train_step returns PEAGLE_ERR_CAPACITY.    */
} peagle_dims;

/* Drafter weights (host or device pointers; dtype = dims.dtype for every float
 * tensor).  nn.Linear layout [out, in], row-major.  Per-layer entries are host
 * arrays of n_layers pointers.  peagle_create copies (and repacks) everything into
 * library-owned device memory, so the caller may free these buffers afterwards. */
typedef struct peagle_weights {
  const void* embed;             /* [Vt, H] token embeddings                        */
  const void* emb_mask;          /* [H]     learnable emb(mask)                     */
  const void* h_shared;          /* [3H]    learnable shared hidden state           */
  const void* fc;                /* [H, 3H] projection of the 3 target states       */
  const void* input_norm;        /* [H]     RMSNorm gain of the embedding half      */
  const void* hidden_norm;       /* [H]     RMSNorm gain of the fc half             */
  const void* const* qkv;        /* N x [(nq+2nkv)hd, 2H (layer 0) | H]             */
  const void* const* o;          /* N x [H, nq hd]                                  */
  const void* const* attn_norm;  /* N x [H] (entry 0 unused, may be NULL)           */
  const void* const* post_norm;  /* N x [H]                                         */
  const void* const* gate;       /* N x [I, H]                                      */
  const void* const* up;         /* N x [I, H]                                      */
  const void* const* down;       /* N x [H, I]                                      */
  const void* final_norm;        /* [H]                                             */
  const void* lm_head;           /* [Vd, H]                                         */
  const int32_t* d2t;            /* [Vd] draft->target offsets: id = i + d2t[i]     */
  /* Efficient LM head ("EAGLE-4", "EAGLE-4 overview"), used when dims.lm_rank > 0,
   * else ignored (may be NULL): */
  const void* lm_proj;           /* [rank, H]  projection of the LM-head input        */
  const void* lm_score;          /* [Vd, rank] scores of the projected input           */
} peagle_weights;

/* Caller-owned drafter KV cache (device).  Layout of k and v:
 *   [n_layers][batch][n_kv_heads][capacity][head_dim], dtype = dims.dtype.
 * Keys are stored after RoPE.  Request b's committed entries are slots
 * 0 .. seq_lens[b]-1. */
typedef struct peagle_kv {
  void* k;
  void* v;
  int32_t capacity; /* slots per (layer, request, kv head)                          */
  int32_t batch;    /* request slots in the buffers (>= the call's batch)           */
} peagle_kv;

/* Create a drafter context ("P-EAGLE: A Technical Deep Dive into Parallel Speculative
 * Decoding", section "2. The P-EAGLE Parallel Drafter": the drafter's weights, including
 * the learnable emb(mask) and h_shared that every MTP position shares, are fixed for the
 * whole deployment; "Speeding LLM inference with P-EAGLE in vLLM/Speculators", section
 * "A learnable mask parameter": h_shared is 3H wide).  Validates dims, allocates all
 * device memory the other calls need (weights, workspaces sized for max_batch x max_K
 * rows and max_rows; with dims.train, also the training step's fp32 weight copies,
 * kept activations and gradient scratch), copies
 * and repacks the weights, precomputes fc(h_shared) (a constant of the weights) and the
 * RoPE table, and synchronises.  The only allocating call of a drafter context.  *out is
 * NULL on failure (PEAGLE_ERR_CUDA when device memory runs out). */
int peagle_create(const peagle_weights* w, const peagle_dims* dims, peagle_ctx** out);

/* One parallel draft pass ("2. The P-EAGLE Parallel Drafter").
 *   batch            requests, 1 .. max_batch (and <= kv->batch)
 *   kv               drafter cache; the pass WRITES row j's key/value of every layer
 *                    into slot seq_lens[b] + j (uncommitted until peagle_append_kv)
 *   seq_lens         device int32 [batch]: committed KV length of each request
 *   target_hidden    device [batch, 3H] (dims dtype): the target's three captured
 *                    hidden states, concatenated early | mid | late
 *   new_token        device int32 [batch]: the newly generated token (target vocab)
 *   K                draft depth, 1 .. max_K; rows r = b*K + j, j = 0 is the NTP row
 *   out_draft_tokens device int32 [batch, K]: argmax over the draft vocabulary
 *                    (lowest index on ties) mapped to the target vocabulary by d2t
 *   out_logits       device fp32 [batch, K, Vd], or NULL to skip writing logits
 * Device checks: new_token in range (else BAD_TOKEN, row treated as token 0);
 * seq_lens[b] + K <= capacity (else KV_OVERFLOW, out-of-range slots skipped). */
int peagle_draft(peagle_ctx* ctx, int32_t batch, const peagle_kv* kv, const int32_t* seq_lens,
                 const void* target_hidden, const int32_t* new_token, int32_t K,
                 int32_t* out_draft_tokens, float* out_logits, void* stream);

/* Drafter catch-up ("P-EAGLE: A Technical Deep Dive into Parallel Speculative Decoding",
 * section "Technical Architecture", stage 1 of a round): the T tokens a request accepted
 * (and their captured target hidden states) run through the drafter as depth-1 rows --
 * row t takes embed[tokens[b, t]] and fc(hidden[b, t]) at position seq_lens[b] + t and
 * attends to the cached context and rows 0..t ("Speeding LLM inference with P-EAGLE in
 * vLLM/Speculators", "Flex-attention mask": depth-1 rows are causal among themselves) --
 * and their keys and values are written to cache slots seq_lens[b] + t.  seq_lens is not
 * advanced: commit with peagle_append_kv (k_rows = NULL, n_commit = T).
 *   hidden    device [batch, T, 3H] (dims dtype); tokens device int32 [batch, T]
 *   out_tokens device int32 [batch, T] (greedy next token of each row, target vocab) or
 *   NULL; out_logits fp32 [batch, T, Vd] or NULL; with both NULL the final norm and the
 *   LM head are skipped.
 * Constraints and device checks as for peagle_draft (T plays K). */
int peagle_catch_up(peagle_ctx* ctx, int32_t batch, const peagle_kv* kv,
                    const int32_t* seq_lens, const void* hidden, const int32_t* tokens,
                    int32_t T, int32_t* out_tokens, float* out_logits, void* stream);

/* Greedy verification ("EAGLE-4 overview"): for each request, the longest prefix of
 * draft_tokens[b, :] equal to target_argmax[b, :], plus one bonus token.
 *   draft_tokens   device int32 [batch, K]
 *   target_argmax  device int32 [batch, K+1]: the target's greedy choice after each
 *                  draft prefix (position K = after all K drafts)
 *   out_accept_len device int32 [batch]: m in 0..K (tokens emitted = m + 1)
 *   out_bonus      device int32 [batch]: target_argmax[b, m]
 * Needs no context; 1 <= K <= 64. */
int peagle_verify_greedy(int32_t batch, int32_t K, const int32_t* draft_tokens,
                         const int32_t* target_argmax, int32_t* out_accept_len,
                         int32_t* out_bonus, void* stream);

/* Commit accepted rows to the drafter's KV cache ("P-EAGLE: A Technical Deep Dive into
 * Parallel Speculative Decoding", section "Technical Architecture": each speculative round
 * ends with the accepted tokens' keys and values entering the drafter's cache, so the next
 * draft pass attends to them; "EAGLE-4", "EAGLE-4 overview": the accepted prefix plus
 * the bonus token are what a round emits) and advance seq_lens (device, in place):
 *   n_commit device int32 [batch]; request b commits n = n_commit[b] + n_extra rows
 *     (e.g. out_accept_len of peagle_verify_greedy with n_extra = 1: the NTP row and
 *     the accepted drafts, without a round trip to the host).
 *   k_rows/v_rows NULL: the first n (0..max_K) draft-block rows already sit in slots
 *     seq_lens[b] .. (written by peagle_draft); only seq_lens advances, n_max ignored.
 *   otherwise device [n_layers][batch][n_max][n_kv_heads][head_dim] (dims dtype)
 *     rows copied into slots seq_lens[b] + i, i < n (0..n_max).
 * Device checks: n_commit range (BAD_COMMIT), capacity (KV_OVERFLOW); a request
 * that fails a check is left unchanged. */
int peagle_append_kv(peagle_ctx* ctx, int32_t batch, const peagle_kv* kv, int32_t* seq_lens,
                     const int32_t* n_commit, int32_t n_extra, const void* k_rows,
                     const void* v_rows, int32_t n_max, void* stream);

/* Training-style parallel-prediction forward ("P-EAGLE: Parallel-Drafting EAGLE with
 * Scalable Training", sections 3.1-3.2; "Speeding LLM inference with P-EAGLE in
 * vLLM/Speculators", section "Flex-attention mask") over M retained rows (p, d),
 * depths 1-based, sorted p-major (by p, then d).  Row (p, 1) takes
 * embed[tokens[p]] and fc(hidden[p]); row (p, d >= 2) takes emb(mask) and
 * fc(h_shared).  RoPE position p.  Row (p, d) attends depth-1 rows p' <= p - d + 1,
 * its chain (p - j, d - j), j = 1 .. d-1, and itself.  The row set must be closed under
 * these dependencies: (p-1, d-1) present for every row with d >= 2, and (p-1, 1) for
 * every depth-1 row with p >= 1 (COD sampling, a prefix p < P0 and a dependency closure
 * all are); a row outside the contract sets BAD_ROW and its outputs are unspecified.
 *   n, K      sequence length (<= max_seq) and depth (<= 16)
 *   tokens    device int32 [n]; hidden device [n, 3H] (dims dtype)
 *   row_p, row_d device int32 [M]; M <= max_rows
 *   out_argmax device int32 [M] draft-vocab argmax (no d2t); out_logits fp32 [M, Vd]
 *   or NULL.  Device checks: BAD_ROW for rows outside the contract. */
int peagle_forward_parallel(peagle_ctx* ctx, int32_t n, int32_t K, const int32_t* tokens,
                            const void* hidden, const int32_t* row_p, const int32_t* row_d,
                            int32_t M, int32_t* out_argmax, float* out_logits, void* stream);

/* Gradients written by peagle_train_step: fp32 device buffers shaped like the weights of
 * peagle_weights (gate and up separate, [I, H] each), owned by the caller and overwritten
 * by the call.  Per-layer entries are host arrays of n_layers device pointers.  embed
 * ([Vt, H]) and attn_norm (and any of its entries) may be NULL: those gradients are then
 * skipped (attn_norm[0] is written as zeros: layer 1 reads the 2H input, not a norm of
 * the residual). */
typedef struct peagle_grads {
  float* embed;
  float* emb_mask;
  float* h_shared;
  float* fc;
  float* input_norm;
  float* hidden_norm;
  float* const* qkv;
  float* const* o;
  float* const* attn_norm;
  float* const* post_norm;
  float* const* gate;
  float* const* up;
  float* const* down;
  float* final_norm;
  float* lm_head;
} peagle_grads;

/* One training step without optimizer ("P-EAGLE: Parallel-Drafting EAGLE with Scalable
 * Training", A2 section 2 and section 3): the training-style forward of
 * peagle_forward_parallel over the rows (row_p, row_d) -- same arguments and the same row
 * contract -- then loss = the mean over the M rows of the cross-entropy of the row's
 * draft-vocabulary logits against labels[i] (device int32 [M], in [0, Vd)), and the
 * gradient of the loss with respect to every parameter into `grads`.
 *   out_loss  device fp32 scalar.
 * Arithmetic: fp32 activations; the projections and the attention's depth-1 products
 * run on the library's own GEMM kernels: TF32 tcgen05 tensor-core MMAs with fp32
 * accumulation for bf16 drafters, fp32 FMA tiles for fp32 drafters; for bf16 drafters
 * with head_dim 64 the whole depth-1 attention (forward and backward) is one fused TF32
 * tensor-core kernel per step, otherwise the dense [G M][n] prefix scores are formed.
 * Needs a context made with dims.train = 1: peagle_create then makes every workspace of
 * the step (fp32 weight copies for bf16 drafters, every layer's kept activations, the
 * GEMMs' scratch operands), so the call allocates nothing.  UNSUPPORTED with attn_window or lm_rank set.
 * Device checks: BAD_ROW for rows outside the contract, BAD_TOKEN for tokens or labels
 * out of range, TIMEOUT if a GEMM's bounded pipeline wait ran out. */
int peagle_train_step(peagle_ctx* ctx, int32_t n, int32_t K, const int32_t* tokens,
                      const void* hidden, const int32_t* row_p, const int32_t* row_d, int32_t M,
                      const int32_t* labels, float* out_loss, const peagle_grads* grads,
                      void* stream);

/* Host-side COD sampling ("COD sampling"; 3.2): depth 1 keeps every position; row
 * (p, d >= 2) exists when p - d + 1 >= 0 and is kept when its dependency (p-1, d-1)
 * was kept and uniforms[p*K + d-1] < ratio.  Writes the retained rows p-major into
 * out_p/out_d (host int32, capacity max_out) and returns their count, or a negative
 * error (PEAGLE_ERR_CAPACITY if max_out is too small). */
int peagle_cod_rows(int32_t n, int32_t K, double ratio, const double* uniforms,
                    int32_t* out_p, int32_t* out_d, int32_t max_out);

/* Host-side sequence partitioning ("P-EAGLE: Parallel-Drafting EAGLE with Scalable
 * Training", section 3.2): assigns each retained row (p, d), given p-major in
 * row_p / row_d (host int32 [M]), to one of n_chunks chunks whose start positions are
 * boundaries[0] = 0 < boundaries[1] < ... (host int32).  Rows of depth 1 and 2 go to the
 * chunk containing their position; a row of depth d >= 3 to the chunk of (p-1, d-1).
 * Writes out_chunk (host int32 [M]).  Chunk c's forward runs on its own rows plus every
 * depth-1 row below its end boundary (a dependency-closed set: one
 * peagle_forward_parallel call).  Returns PEAGLE_OK, or PEAGLE_ERR_INVALID for
 * non-increasing boundaries, rows not p-major, depth > 64 or a missing dependency. */
int peagle_sequence_partition(int32_t M, const int32_t* row_p, const int32_t* row_d,
                              int32_t n_chunks, const int32_t* boundaries, int32_t* out_chunk);

/* Synchronise the context's device work and return PEAGLE_OK, PEAGLE_ERR_DEVICE if
 * the device error word is non-zero (the word is then cleared; after a TIMEOUT the
 * context's accumulators are also reset), or PEAGLE_ERR_CUDA if a sticky CUDA error is
 * pending. */
int peagle_status(peagle_ctx* ctx);

/* Per-stage timing (diagnostics).  Stages of the pass: */
#define PEAGLE_STAGE_FC 0      /* fc projection of the target hidden states       */
#define PEAGLE_STAGE_QKV 1     /* QKV projection + RoPE + KV write                */
#define PEAGLE_STAGE_ATTN 2    /* attention (split-KV decode or masked)           */
#define PEAGLE_STAGE_OPROJ 3   /* o-projection + residual                         */
#define PEAGLE_STAGE_GATEUP 4  /* gate/up projection + SwiGLU                     */
#define PEAGLE_STAGE_DOWN 5    /* down projection + residual                      */
#define PEAGLE_STAGE_LMHEAD 6  /* LM head + argmax                                */
#define PEAGLE_STAGE_NORM 7    /* input fusion and RMSNorms                       */
#define PEAGLE_STAGE_SMALL 8   /* argmax decode, KV commit, row table             */
#define PEAGLE_NUM_STAGES 9

/* Enable (1) or disable (0) timing: while enabled, every kernel launch of peagle_draft,
 * peagle_append_kv and peagle_forward_parallel is bracketed by CUDA events recorded on
 * the call's stream (which serialises launches that would otherwise overlap).  The first
 * enable creates the event pool (up to 512 launches between reads); call it outside
 * stream capture. */
int peagle_set_timing(peagle_ctx* ctx, int32_t enable);

/* Wait for the recorded events, write the summed milliseconds and launch counts per
 * stage (arrays of PEAGLE_NUM_STAGES) since the previous read, and reset them. */
int peagle_read_timing(peagle_ctx* ctx, float* stage_ms, int32_t* stage_launches);

/* Diagnostics of the persistent pass kernel (the bf16 draft pass as one launch of one CTA
 * per SM; by default it runs passes of up to 16 draft rows, peagle_set_pass_kernel(ctx, 1)
 * uses it for every shape it supports and peagle_set_pass_kernel(ctx, 0) never).  For the
 * latest pass run while timing was enabled, writes four
 * globaltimer values (ns) per step of the pass and CTA, as out[(phase * ctas + cta) * 4 + k]:
 * projections: k = 0 the step's activations were seen ready, 1 its first MMA was issued,
 * 2 its last accumulator was committed; other steps: 0 the previous step was seen complete,
 * and for attention 1 the CTA's item wrote its partials, 2 every item of its (request, kv
 * head) was in (else 0); 3 the CTA finished the step; and
 * the two sizes.  Returns the number of entries (0 if no pass was traced),
 * PEAGLE_ERR_CAPACITY if max_entries is too small.  The paper has no counterpart: this
 * reports how this library schedules the pass. */
int32_t peagle_read_pass_trace(peagle_ctx* ctx, uint64_t* out, int32_t max_entries,
                               int32_t* out_phases, int32_t* out_ctas);

/* Failure-path drill of the bounded waits (diagnostics; the pages have no counterpart:
 * this tests how the library leaves a wait that cannot end).  Every wait of the persistent
 * pass kernel (step completions, ring stages, accumulators) gives up after limit_ns
 * nanoseconds (0 restores the default of 2 s); on expiry the kernel latches
 * PEAGLE_DEV_TIMEOUT, raises its abort flag so every CTA leaves its waits, lets the loads
 * and tensor-core operations it issued complete, frees its tensor memory and returns.
 * unreachable_step >= 0 names a step of the pass (its index in pass order: 0 the fc
 * projection, 1 the input rows, then per layer the norm (from the second layer on), the
 * QKV projection (two in the first layer, one per half of its input), attention,
 * o-projection, norm, gate/up, down; then the final norm, the LM head and the argmax)
 * whose waits require one completion signal more than the grid gives, so that they run
 * out; -1 none.  Applies to
 * the following draft and catch-up passes of this context.  peagle_status reports the
 * TIMEOUT bit and resets the context's accumulators, so the next pass starts clean.
 * Returns PEAGLE_ERR_INVALID for a step index outside the kernel's range. */
int peagle_set_wait_limit(peagle_ctx* ctx, uint64_t limit_ns, int32_t unreachable_step);

/* Which implementation runs the bf16 draft and catch-up passes.  Both compute the same
 * pass ("2. The P-EAGLE Parallel Drafter"); they differ in speed with the number of draft
 * rows R = batch x K.  mode -1 (the default): the persistent pass kernel (one launch per
 * pass, one CTA per SM) up to R = 16, separate kernel launches above; 0: always the
 * separate launches; 1: always the persistent kernel (up to its limits, R <= 120).
 * Returns PEAGLE_ERR_INVALID for another mode, PEAGLE_ERR_UNSUPPORTED for mode 1 on a
 * context without the persistent kernel (fp32 drafters, more than 8 layers, no
 * cooperative launch). */
int peagle_set_pass_kernel(peagle_ctx* ctx, int32_t mode);

/* Size of the library's static scratch array used by peagle_decode_attention_static. */
#define PEAGLE_STATIC_ATTN_SCRATCH_BYTES (8u << 20)

/* Decode attention for callers that cannot allocate device memory.  The pages have no
 * counterpart for this call: it exists for users of the library whose code may not call
 * cudaMalloc -- for example a process whose device memory is entirely handed out by its
 * own arena allocator, or code that may not make allocating CUDA calls at the point where
 * attention runs -- and who therefore cannot hold a peagle_ctx and its workspaces.
 *
 * It computes the draft pass's attention step for one layer: for request b, query row j
 * (rows b*K + j) and query head h, softmax(q . k / sqrt(head_dim)) . v over the cached
 * keys/values of kv head h / (n_q_heads / n_kv_heads) at slots 0 .. seq_lens[b] + j.
 *   q        device fp32 [batch*K][n_q_heads][head_dim] (keys are not rotated here: q and
 *            the cache are taken as already RoPE-rotated).  The kernel rounds each query
 *            element to bf16 (round to nearest even) before the score products, as the
 *            draft pass does; softmax and accumulation stay fp32.
 *   k_cache, v_cache  device bf16 [batch][n_kv_heads][capacity][head_dim] (one layer)
 *   seq_lens device int32 [batch]; keys at slots >= min(seq_lens[b] + K, capacity) unused
 *            (a row whose slot seq_lens[b] + j is at or beyond capacity sees the keys
 *            below capacity only); a request with seq_lens[b] < 0 is skipped and its
 *            output rows are left unwritten
 *   out      device fp32 [batch*K][n_q_heads][head_dim]
 * Limits: head_dim 64 or 128; K * n_q_heads / n_kv_heads <= 128; the split-KV partials,
 * batch * n_kv_heads * chunks * K * (n_q_heads/n_kv_heads) * (head_dim + 2) floats, must fit
 * PEAGLE_STATIC_ATTN_SCRATCH_BYTES (fewer, longer chunks are used when needed; a batch
 * too large for even one chunk is rejected with PEAGLE_ERR_CAPACITY and a message on
 * stderr).  No allocation and no host synchronisation.
 * The scratch is one array per GPU, shared by every call and keeping the last call's
 * contents (nothing in it needs to start at zero); calls that overlap on the GPU (other
 * streams, other threads) race on it, so order them on one stream.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) and sets kernel
 * attributes: make that first call before any stream capture. */
int peagle_decode_attention_static(int32_t batch, int32_t K, int32_t n_q_heads,
                                   int32_t n_kv_heads, int32_t head_dim, const float* q,
                                   const void* k_cache, const void* v_cache, int32_t capacity,
                                   const int32_t* seq_lens, float* out, void* stream);

/* Raw device error bits observed by the last peagle_status call. */
int32_t peagle_device_error_bits(const peagle_ctx* ctx);

/* Static description of an error code. */
const char* peagle_strerror(int code);

/* Free all device memory of the context (synchronises). NULL is ignored. */
void peagle_destroy(peagle_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* PEAGLE_H */
