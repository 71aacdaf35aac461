/*
 * spec.h -- C ABI of the GB300 verify-step library (libspec.so).
 *
 * The library runs the greedy, lossless speculative-decoding verify step of a
 * DeepSeekMoE-style (or dense SwiGLU) decoder on one GPU: one target forward
 * scores each sequence's last committed token plus K draft tokens against a
 * paged, prefix-shared KV cache, takes the greedy argmax of every row, keeps
 * the longest draft prefix that agrees with it, appends the target's bonus
 * token, and commits or rolls back the KV rows on the device.
 *
 * Sources for the operations (page title and section):
 *  - "End-to-end OCR expert model architecture and acceleration principles",
 *    section 6.1 (the target scores all draft positions in one teacher-forced
 *    forward; accept the agreeing prefix left to right, the target supplies
 *    the token at the first divergence) and section 7 (draft -> verify ->
 *    append loop); section 9 (continuous batching, KV-cache management).
 *  - "Jina-OCR-v1: efficient document parsing with speculative decoding and
 *    dense verifiable rewards", abstract (greedy verification is lossless),
 *    section 3 (compressed visual prefix, DeepSeekMoE decoder ~570M active).
 *  - "Jina AI releases jina-ocr-v1" (64 routed + 2 shared experts, top-6;
 *    greedy verification keeps the longest matching prefix).
 *  - "OCRia-1 technical report guide", inference stack (31-token block drafts,
 *    FP8 weights, shared prompt-prefix reuse).
 *
 * Conventions for every entry point:
 *  - Return 0 on success or a negative SPEC_ERR_* code; spec_strerror() names
 *    it and spec_last_error() gives a message for the last failure on the
 *    calling thread. No C++ exception crosses this boundary.
 *  - On failure the sequence state is unchanged (a verify step commits all of
 *    its sequences or none).
 *  - The caller owns every array it passes and may reuse it once the call
 *    returns. Arguments are host pointers unless the name ends in "_dev".
 *  - The library owns the weights, the KV page pool and its CUDA graphs. All
 *    device work is ordered on the stream given to spec_init_model. Calls
 *    without a "_dev" suffix return only after their results are in host
 *    memory; "_dev" calls only enqueue work.
 *  - A model handle is not thread-safe; distinct handles are independent.
 */
#ifndef SPEC_H_
#define SPEC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes ------------------------------------------------------- */
#define SPEC_OK            0
#define SPEC_ERR_ARG      -1   /* bad argument (id, size, token out of range) */
#define SPEC_ERR_NO_PAGES -2   /* KV page pool exhausted                       */
#define SPEC_ERR_CUDA     -3   /* a CUDA call failed (see spec_last_error)     */
#define SPEC_ERR_STATE    -4   /* call not valid in the sequence's state       */
#define SPEC_ERR_NOMEM    -5   /* host or device allocation failed             */
#define SPEC_ERR_UNSUPPORTED -6 /* configuration outside what the kernels take */

/* ---- storage dtypes ------------------------------------------------------ */
#define SPEC_F32  0   /* IEEE binary32                                         */
#define SPEC_BF16 1   /* bfloat16 (top half of binary32, round-to-nearest-even) */
#define SPEC_FP8  2   /* OCP E4M3 codes + one fp32 scale per output row        */
#define SPEC_NVFP4 3  /* E2M1 codes + E4M3 scale per 16 elements + fp32 scale  */
                      /* per matrix ("OCRia-1 technical report guide",          */
                      /* inference stack: NVFP4 weights)                        */

/* Model and pool shape. n_experts == 0 selects a dense SwiGLU FFN, stored as
 * one always-on ("shared") expert of width `inter` (n_shared must be 1).
 * Routed experts use top_k of n_experts, softmax weights without
 * renormalisation; shared experts are added with weight 1.
 * head_dim must be 64 or 128; page_size a multiple of 16; max_draft <= 31. */
typedef struct spec_config {
  int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim;
  int32_t n_experts, top_k, n_shared, inter, vocab;
  int32_t wdtype;        /* SPEC_F32 / SPEC_BF16 / SPEC_FP8 (attention + experts) */
  int32_t page_size;     /* tokens per KV page                                    */
  int32_t n_pages;       /* pages in the pool                                     */
  int32_t max_seqs;      /* sequence slots (ids 0..max_seqs-1)                    */
  int32_t max_ctx;       /* longest sequence (prompt + output + max_draft + 1)    */
  int32_t max_draft;     /* K: every verify step scores K+1 rows per sequence     */
  int32_t max_batch;     /* sequences per verify step                             */
  int32_t prefill_chunk; /* rows per prefill pass (0 = library default)           */
  float rope_theta, rms_eps;
} spec_config;

/* ---- weights ------------------------------------------------------------- */
/* Tensors are passed as an array of host pointers in this order (global, then
 * 13 per layer):
 *   0 tok_embed [V, h]          f32 if wdtype == F32, else bf16
 *   1 final_norm [h]            f32
 *   2 lm_head [V, h]            f32 if wdtype == F32, else bf16
 *   per layer l, index 3 + 13 l + j:
 *   j=0 attn_norm [h] f32       j=1 w_qkv [(Hq+2Hkv) d, h] wdtype (rows: q heads,
 *                                   then k heads, then v heads; each head d rows)
 *   j=2 s_qkv [(Hq+2Hkv) d] f32 (FP8) / [1] f32 (NVFP4)
 *   j=3 w_o [h, Hq d] wdtype    j=4 s_o [h] f32 (FP8) / [1] (NVFP4)
 *   j=5 ffn_norm [h] f32        j=6 w_router [E, h] (f32 if F32 model, else bf16;
 *                                   absent when E == 0)
 *   j=7 w_gate [E+S, inter, h]  j=8 s_gate [E+S, inter] f32 (FP8) / [E+S] (NVFP4)
 *   j=9 w_up [E+S, inter, h]    j=10 s_up [E+S, inter] f32 (FP8) / [E+S] (NVFP4)
 *   j=11 w_down [E+S, h, inter] j=12 s_down [E+S, h] f32 (FP8) / [E+S] (NVFP4)
 * Matrices are row-major [out, in]; experts 0..E-1 are routed, E..E+S-1
 * shared. Absent tensors have 0 bytes and their pointer may be NULL.
 * An NVFP4 matrix [rows, K] (each expert of a stack in turn) is one record:
 * its E2M1 codes, two per byte (element 2j of a row in the low nibble of
 * byte j), rows * K / 2 bytes, then its E4M3 block-scale codes [rows, K / 16];
 * value = e2m1 * e4m3(block scale) * the matrix's fp32 scale (the s_ tensor).
 * NVFP4 models take at most 8 rows per verify step (max_batch * (max_draft +
 * 1) <= 8), and hidden, inter and Hq * head_dim multiples of 128
 * (SPEC_ERR_UNSUPPORTED otherwise). */
int spec_tensor_count(const spec_config* cfg);
/* Byte size of tensor `index` (0 for absent ones), or a negative error. */
int64_t spec_tensor_bytes(const spec_config* cfg, int index);

typedef struct spec_model spec_model;

/* Validate `cfg`, allocate the device weights, KV pool and step buffers,
 * upload `host_tensors` (spec_tensor_count() pointers in the order above) and
 * build the RoPE tables. `cuda_stream` is a cudaStream_t; 0 makes the library
 * create and own a non-blocking stream (the legacy default stream cannot be
 * captured into the CUDA graphs the steps replay). Errors: SPEC_ERR_ARG (bad shape), SPEC_ERR_UNSUPPORTED,
 * SPEC_ERR_NOMEM, SPEC_ERR_CUDA. */
int spec_init_model(const spec_config* cfg, const void* const* host_tensors,
                    uintptr_t cuda_stream, spec_model** out_model);
int spec_free_model(spec_model* m);

/* Register a prompt prefix shared by many sequences (the OCRia-1 guide's
 * shared prompt-prefix reuse): its KV rows are computed once, and its full
 * pages are referenced (refcounted) by every sequence prefilled with it.
 * tok: n_tok host token ids. */
int spec_register_prefix(spec_model* m, const int32_t* tok, int n_tok,
                         int32_t* out_prefix_id);
int spec_release_prefix(spec_model* m, int32_t prefix_id);

/* Prefill sequence slot `seq_id` (must be free) with the prompt
 * [prefix tokens (prefix_id >= 0)] ++ vis_embeds_dev rows ++ tok. vis_embeds_dev
 * is a DEVICE pointer to n_vis rows of `hidden` values in the activation
 * storage type (f32 for F32 models, bf16 otherwise); tok are host ids.
 * Writes the first generated token (greedy argmax of the last prompt row).
 * Errors: SPEC_ERR_ARG, SPEC_ERR_STATE (slot busy), SPEC_ERR_NO_PAGES. */
int spec_prefill(spec_model* m, int32_t seq_id, int32_t prefix_id,
                 const void* vis_embeds_dev, int n_vis, const int32_t* tok, int n_tok,
                 int32_t* out_first_token);

/* One verify step for one sequence: scores [last committed token, draft_tokens
 * (n_draft of them, 0 <= n_draft <= max_draft)], then commits the accepted
 * prefix and the bonus token. n_draft = 0 is a plain greedy decoding step.
 * out_accepted_len = number of drafts accepted (0..n_draft); the step commits
 * out_accepted_len + 1 tokens: the accepted drafts then *out_bonus_token. */
int spec_verify_step(spec_model* m, int32_t seq_id, const int32_t* draft_tokens,
                     int n_draft, int32_t* out_accepted_len, int32_t* out_bonus_token);

/* Batched verify step over n_seq distinct sequences (1 <= n_seq <= max_batch).
 * drafts: [n_seq, max_draft] host ids (row s uses its first n_draft[s]).
 * Outputs out_accepted[n_seq], out_bonus[n_seq] (host). */
int spec_verify_step_batch(spec_model* m, int n_seq, const int32_t* seq_ids,
                           const int32_t* drafts, const int32_t* n_draft,
                           int32_t* out_accepted, int32_t* out_bonus);

/* Device-resident variant: all arrays are device pointers, nothing is copied
 * to or read back by the host and the call returns once the step is enqueued.
 * The sequences must have KV pages reserved for the step (spec_reserve_seq);
 * the host's view of their lengths is refreshed by spec_sync_seqs(). */
int spec_verify_step_batch_dev(spec_model* m, int n_seq, const int32_t* seq_ids_dev,
                               const int32_t* drafts_dev, const int32_t* n_draft_dev,
                               int32_t* out_accepted_dev, int32_t* out_bonus_dev);

/* Batched verify step with rejection-sampling acceptance instead of the greedy
 * rule ("End-to-end OCR expert model architecture and acceleration
 * principles", section 6.1 and section 11 item 2: the output keeps the target
 * model's own distribution). The drafter is taken as certain of its drafts
 * (q one-hot at each draft), which keeps the rule lossless for any drafter.
 * One captured graph: the decoder forward, the LM head, the rejection
 * sampler, then the device commit of what it decided. On the tensor-core
 * path (more than 8 rows a step), the LM head's epilogue leaves per-tile
 * softmax statistics (max, sum of exp) instead of logits. A one-block-per-
 * sequence sampler then draws from them and recomputes only the drawn tile's
 * 128 logits. Otherwise the LM head writes the step's logits into a
 * model-owned buffer and spec_rejection_sample_ws's cooperative kernel
 * samples them. With p_j the
 * softmax of row j-1 of the step's logits at `temperature`, for sequence s:
 *   accept d_j while u_accept[s][j-1] < p_j(d_j), j = 1..n_draft[s];
 *   at the first rejection append a draw from p_j without d_j (normalised)
 *   with u_sample[s][j-1]; if all are accepted append a draw from
 *   p_(n_draft+1) with u_sample[s][n_draft].
 * A draw is the inverse CDF in index order (see spec_rejection_sample).
 * Arguments as spec_verify_step_batch, plus:
 *   u_accept: [n_seq][max_draft] f32 uniforms in [0, 1) (may be NULL when
 *             max_draft = 0);
 *   u_sample: [n_seq][max_draft + 1] f32 uniforms in [0, 1);
 *   temperature > 0.
 * out_accepted[s] drafts accepted, then out_token[s] appended: the step commits
 * out_accepted[s] + 1 tokens, like a greedy step. The first sampled call
 * allocates the statistics (max_batch x (max_draft + 1) x vocab / 128 x 16
 * bytes) or the logits buffer (max_batch x (max_draft + 1) x vocab f32) and
 * the sampler's workspace. Needs vocab % 4 == 0 and vocab <= 262144.
 * Errors: as spec_verify_step_batch; SPEC_ERR_UNSUPPORTED for the vocabulary;
 * SPEC_ERR_CUDA when the cooperative launch cannot be made. */
int spec_verify_step_sample_batch(spec_model* m, int n_seq, const int32_t* seq_ids,
                                  const int32_t* drafts, const int32_t* n_draft,
                                  const float* u_accept, const float* u_sample, float temperature,
                                  int32_t* out_accepted, int32_t* out_token);
/* Device-resident variant (every array a device pointer; see
 * spec_verify_step_batch_dev). A sequence whose draft is not a token
 * reports (-1, -1) and is not committed; the step then raises the token error
 * bit, read back by spec_sync_seqs. */
int spec_verify_step_sample_dev(spec_model* m, int n_seq, const int32_t* seq_ids_dev,
                                const int32_t* drafts_dev, const int32_t* n_draft_dev,
                                const float* u_accept_dev, const float* u_sample_dev, float temperature,
                                int32_t* out_accepted_dev, int32_t* out_token_dev);

/* Reserve KV pages so sequence `seq_id` can grow to n_tokens positions without
 * host involvement; the commit kernel keeps these pages. */
int spec_reserve_seq(spec_model* m, int32_t seq_id, int n_tokens);
/* Wait for the stream, then read back every sequence's length and block table
 * into the host allocator's view. */
int spec_sync_seqs(spec_model* m);

/* Release sequence slot `seq_id`: its pages return to the pool (shared prefix
 * pages only when their last reference goes). */
int spec_release_seq(spec_model* m, int32_t seq_id);

/* Sequence state queries (host view; call spec_sync_seqs after _dev steps).
 * out_len = KV positions held (prompt + committed tokens - 1);
 * generated tokens so far are copied to out_tokens (up to cap). */
int spec_seq_info(spec_model* m, int32_t seq_id, int32_t* out_len, int32_t* out_n_generated);
int spec_seq_tokens(spec_model* m, int32_t seq_id, int32_t* out_tokens, int cap);
/* Block table of `seq_id` as held on the device (page ids, -1 = none). */
int spec_seq_block_table(spec_model* m, int32_t seq_id, int32_t* out_pages, int cap,
                         int32_t* out_n);
int spec_free_pages(spec_model* m);

/* Debug: like spec_verify_step_batch but writes the fp32 logits of every
 * scored row to logits_dev ([n_seq * (max_draft+1), vocab], device) and does
 * NOT commit (sequence state unchanged). */
int spec_debug_logits(spec_model* m, int n_seq, const int32_t* seq_ids,
                      const int32_t* drafts, float* logits_dev);

/* Number of kernel launches one verify step of n_seq sequences enqueues. */
int spec_step_launches(spec_model* m, int n_seq);

/* ---- FastMTP draft head ----------------------------------------------------
 * "Jina-OCR-v1: efficient document parsing with speculative decoding and
 * dense verifiable rewards", section 3.1: one shared draft block applied
 * recursively, K steps per verify step. For position p and depth k, with b_p
 * the decoder's final-normed state of row p and N_o the decoder's final norm:
 *   a_p^(1) = b_p,  a_p^(k) = u_(p-1)^(k-1),
 *   z_p^(k) = P [N_e(E(x_(p+1))) ; N_h(a_p^(k))],
 *   u_p^(k) = N_o(B(z_p^(k); RoPE position p)),  d_k = argmax W_lm u_(p+k-1)^(k)
 * where x_(p+1), ... are the committed tokens followed by d_1..d_(k-1). E, N_o
 * and W_lm are the decoder's (tied). B is one pre-norm decoder layer of the
 * decoder's attention shape with a dense SwiGLU FFN of width `inter`, causal
 * over the rows of its own depth; its keys and values are stored like the
 * decoder's (bf16, f32 for an f32 decoder). Depth k's rows start at row
 * p0 + k - 1, p0 the last visual row of the prompt (0 without visual rows).
 * Ties keep the lowest token id.
 *
 * spec_mtp_init attaches a head to a model with max_draft <= 4.
 * host_tensors[13] (host memory, copied; the caller keeps ownership), row-major:
 *   0 tok_embed, 1 final_norm, 2 lm_head: the decoder's tensors 0..2 as given
 *     to spec_init_model;
 *   3 enorm [hidden] f32, 4 hnorm [hidden] f32,
 *   5 eh_proj [hidden][2 hidden], 6 attn_norm [hidden] f32,
 *   7 w_qkv [(Hq + 2 Hkv) head_dim][hidden], 8 w_o [hidden][Hq head_dim],
 *   9 ffn_norm [hidden] f32, 10 w_gate [inter][hidden], 11 w_up [inter][hidden],
 *   12 w_down [hidden][inter];
 *   matrices in f32 for an f32 decoder, else bf16 (also for e4m3 decoders).
 * Errors: SPEC_ERR_STATE if the model already has a head; SPEC_ERR_UNSUPPORTED
 * for max_draft > 4; SPEC_ERR_NOMEM.
 *
 * spec_mtp_draft writes d_1..d_K (1 <= K <= max_draft) for sequence seq_id
 * after its committed tokens to out_drafts[K] (host). Each depth's cache
 * keeps the committed rows; the rows made from drafts are recomputed by the
 * next call. Valid right after spec_prefill (prompt tail <= 256 rows after
 * p0) or right after the host-mode verify step that committed the new tokens
 * (any step call in between, or a _dev step, makes it SPEC_ERR_STATE; so does
 * a second draft with no new committed token); sequences prefilled with a
 * shared prefix give SPEC_ERR_UNSUPPORTED. The call synchronizes the model's
 * stream once. */
int spec_mtp_init(spec_model* m, const void* const* host_tensors, int inter);
int spec_mtp_draft(spec_model* m, int32_t seq_id, int K, int32_t* out_drafts);
/* Debug: spec_mtp_draft that also writes
 *  - the fp32 logits W_lm u_(p+k-1)^(k) of each depth's draft row to
 *    logits_dev ([K][vocab], device, depth order);
 *  - the decoder states this call reads for depth 1 -- the final residual
 *    rows (before N_o) of positions max(p_last + 1, p0) .. p, p_last the
 *    previous call's p -- to states_dev ([states_cap][hidden] fp32, device),
 *    their count to *out_n_states (SPEC_ERR_ARG if above states_cap).
 * The sequence's head state advances exactly as in spec_mtp_draft. */
int spec_mtp_debug_draft(spec_model* m, int32_t seq_id, int K, int32_t* out_drafts, float* logits_dev,
                         float* states_dev, int states_cap, int32_t* out_n_states);

/* ---- profiling ------------------------------------------------------------ */
/* Per kernel class: summed device time (ms, CUDA events on the model's stream
 * around each launch), launch count, and work units (active experts for the
 * expert kernels, 0 otherwise). */
typedef struct spec_kernel_stat {
  float ms;
  int32_t launches;
  int64_t units;
} spec_kernel_stat;
#define SPEC_KCLASS_COUNT 11
/* Run n_steps device-resident verify steps WITHOUT graph replay, bracketing
 * every kernel launch with CUDA events. Arguments as in
 * spec_verify_step_batch_dev; step s reads drafts_dev + s * drafts_step_stride.
 * Fills out[0..n_out) and returns the number of classes written. The host view
 * of the sequences must be refreshed with spec_sync_seqs afterwards. */
int spec_profile_steps_dev(spec_model* m, int n_seq, const int32_t* seq_ids_dev, const int32_t* drafts_dev,
                           const int32_t* n_draft_dev, int n_steps, int drafts_step_stride,
                           spec_kernel_stat* out, int n_out);
const char* spec_kernel_class_name(int cls);
/* Host<->device bytes moved by the library's step calls since init (inputs
 * staged, block-table rows uploaded, results read back). */
int spec_io_bytes(spec_model* m, int64_t* out_h2d, int64_t* out_d2h);

const char* spec_strerror(int code);
const char* spec_last_error(void);

/* ---- kernel-level entry points (device pointers, enqueued on cuda_stream) - */
/* Final RMSNorm + LM head + greedy argmax for T rows without writing logits
 * (the target's token at every verified position: "Jina-OCR-v1", abstract,
 * greedy verification; "End-to-end OCR expert model ...", section 6.1):
 *   out_tokens_dev[t] = argmax_v  sum_k W[v][k] * gamma[k] * x[t][k] / rms(x[t]),
 *   rms(z) = sqrt(mean(z^2) + eps); ties keep the lowest index v; a NaN logit
 *   ranks below every number (a row of NaNs gives 0), so the token is always
 *   a valid index.
 * x_dev: [T, hidden] f32. w_dev: [vocab, hidden] row-major, w_dtype SPEC_F32 or
 * SPEC_BF16. gamma_dev: [hidden] f32. scratch_dev: caller-owned device memory
 * of at least spec_lmhead_argmax_scratch_bytes(T, vocab) bytes (per-block
 * (max, index) candidates), fully rewritten by each call. vocab must be a
 * multiple of 4, a weight row a multiple of 16 bytes, hidden <= 12288.
 * Returns after enqueueing; errors: SPEC_ERR_ARG, SPEC_ERR_UNSUPPORTED,
 * SPEC_ERR_CUDA (launch failure). */
int64_t spec_lmhead_argmax_scratch_bytes(int T, int vocab);
int spec_lmhead_argmax(const float* x_dev, int T, int hidden, int vocab, const void* w_dev, int w_dtype,
                       const float* gamma_dev, float eps, void* scratch_dev, size_t scratch_bytes,
                       int32_t* out_tokens_dev, uintptr_t cuda_stream);

/* Tensor-core GEMM check: with weights A [M, K] (bf16, or e4m3 when a_fp8,
 * then scaled per row by a_scale_dev[m]) and activations X = B + B_lo (bf16
 * [N, K] each, row-major, device; b_lo_dev may be NULL; with a_fp8 the
 * operands are f16 and B + B_lo = 256 X, the f16 parts the e4m3-weight GEMMs
 * of a model take, and the dual output is f16(256 h)), in CTAs of n_tile
 * activation rows (32, 64 or 128; 0 = 128) and k_split K splits (0 or 1: none;
 * partials summed in split order by the tile's last split), dual = 0 writes
 * out_dev[n][m] = sum_k A[m][k] * X[n][k] (fp32 [N, M]); dual = 1 writes
 * out_dev[n][m] = bf16(silu(A[m]·X[n]) * (A2[m]·X[n])) (bf16 [N, M]) -- the
 * epilogues the expert GEMMs use. The scale pointers may be NULL (1.0). M a
 * multiple of 128, K of 64. err_dev: device int that receives error bits
 * (8 = an mbarrier wait ran out: every wait ends by a 250 ms deadline, after
 * which the kernel stops, drains what it has in flight and returns).
 * flags: 0 normally; SPEC_TC_TEST_STALL makes the kernel issue no loads, so
 * its waits run out (a check of the deadline: err_dev gets bit 8, out_dev is
 * not written and the context stays usable). Enqueued on cuda_stream. */
#define SPEC_TC_TEST_STALL 1
int spec_tc_gemm_test(const void* a_dev, const void* a2_dev, const float* a_scale_dev, const float* a2_scale_dev,
                      int a_fp8, const void* b_dev, const void* b_lo_dev, int M, int N, int K, int dual, int n_tile,
                      int k_split, int flags, void* out_dev, int* err_dev, uintptr_t cuda_stream);

/* Rejection-sampling verification, the stochastic counterpart of the greedy
 * acceptance rule ("End-to-end OCR expert model architecture and acceleration
 * principles", section 6.1 and section 11 item 2: rejection sampling keeps
 * the output distribution equal to the target model's own). Read as the
 * published speculative-sampling rule: with p_j = softmax(row j-1 of the
 * sequence's logits / temperature), j = 1..K+1, and the drafter's q_j:
 *   accept d_j while u_accept[j-1] * q_j(d_j) < p_j(d_j);
 *   at the first rejection (draft j) append a draw from max(0, p_j - q_j)
 *   (normalised; p_j itself if that is zero everywhere) with u_sample[j-1];
 *   if all K are accepted append a draw from p_(K+1) with u_sample[K].
 * A draw with weights w and uniform u is the smallest v whose running sum of
 * w (index order) exceeds u * sum(w). Computed in fp32 with fixed reduction
 * orders (rounding can move a draw across a bucket edge that u * sum(w) lies
 * within about 1e-6 of sum(w)).
 *   logits_dev:  [n_seq][K+1][vocab] f32, 16-byte aligned (the layout
 *                spec_debug_logits writes).
 *   drafts_dev:  [n_seq][K] int32 draft tokens.
 *   q_dev:       [n_seq][K][vocab] f32 drafter probabilities (16-byte
 *                aligned), or NULL for a drafter certain of its drafts (q_j
 *                one-hot at d_j).
 *   u_accept_dev [n_seq][K], u_sample_dev [n_seq][K+1]: f32 uniforms in [0, 1).
 *   out_accepted_dev / out_token_dev: [n_seq] int32: drafts accepted and the
 *                appended token; -1 / -1 for a sequence with a draft outside
 *                [0, vocab).
 * All device pointers, caller-owned; enqueued on cuda_stream. vocab must be a
 * multiple of 4 and at most 262144; K >= 0 (K = 0 samples row 0).
 * Errors: SPEC_ERR_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA (launch). */
int spec_rejection_sample(const float* logits_dev, const int32_t* drafts_dev, const float* q_dev,
                          const float* u_accept_dev, const float* u_sample_dev, int n_seq, int K, int vocab,
                          float temperature, int32_t* out_accepted_dev, int32_t* out_token_dev,
                          uintptr_t cuda_stream);
/* The same rule as one cooperative launch that spreads each sequence over
 * several blocks, all resident at once. Each row is cut into tiles of 1,024
 * values; the blocks of a sequence share the row's tiles and meet at a
 * counter of the sequence after each row, and only the rows the rule reaches
 * are read. The draw picks its tile from per-tile sums and then scans that
 * one tile. Same arguments, plus:
 *   ws_dev:   a caller-owned device workspace, 16-byte aligned, of at least
 *             spec_rejection_sample_ws_bytes(n_seq, K) bytes. It must be
 *             zero-filled before its first use; every call leaves its
 *             counters at zero again, so it can be reused by later calls on
 *             the same stream. One call at a time per workspace.
 * The per-tile sums use the fast hardware exponential and another summation
 * order than spec_rejection_sample's, so the two can differ where a decision
 * lies within rounding of its threshold. A sequence reports (-2, -1) if a
 * wait between its blocks ran past its deadline (not expected: the launch is
 * cooperative); its workspace must then be zero-filled again.
 * Errors: as spec_rejection_sample; SPEC_ERR_ARG for a small or misaligned
 * workspace; SPEC_ERR_CUDA when the launch cannot be made cooperative. */
int64_t spec_rejection_sample_ws_bytes(int n_seq, int K);
int spec_rejection_sample_ws(const float* logits_dev, const int32_t* drafts_dev, const float* q_dev,
                             const float* u_accept_dev, const float* u_sample_dev, int n_seq, int K, int vocab,
                             float temperature, int32_t* out_accepted_dev, int32_t* out_token_dev, void* ws_dev,
                             size_t ws_bytes, uintptr_t cuda_stream);

/* Same computation as spec_lmhead_argmax for callers that cannot allocate
 * device memory (no cudaMalloc of their own, none by the library): the
 * candidate scratch is a fixed device array inside the library, sized for
 * SPEC_LMHEAD_NOALLOC_MAX_PAIRS (max, index) pairs (2 MiB), which every GPU
 * that loads the library holds until the process exits. The pages describe
 * nothing like it; it exists only for such callers.
 *  - Sizes with T * ceil(vocab / 32) > SPEC_LMHEAD_NOALLOC_MAX_PAIRS are
 *    rejected with SPEC_ERR_ARG.
 *  - The first call on a device resolves the array's address and sets the
 *    kernels' attributes (with that device current); make that first call
 *    before any stream capture.
 *  - All calls on a device share the array and each call rewrites every
 *    candidate it reads, so no state carries over; calls whose kernels
 *    overlap on the GPU (different streams, no ordering) race on it.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine. */
#define SPEC_LMHEAD_NOALLOC_MAX_PAIRS 262144
int spec_lmhead_argmax_noalloc(const float* x_dev, int T, int hidden, int vocab, const void* w_dev,
                               int w_dtype, const float* gamma_dev, float eps, int32_t* out_tokens_dev,
                               uintptr_t cuda_stream);

/* ---- paged KV allocator (host only; usable without a GPU) ---------------- */
/* The same allocator the model uses, exposed for tests and tooling. Pages
 * hold page_size consecutive positions; a sequence's block table lists its
 * pages in position order. Prefix pages are refcounted. */
typedef struct spec_pool spec_pool;
int spec_pool_create(int n_pages, int page_size, int max_seqs, int max_pages_per_seq,
                     spec_pool** out);
int spec_pool_destroy(spec_pool* p);
/* Make seq hold pages for positions [0, n_tokens); allocates as needed. */
int spec_pool_reserve(spec_pool* p, int32_t seq, int n_tokens);
/* Commit: keep pages covering max(new_len, keep_pages*page_size) positions,
 * release the rest; the sequence length becomes new_len. */
int spec_pool_commit(spec_pool* p, int32_t seq, int new_len, int keep_pages);
int spec_pool_release(spec_pool* p, int32_t seq);
/* Share the first n_pages pages of `src_seq` with the empty sequence `dst`
 * (refcount + 1 each). */
int spec_pool_share(spec_pool* p, int32_t src_seq, int n_pages, int32_t dst);
int spec_pool_block_table(spec_pool* p, int32_t seq, int32_t* out, int cap, int32_t* out_n);
int spec_pool_refcount(spec_pool* p, int32_t page);
int spec_pool_free_count(spec_pool* p);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_H_ */
