/*
 * tim.h -- batch-invariant linear logprob and three-way score comparison on
 * one GB300 (sm_103a).  Plain C ABI: raw pointers and sizes only.
 *
 * The operations are defined by these passages:
 *
 *  - selected-token logprob l_t = z_t[x_t] - log sum_v exp z_t[v] in nats,
 *    temperature applied to the logits before the softmax:
 *      "Debugging Logprob Mismatches in LLM Reinforcement Learning",
 *      Case 2: A and B Stay Close; C Changes (the l_t equation);
 *      What a Logprob Difference Means (natural log, nats);
 *      Make Sure Both Scores Describe the Same Probability (score-definition
 *      table) and "How this differs from a real temperature mismatch".
 *  - the "linear logprob" of the strict path: final RMSNorm (fixed reduction
 *    domain and epsilon), LM-head GEMM with a fixed K-dimension reduction,
 *    normaliser over the true vocabulary range merged across vocabulary chunks
 *    in a fixed order:
 *      "Training and rollout stop disagreeing: vime and RL-Kernel hold
 *      logprobs bitwise identical for 200 steps on AMD MI300X", Interpretation.
 *  - no batch-size dependent GEMM path:
 *      "Rollout-Training Mismatch in LLM RL", section 5.2 (table: remove
 *      small-batch backend switches, batch-invariant accumulation).
 *  - the per-sequence comparison of generation (A), replay (B) and trainer (C)
 *    scores: "Fault localization and mismatch bisect", Per-sequence
 *    observation patterns, Metric measurement basis and Compare per-token
 *    logprobs; "Debugging Logprob Mismatches ...", Check Whether the Pattern
 *    Extends Across the Response; eq. (1) of "Rollout-Training Mismatch in
 *    LLM RL" (section 1.2); token TIS of "Diagnosing Training Inference
 *    Mismatch in LLM Reinforcement Learning", 3. TIS.
 *
 * Conventions for every entry point
 *  - All data pointers are DEVICE pointers owned by the caller (the library
 *    allocates nothing per call and keeps no per-call global state).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  Nothing is synchronised unless stated.
 *  - Argument errors (null pointers, bad sizes, bad alignment, workspace too
 *    small, wrong GPU) are returned immediately and nothing is enqueued.
 *  - Data-dependent errors found by the kernels (token id out of range,
 *    non-finite values, empty sequence, bad mask, bad offsets, a bounded wait
 *    that timed out) are recorded in a status word inside the workspace; the
 *    first recorded error is kept.  tim_status_sync() returns and clears it.
 *    Once an error is reported, the numbers of that call are not to be trusted.
 *  - A workspace must be zero-initialised once (tim_workspace_init) before its
 *    first use; it may then be reused by any number of calls on one stream,
 *    of any shape whose workspace size it covers.  Calls that share a
 *    workspace must not overlap in time.  A workspace serves one family of
 *    calls: either the tim_logprob family or tim_compare / tim_compare_diag
 *    (these keep per-sequence counters in the workspace; each call zeroes its
 *    own before use).
 *
 * Only sm_103 devices (GB300) are supported.
 */
#ifndef TIM_H_
#define TIM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle type, declared here without CUDA headers. */
typedef struct CUstream_st *tim_stream_t;

typedef enum tim_status {
  TIM_OK = 0,
  TIM_ERR_INVALID_ARG = 1,         /* null pointer, bad size/scalar, bad offsets */
  TIM_ERR_SHAPE = 2,               /* d not a multiple of 64, d/V/T out of range */
  TIM_ERR_TOKEN_RANGE = 3,         /* a token id outside [0, V) (row -> NaN)     */
  TIM_ERR_NONFINITE = 4,           /* non-finite hidden value, lse or score      */
  TIM_ERR_EMPTY_SEQUENCE = 5,      /* a sequence with no active token            */
  TIM_ERR_BAD_MASK = 6,            /* a mask byte that is neither 0 nor 1        */
  TIM_ERR_WORKSPACE = 7,           /* workspace pointer/size insufficient        */
  TIM_ERR_CUDA = 8,                /* a CUDA runtime/driver call failed          */
  TIM_ERR_TIMEOUT = 9,             /* a bounded device-side wait gave up         */
  TIM_ERR_UNSUPPORTED_DEVICE = 10, /* current device is not sm_103               */
  TIM_ERR_CAPACITY = 11            /* a row had more top-k candidates than fit   */
} tim_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *tim_status_string(tim_status s);

/* ABI version of this header (bumped on any signature or struct change). */
int32_t tim_abi_version(void);
#define TIM_ABI_VERSION 1

/* Zero a whole workspace, status word included (enqueued on `stream`).  Call
 * once after allocating a workspace, before its first use. */
tim_status tim_workspace_init(void *workspace, size_t workspace_bytes, tim_stream_t stream);

/* Synchronise `stream`, then return the first data-dependent error recorded
 * in `workspace` since the last tim_status_sync / tim_workspace_init and
 * clear it.  Returns TIM_ERR_CUDA if a CUDA call failed. */
tim_status tim_status_sync(void *workspace, tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Linear logprob.
 *
 * For every row t in [0, T) (rows are pre-aligned: hidden row t predicts
 * token_ids[t]):
 *   rstd_t      = 1 / sqrt(mean_i(h_ti^2) + eps)              (fp32)
 *   y_ti        = bf16_round_nearest_even(h_ti * rstd_t * gamma_i)
 *   z_tv        = sum_i y_ti * W_vi                           (fp32 accumulation)
 *   s_tv        = z_tv / temperature
 *   out_lse[t]  = ln sum_{v<V} exp(s_tv)                      (nats)
 *   out_logprob[t] = s_t[token_ids[t]] - out_lse[t]
 *   out_top1[t] = smallest v with z_tv maximal (unscaled logits)
 * The [T, V] logits are never written to memory.
 *
 * Batch invariance: the bits of every output of row t depend only on row t's
 * inputs (hidden row, token id), W, gamma, V, d, temperature and eps -- not on
 * T, on the other rows, on the row's position, or on the number of SMs.
 *
 * Arguments
 *   hidden      bf16 [T, d] row-major (row stride d elements), 16-byte aligned.
 *   gamma       bf16 [d], 16-byte aligned.
 *   W           bf16 [V, d] row-major (nn.Linear weight layout), 16-byte aligned.
 *   token_ids   int32 [T].
 *   T           rows, 1 <= T <= 2^31 - 1.
 *   d           hidden size, a multiple of 64, 64 <= d <= 65536.
 *   V           vocabulary size, 1 <= V <= 2^31 - 256.
 *   temperature finite and > 0 (1.0 gives the raw-model score).
 *   eps         finite and >= 0.
 *   out_logprob float32 [T]; NaN where the token id is out of range.
 *   out_lse     float32 [T].
 *   out_top1    int32 [T].
 *   workspace   device buffer of at least tim_logprob_workspace_size(T, d, V)
 *               bytes, 256-byte aligned, zero-initialised once.
 * Errors: TIM_ERR_INVALID_ARG, TIM_ERR_SHAPE, TIM_ERR_WORKSPACE,
 *   TIM_ERR_UNSUPPORTED_DEVICE, TIM_ERR_CUDA (immediate); TIM_ERR_TOKEN_RANGE,
 *   TIM_ERR_NONFINITE, TIM_ERR_TIMEOUT (via tim_status_sync).
 * ------------------------------------------------------------------------ */
size_t tim_logprob_workspace_size(int64_t T, int32_t d, int32_t V);

tim_status tim_logprob(const void *hidden, const void *gamma, const void *W,
                       const int32_t *token_ids, int64_t T, int32_t d, int32_t V,
                       float temperature, float eps, float *out_logprob, float *out_lse,
                       int32_t *out_top1, void *workspace, size_t workspace_bytes,
                       tim_stream_t stream);

/* The three stages of tim_logprob, exposed so that callers can time or
 * overlap them.  tim_logprob is exactly these three calls in this order on
 * the same workspace; the arguments mean the same as above and must be the
 * same (T, d, V, temperature) across the three calls.
 *
 * Stage 1, RMSNorm: writes y (bf16 [T, d]) into the workspace.
 * Stage 2, LM head + per-vocabulary-tile softmax statistics: reads y and W,
 *          writes one (max, sum of exponentials, best logit, best id) record
 *          per (row, 256-column vocabulary tile) and the target logit of each
 *          row into the workspace.
 * Stage 3, finalize: merges each row's tile records in a fixed order and
 *          writes out_logprob, out_lse and out_top1. */
tim_status tim_rmsnorm_rows(const void *hidden, const void *gamma, int64_t T, int32_t d,
                            int32_t V, float eps, void *workspace, size_t workspace_bytes,
                            tim_stream_t stream);
tim_status tim_lmhead_lse(const void *W, const int32_t *token_ids, int64_t T, int32_t d,
                          int32_t V, float temperature, void *workspace,
                          size_t workspace_bytes, tim_stream_t stream);
tim_status tim_lse_finalize(const int32_t *token_ids, int64_t T, int32_t d, int32_t V,
                            float temperature, float *out_logprob, float *out_lse,
                            int32_t *out_top1, void *workspace, size_t workspace_bytes,
                            tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Three-way compare.
 *
 * Score sets for the same saved tokens: A = lp_gen (generation), B =
 * lp_replay (rollout prefill replay), C = lp_train (frozen trainer forward).
 * Sequence j covers rows [seq_offsets[j], seq_offsets[j+1]); its active
 * tokens are the rows with mask == 1, numbered 0, 1, ... in row order.
 *
 * For each pair p (0: A-B, 1: B-C, 2: A-C; left minus right):
 *   mismatch_count  active tokens whose float32 bit patterns differ
 *                   (+0.0 and -0.0 differ);
 *   first_div       ordinal of the first such token, -1 if none;
 *   longest_run     longest run of consecutive active ordinals that differ;
 *   max_abs_diff    max |double(x) - double(y)|  (exact);
 *   signed_mean     mean of double(x) - double(y);
 *   mae             mean of |double(x) - double(y)|.
 * With d = double(C) - double(A) per active token:
 *   mean_log_ratio = mean(C - A) = mean_weight_move + mean_same_version,
 *   mean_weight_move = mean(C - B), mean_same_version = mean(B - A)  (eq. 1),
 *   k3_mean = mean(expm1(d) - d)  (Schulman k3; not clipped: overflow gives
 *             +inf and sets TIM_SEQ_K3_OVERFLOW),
 *   token TIS weight w = cap if d > ln(cap) else exp(d);
 *   tis_mean = mean(w), tis_clipped = number of tokens with d > ln(cap).
 * out_tis_w[t] = float(w) for active rows, 0 for inactive rows of a
 * sequence; rows outside every sequence are not written.
 * Means are fp64 sums in a fixed order divided by n_valid.
 *
 * Arguments
 *   lp_gen, lp_replay, lp_train  float32 [T] (any alignment; 16-byte aligned
 *                                arrays take the 128-bit load path).
 *   seq_offsets  int64 [n_seq + 1]; each sequence needs
 *                0 <= seq_offsets[j] <= seq_offsets[j+1] <= T.
 *   n_seq        >= 1.
 *   mask         uint8 [T], values 0 or 1.
 *   T            1 <= T <= 2^31 - 1.
 *   tis_cap      finite and > 0.
 *   out_stats    tim_seq_stats [n_seq] (device memory).
 *   out_tis_w    float32 [T] or NULL.
 *   workspace    >= tim_compare_workspace_size(T, n_seq) bytes, zero-initialised once.
 * Per-sequence problems set bits in tim_seq_stats.flags and the status word:
 *   bad offsets -> TIM_SEQ_BAD_OFFSETS / TIM_ERR_INVALID_ARG (stats zeroed),
 *   mask byte not 0/1 -> TIM_SEQ_BAD_MASK / TIM_ERR_BAD_MASK (stats zeroed),
 *   no active token -> TIM_SEQ_EMPTY / TIM_ERR_EMPTY_SEQUENCE,
 *   non-finite active score -> TIM_SEQ_NONFINITE / TIM_ERR_NONFINITE.
 * out_tis_w rows of a sequence flagged BAD_OFFSETS or BAD_MASK are unspecified.
 * ------------------------------------------------------------------------ */
typedef struct tim_pair_stats {
  int64_t mismatch_count;
  int64_t first_div;
  int64_t longest_run;
  double max_abs_diff;
  double signed_mean;
  double mae;
} tim_pair_stats;

typedef struct tim_seq_stats {
  int64_t n_valid;
  tim_pair_stats pair[3]; /* 0: A-B, 1: B-C, 2: A-C */
  double mean_log_ratio;    /* C - A */
  double mean_weight_move;  /* C - B */
  double mean_same_version; /* B - A */
  double k3_mean;
  double tis_mean;
  int64_t tis_clipped;
  int32_t flags;
  int32_t reserved;
} tim_seq_stats;

#define TIM_SEQ_EMPTY 1
#define TIM_SEQ_BAD_MASK 2
#define TIM_SEQ_NONFINITE 4
#define TIM_SEQ_BAD_OFFSETS 8
#define TIM_SEQ_K3_OVERFLOW 16

/* Each sequence is reduced in parts cut from its own length (256 tokens a part,
 * at most 256 parts) and the parts are folded in order, so a sequence's
 * statistics, fp64 sums included, are the same bits in any batch. */
size_t tim_compare_workspace_size(int64_t T, int32_t n_seq);

tim_status tim_compare(const float *lp_gen, const float *lp_replay, const float *lp_train,
                       const int64_t *seq_offsets, int32_t n_seq, const uint8_t *mask,
                       int64_t T, float tis_cap, tim_seq_stats *out_stats, float *out_tis_w,
                       void *workspace, size_t workspace_bytes, tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * FP8 (e4m3) variant of the linear logprob.
 *
 * "Rollout-Training Mismatch in LLM RL", section 3 (Unified FP8 table): FP8
 * quantize-dequantize forward values, and native FP8 GEMMs consuming codes and
 * scales.  Quantisation here: one power-of-two scale per row, the smallest s
 * with max|row| / s <= 448 (1 for an all-zero row); code = e4m3(x / s), round
 * to nearest-even, saturating.  W is quantised by vocabulary row (once, with
 * tim_quantize_fp8_rows); y (the bf16 output of the final RMSNorm, exactly as
 * in tim_logprob) by token row inside tim_logprob_fp8.  The LM head runs on
 * the e4m3 codes (tcgen05 kind::f8f6f4, fp32 accumulation) and multiplies each
 * logit by s_y[t] * s_W[v]; because the scales are powers of two this equals
 * the GEMM of the quantize-dequantize operands.  Everything after the logits is
 * the tim_logprob path.  Batch-invariant like tim_logprob.
 *
 * tim_quantize_fp8_rows: x = bf16 [rows, K] (16-byte aligned, K a multiple of
 *   16) -> codes = e4m3 bytes [rows, K] (8-byte aligned), scales = float32
 *   [rows].  Asynchronous on `stream`; needs no workspace.
 * tim_logprob_fp8: as tim_logprob, with W_codes = e4m3 [V, d] and W_scales =
 *   float32 [V] from tim_quantize_fp8_rows, d a multiple of 128, and a
 *   workspace of tim_logprob_fp8_workspace_size bytes.
 * ------------------------------------------------------------------------ */
tim_status tim_quantize_fp8_rows(const void *x, int64_t rows, int32_t K, void *codes,
                                 float *scales, tim_stream_t stream);

size_t tim_logprob_fp8_workspace_size(int64_t T, int32_t d, int32_t V);

tim_status tim_logprob_fp8(const void *hidden, const void *gamma, const void *W_codes,
                           const float *W_scales, const int32_t *token_ids, int64_t T, int32_t d,
                           int32_t V, float temperature, float eps, float *out_logprob,
                           float *out_lse, int32_t *out_top1, void *workspace,
                           size_t workspace_bytes, tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * FP32 variant of the linear logprob.
 *
 * "Rollout-Training Mismatch in LLM RL", section 4.3 (an FP32 rollout LM head)
 * and section 5.2 (wider arithmetic beside the aligned forward): the head in
 * fp32.  y = (h * rstd) * gamma stays fp32 (no bf16 rounding; RMSNorm as in
 * tim_logprob otherwise) and W is fp32 [V, d] (fp32 master weights, or bf16
 * weights widened).  The GEMM runs on the tcgen05 tensor cores as three tf32
 * products per K step: each fp32 operand x is given as big = x with its low 13
 * mantissa bits cleared (a tf32 value) and small = x - big (exact), and
 * z = big_y.big_W + big_y.small_W + small_y.big_W with fp32 accumulation
 * (the dropped small.small term is below 2^-20 of each product).  Everything
 * after the logits is the tim_logprob path.  Batch-invariant like tim_logprob.
 *
 * tim_split_tf32: x fp32 [n] -> big, small fp32 [n] (all 16-byte aligned, n a
 *   multiple of 4).  Asynchronous on `stream`.  Run once per weight version on
 *   W (the caller keeps W_big and W_small, 8 V d bytes).
 * tim_logprob_fp32: as tim_logprob, with W_big / W_small fp32 [V, d] from
 *   tim_split_tf32 and a workspace of tim_logprob_fp32_workspace_size bytes.
 * ------------------------------------------------------------------------ */
tim_status tim_split_tf32(const float *x, int64_t n, float *big, float *small,
                          tim_stream_t stream);

size_t tim_logprob_fp32_workspace_size(int64_t T, int32_t d, int32_t V);

tim_status tim_logprob_fp32(const void *hidden, const void *gamma, const float *W_big,
                            const float *W_small, const int32_t *token_ids, int64_t T, int32_t d,
                            int32_t V, float temperature, float eps, float *out_logprob,
                            float *out_lse, int32_t *out_top1, void *workspace,
                            size_t workspace_bytes, tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Backward of the linear logprob.
 *
 * "Rollout-Training Mismatch in LLM RL", section 5.2: the inference kernels
 * define the forward values, the trainer supplies the backward through a
 * custom autograd wrapper, and the recipe recomputes the forward rather than
 * saving its intermediates.  For L = sum_t g_t * logprob_t (g = grad_logprob,
 * the upstream gradient) this computes, with y the bf16 RMSNorm output exactly
 * as tim_logprob computes it:
 *   G_tv  = (g_t / temperature) * (1[v = x_t] - p_tv),
 *           p_tv = exp(z_tv / temperature - lse_t),  z = y . W^T recomputed;
 *   out_dy = dL/dy = G . W     fp32 [T, d]  (row-major, 16-byte aligned);
 *   out_dW = dL/dW = G^T . y   fp32 [V, d]  (row-major, 16-byte aligned);
 *           accumulate_dW = 1 adds to out_dW instead (for callers that split a
 *           batch into row chunks), 0 overwrites it.
 * lse: fp32 [T], the out_lse of the tim_logprob call on the same inputs.  G is
 * rounded to bf16 for the two tensor-core products (fp32 accumulation).  A row
 * whose token id is outside [0, V) contributes nothing and records
 * TIM_ERR_TOKEN_RANGE.  Each out_dy row depends only on its own row (batch-
 * invariant); out_dW sums over the rows in a fixed order.
 * Workspace: tim_logprob_backward_workspace_size(T, d, V) bytes (it holds y and
 * G, about 2 T V bytes: the two products read G, W and y where they lie, G and y
 * as MN-major operands), 256-byte aligned, zero-initialised once;
 * T up to 4.19 M rows and V up to 4.19 M.  Errors as tim_logprob.
 * ------------------------------------------------------------------------ */
size_t tim_logprob_backward_workspace_size(int64_t T, int32_t d, int32_t V);

tim_status tim_logprob_backward(const void *hidden, const void *gamma, const void *W,
                                const int32_t *token_ids, const float *lse,
                                const float *grad_logprob, int64_t T, int32_t d, int32_t V,
                                float temperature, float eps, float *out_dy, float *out_dW,
                                int32_t accumulate_dW, void *workspace, size_t workspace_bytes,
                                tim_stream_t stream);

/* RMSNorm backward, to carry out_dy of tim_logprob_backward on to the hidden
 * states and gamma (same section: a custom autograd wrapper around the forward
 * needs the gradients of its inputs).  The bf16 rounding of y is passed straight
 * through; with r_t = 1 / sqrt(mean_i h_ti^2 + eps) computed exactly as the
 * forward computes it:
 *   out_dh[t, i]    = r_t gamma_i dy_ti - (r_t^3 / d) h_ti sum_j gamma_j dy_tj h_tj
 *   out_dgamma[i]   = sum_t dy_ti h_ti r_t   (+= when accumulate_dgamma = 1)
 * hidden bf16 [T, d], gamma bf16 [d], dy fp32 [T, d] (16-byte aligned), out_dh
 * fp32 [T, d] (16-byte aligned), out_dgamma fp32 [d].  Rows are independent;
 * out_dgamma sums rows in a fixed order.  Workspace:
 * tim_rmsnorm_backward_workspace_size(T, d) bytes; T up to 16.7 M rows.  Errors
 * as tim_logprob (non-finite hidden values: TIM_ERR_NONFINITE via
 * tim_status_sync). */
size_t tim_rmsnorm_backward_workspace_size(int64_t T, int32_t d);

tim_status tim_rmsnorm_backward(const void *hidden, const void *gamma, const float *dy, int64_t T,
                                int32_t d, float eps, float *out_dh, float *out_dgamma,
                                int32_t accumulate_dgamma, void *workspace,
                                size_t workspace_bytes, tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Processed (top-k, then top-p) selected-token logprob.
 *
 * "Debugging Logprob Mismatches in LLM Reinforcement Learning", Make Sure
 * Both Scores Describe the Same Probability: the sampling score is taken on
 * the distribution left after the sampler's filters, renormalised (top-k with
 * k = 2 turns (0.50, 0.30, 0.20) into (0.625, 0.375, 0)).
 *
 * With s_v = z_v / temperature (z as in tim_logprob):
 *   top-k set K = the top_k tokens by z (equal logits: lower id first);
 *   q = softmax of s over K; walking K in that order, a token is kept when the
 *   q-mass of the tokens before it is < top_p (the first is always kept);
 *   out_lse_kept[t] = ln sum_{v kept} exp(s_v);
 *   out_logprob[t]  = s_x - out_lse_kept[t] if the target x is kept, else -inf;
 *   out_kept[t]     = number of kept tokens.
 * Cost: one LM-head GEMM pass that keeps the four largest logits of every
 * (row, 256-column tile).  The k-th largest tile maximum is a bound every
 * top-k logit meets; a row with a tile holding four or more logits at or above
 * it (or a vocabulary of fewer than top_k tiles) is gathered and rescored,
 * collecting every logit at or above the bound.  Results are batch-invariant
 * like tim_logprob's and do not depend on which route a row took.
 *
 * Limits: 1 <= top_k <= TIM_PROCESSED_MAX_K, 0 < top_p <= 1, at most 2048
 * vocabulary tiles (V <= 524288), and either V >= 256 * top_k or
 * V <= TIM_PROCESSED_CAPACITY.  A row with more than TIM_PROCESSED_CAPACITY
 * candidates (many logits tied near the top) reports TIM_ERR_CAPACITY and NaN.
 * Other arguments and errors as tim_logprob; the workspace is
 * tim_processed_logprob_workspace_size bytes.
 * ------------------------------------------------------------------------ */
#define TIM_PROCESSED_MAX_K 64
#define TIM_PROCESSED_CAPACITY 2048

size_t tim_processed_logprob_workspace_size(int64_t T, int32_t d, int32_t V);

tim_status tim_processed_logprob(const void *hidden, const void *gamma, const void *W,
                                 const int32_t *token_ids, int64_t T, int32_t d, int32_t V,
                                 float temperature, float eps, int32_t top_k, float top_p,
                                 float *out_logprob, float *out_lse_kept, int32_t *out_kept,
                                 void *workspace, size_t workspace_bytes, tim_stream_t stream);

/* The same score, also returning the sampler's top-k head of every row: the
 * K = min(top_k, V) token ids in top-k order (logit descending, lower id first
 * on equal logits) and their processed logprobs, s_v - out_lse_kept[t] for a
 * kept token and -inf for one past the top-p cut.  "Rollout-Training Mismatch
 * in LLM RL", section 4.3: score centering needs the sampler-expected trainer
 * score, and its reference implementation stores a top-k head.
 *   out_head_ids      int32 [T, K] row-major; out_head_logprob fp32 [T, K].
 * Both NULL is tim_processed_logprob; one NULL is TIM_ERR_INVALID_ARG.  A row
 * that reports TIM_ERR_CAPACITY gets ids -1 and NaN logprobs. */
tim_status tim_processed_logprob_head(const void *hidden, const void *gamma, const void *W,
                                      const int32_t *token_ids, int64_t T, int32_t d, int32_t V,
                                      float temperature, float eps, int32_t top_k, float top_p,
                                      float *out_logprob, float *out_lse_kept, int32_t *out_kept,
                                      int32_t *out_head_ids, float *out_head_logprob,
                                      void *workspace, size_t workspace_bytes,
                                      tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Vocabulary-parallel linear logprob.
 *
 * "Debugging Logprob Mismatches in LLM Reinforcement Learning", Collect A/B
 * and C in Your Own Run: with a vocabulary-parallel LM head the normaliser
 * must run over all shards together; "Training and rollout stop disagreeing:
 * vime and RL-Kernel ...", Interpretation: cross-rank LSE merge, fixed rank
 * reduction order.
 *
 * The vocabulary is split over G ranks (G = 1, 2, 4, 8 or 16) along the 16
 * fixed merge ranges of tim_lse_finalize: rank g owns global ids
 * [v0, v0 + v_len) from tim_vocab_shard (whole 256-column tiles; the last
 * shards may be empty for small V).  Rank g calls tim_logprob_shard with its
 * W rows; the callers all-gather the per-row records (16 bytes) and target
 * logits (4 bytes) into [G][T] arrays in rank order; every rank then calls
 * tim_logprob_merge_shards.  The outputs are bitwise identical to
 * tim_logprob's on the full W for every G.
 *
 * tim_logprob_shard arguments: hidden, gamma, token_ids, T, d, temperature and
 *   eps as for tim_logprob; V = the FULL vocabulary size; W_shard = bf16
 *   [v_len, d] rows v0 .. v0+v_len-1 of W (may be NULL when v_len = 0, in
 *   which case nothing is enqueued); out_rec = 16-byte records [T] (16-byte
 *   aligned); out_tgt = float32 [T] (the target's scaled logit, meaningful on
 *   the rank that owns the target id); workspace of
 *   tim_logprob_shard_workspace_size bytes.
 * tim_logprob_merge_shards arguments: recs = [G][T] records, tgts = [G][T]
 *   float32, token_ids [T], T, V (full), G; outputs as tim_logprob; workspace
 *   of tim_logprob_merge_workspace_size bytes (status word: token range,
 *   non-finite lse).
 * ------------------------------------------------------------------------ */
tim_status tim_vocab_shard(int32_t V, int32_t G, int32_t g, int32_t *v0, int32_t *v_len);
size_t tim_logprob_shard_workspace_size(int64_t T, int32_t d, int32_t V, int32_t G, int32_t g);
tim_status tim_logprob_shard(const void *hidden, const void *gamma, const void *W_shard,
                             const int32_t *token_ids, int64_t T, int32_t d, int32_t V,
                             int32_t G, int32_t g, float temperature, float eps, void *out_rec,
                             float *out_tgt, void *workspace, size_t workspace_bytes,
                             tim_stream_t stream);
size_t tim_logprob_merge_workspace_size(int64_t T);
tim_status tim_logprob_merge_shards(const void *recs, const float *tgts, const int32_t *token_ids,
                                    int64_t T, int32_t V, int32_t G, float *out_logprob,
                                    float *out_lse, int32_t *out_top1, void *workspace,
                                    size_t workspace_bytes, tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Extended per-sequence diagnostics.
 *
 * Same score sets, sequences, masks and pair order as tim_compare.  With
 * d = double(C) - double(A) per active token, each sequence gets:
 *   abs_q50/abs_q95/abs_q99[p]  quantiles of |left - right| for pair p,
 *       linear interpolation between order statistics: h = (n-1) q,
 *       Q = x[floor h] + (h - floor h) (x[floor h + 1] - x[floor h])
 *       ("Diagnosing Training Inference Mismatch in LLM Reinforcement Learning",
 *       5. practical indicators: abs(delta_logprob) p50/p95/p99/max);
 *   prob_mae[p]     mean |exp(left) - exp(right)| ("Fault localization and
 *       mismatch bisect", Metric measurement basis: probability_mae);
 *   top1_flips[p]   active tokens whose top-1 ids differ (practical indicators:
 *       top-1 flip rate), -1 unless both top-1 arrays of the pair are given;
 *   log_ratio_sum = sum d, k1_sum = -sum d, k3_sum = sum(expm1(d) - d)
 *       (sequence rejection by sum_t K1 / K3 of the correction ratio,
 *       "Diagnosing ...", 3. TIS);
 *   seq_tis = cap if sum d > ln(cap) else exp(sum d) (sequence TIS, same section);
 *   ratio_err_mean = mean |exp(d) - 1| (practical indicators: PPO ratio error);
 *   mis_mean = mean of w 1[mis_lo <= w <= mis_hi] with w = exp(d), the interval
 *       test taken as ln(mis_lo) <= d <= ln(mis_hi); mis_kept = tokens inside
 *       ("Rollout-Training Mismatch in LLM RL", section 2.1, w_MIS);
 *   w2_mean = mean exp(2 d) (E_q[w^2] = exp D_2(p||q), same page, section 5.3).
 * The quantiles are exact for a sequence of any length; a sequence with more
 * than 16384 active tokens takes a slower select that re-reads its scores on
 * every pass instead of holding its keys in shared memory.
 * Flags and errors as for tim_compare.
 *
 * Arguments: those of tim_compare, plus top1_gen / top1_replay / top1_train
 * (int32 [T] device arrays or NULL), mis_lo / mis_hi (finite,
 * 0 < mis_lo <= mis_hi), out_diag (tim_seq_diag [n_seq], device memory).
 * The workspace (tim_compare_diag_workspace_size(T, n_seq) bytes, zero-
 * initialised once) holds the status word, the per-sequence part bookkeeping
 * and, for sequences with more than 16384 active tokens, the quantile keys past
 * the first 16384 (24 bytes per token of T).
 * ------------------------------------------------------------------------ */

typedef struct tim_seq_diag {
  int64_t n_valid;
  double abs_q50[3];
  double abs_q95[3];
  double abs_q99[3];
  double prob_mae[3];
  int64_t top1_flips[3];
  double log_ratio_sum;
  double k1_sum;
  double k3_sum;
  double seq_tis;
  double ratio_err_mean;
  double mis_mean;
  int64_t mis_kept;
  double w2_mean;
  int32_t flags;
  int32_t reserved;
} tim_seq_diag;

size_t tim_compare_diag_workspace_size(int64_t T, int32_t n_seq);

tim_status tim_compare_diag(const float *lp_gen, const float *lp_replay, const float *lp_train,
                            const int32_t *top1_gen, const int32_t *top1_replay,
                            const int32_t *top1_train, const int64_t *seq_offsets,
                            int32_t n_seq, const uint8_t *mask, int64_t T, float tis_cap,
                            float mis_lo, float mis_hi, tim_seq_diag *out_diag, void *workspace,
                            size_t workspace_bytes, tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * tim_logprob without a caller-supplied workspace.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory: for example a scoring hook inside a
 * rollout or serving engine that has already claimed nearly all free device
 * memory for its own caches and pools (so cudaMalloc fails, and the engine's
 * allocator is not reachable from C), or latency-sensitive code that must not
 * call cudaMalloc/cudaFree because they can synchronise the device.
 *
 * Computes exactly what tim_logprob computes, with the same kernels, but keeps
 * its scratch (y, the per-vocabulary-tile records, the target logits and the
 * status word) in one 8 MiB device array owned by the library.  Every GPU
 * that loads the library holds that array until the process exits.  It
 * allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *
 * Limit: tim_logprob_workspace_size(T, d, V) must not exceed 8 MiB (8388608
 * bytes) -- e.g. up to 416 rows at d = 4096 or 384 rows at d = 5120 with
 * V = 151936; larger sizes return TIM_ERR_WORKSPACE with nothing enqueued.
 *
 * Arguments are those of tim_logprob (device pointers, same layouts and
 * alignment), plus out_status: a device int32 that receives this call's first
 * data-dependent error code (0 = none; TIM_ERR_TOKEN_RANGE, TIM_ERR_NONFINITE,
 * TIM_ERR_TIMEOUT), or NULL to skip it.
 *
 * The first call in each CUDA context (once per device in the usual case; again
 * after a cudaDeviceReset) performs a one-time set-up with that context current:
 * it looks up the device address of the array, which places the library's code
 * and the array on the device, and loads every kernel this path launches (the
 * CUDA runtime otherwise loads kernels lazily, at their first launch, and
 * loading takes device memory).  That set-up is the only point where device
 * memory is taken, so a caller that later claims the remaining free memory
 * should make its first call (a warm-up at any accepted size) before doing so,
 * and before any stream capture.  Later calls, at any accepted size, take no
 * device memory.  All calls on a device share the one array and it
 * keeps the previous call's contents (each call clears the status word it
 * needs zeroed): calls whose work overlaps on the GPU -- on different streams,
 * or from different threads -- race on the array and must be serialised by the
 * caller, for instance by issuing them on one stream.
 * ------------------------------------------------------------------------ */
tim_status tim_logprob_noalloc(const void *hidden, const void *gamma, const void *W,
                               const int32_t *token_ids, int64_t T, int32_t d, int32_t V,
                               float temperature, float eps, float *out_logprob, float *out_lse,
                               int32_t *out_top1, int32_t *out_status, tim_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Self-test of the bounded waits (the pages have no counterpart: it exercises
 * this library's own failure detection).  Every mbarrier wait in the LM-head
 * kernel gives up after a time limit, records TIM_ERR_TIMEOUT in the status
 * word, winds the CTA down (waiting, bounded, for its own copies and MMAs in
 * flight) and frees its tensor memory, so the CUDA context stays usable.  This
 * call runs that kernel on a 128 x 64 x 512 problem with its TMA producer
 * stalled: nothing ever arrives on the pipeline barriers, the waits run out
 * after limit_ms (1 .. 2000), and tim_status_sync(workspace, stream) then
 * returns TIM_ERR_TIMEOUT.  No fault, trap or unbounded wait is involved.
 * workspace: tim_selftest_workspace_size() bytes, zero-initialised once.
 * ------------------------------------------------------------------------ */
size_t tim_selftest_workspace_size(void);

tim_status tim_selftest_wait_timeout(int32_t limit_ms, void *workspace, size_t workspace_bytes,
                                     tim_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TIM_H_ */
