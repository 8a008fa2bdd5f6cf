/*
 * sv.h -- C ABI of the GB300 speculative-decoding verify library (libsv.so).
 *
 * The library computes the verify step of block speculative decoding on one
 * GPU: the per-request target distribution (temperature, top-k, top-p), the
 * chain rejection test against the draft distribution, the residual / bonus
 * resample, and the confidence-scheduled verify-budget planner that lays the
 * ragged windows out.  Pages cited by title and section:
 *
 *   [P2] jianc99/sglang PR #8 (adaptive verification for DFLASH), commit
 *        "build_speculative_verify_target_probs ...": per-row temperature,
 *        top-k and top-p on [rows, vocab] logits; top-k on the raw logits
 *        commutes with a positive temperature; deterministic ties; and the
 *        DFLASH adaptive-verification commit: accept paths stop at the
 *        planned verify length, the bonus comes from the last verified row.
 *   [P3] local-inference-lab/rtx6kpro, dspark-upstream-consolidation.md,
 *        "Identical rejection scheme": greedy accepts iff draft == target
 *        argmax; temperature > 0 runs the Leviathan ratio test; block
 *        verification reweights the residual mass.
 *   [P4] NVIDIA/TensorRT-LLM PR #17056: description, "Scheduler" (cumulative
 *        product survival, global survival rank, value-independent
 *        tie-break, sync-free) and "Ragged (per-request) verification"
 *        (qo_indptr, token bucket); review commit "Cost model" (tokens
 *        submitted = bs * (verify_len + 1)); the `_rejection_buffers_valid`
 *        commit (padding rows never accepted, accept clamped to verify_lens).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Pointers marked (device) are device memory owned by the caller; the
 *    library allocates and frees nothing.  Scratch comes from the caller's
 *    workspace `ws` of `ws_bytes` (>= sv_workspace_size(...)), 256-byte
 *    aligned, which must not be shared by calls that run concurrently.
 *  - Every call is asynchronous on `stream`: no host synchronisation and no
 *    device-to-host copy, so every call can be captured in a CUDA graph.
 *  - Argument errors the host can see (null pointers, sizes, dtype, small
 *    workspace) return a status before any launch.  Data-dependent errors
 *    (non-finite logits, bad tokens, bad per-request parameters, inconsistent
 *    ragged windows) are reported per position in `row_status`; the affected
 *    request gets accept_len = 0, num_emitted = 0 and out_tokens all -1.
 *    Unsupported combinations are refused (status bit SV_ROW_UNSUPPORTED),
 *    never silently degraded.
 *  - A launch failure returns SV_ERR_CUDA (cudaGetLastError after launch).
 *  - Logits rows are contiguous along the vocabulary; `row_stride` is in
 *    elements.
 *  - Sampling parameters are per request (device arrays of length n_req):
 *      temperature == 0 -> greedy (argmax, lowest index wins ties);
 *      top_k <= 0 or >= vocab -> top-k off (top_k may be NULL: off);
 *      top_p >= 1 -> top-p off (top_p may be NULL: off);
 *      temperature < 0 / NaN / inf, or top_p <= 0 / NaN -> SV_ROW_BAD_PARAM.
 *  - Target distribution p of a row (T > 0): tokens ordered by (logit desc,
 *    index asc), the first k kept (top-k), then the shortest prefix whose
 *    mass exp((l - m) / T) reaches top_p times the top-k mass (the crossing
 *    token is kept), p = mass / kept mass.  The draft distribution q is the
 *    same transform of the draft logits with the same request parameters.
 *  - Uniforms: Philox4x32-10 with key (seed low 32 bits, seed high 32 bits)
 *    and counter (request, position, draw, 0); u = (word0 >> 8) * 2^-24.
 *    draw 0 decides acceptance at a position, draw 1 samples the token
 *    emitted at the first rejection (residual) or after full acceptance
 *    (bonus).  request = the request's index in the call.
 */
#ifndef SV_H
#define SV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is struct CUstream_st* */
typedef struct CUstream_st* sv_stream_t;

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1, /* null pointer, negative/zero size, inconsistent sizes */
    SV_ERR_WORKSPACE = 2,   /* ws NULL, misaligned or smaller than sv_workspace_size */
    SV_ERR_CUDA = 3,        /* a kernel launch failed                                */
    SV_ERR_UNSUPPORTED = 4  /* a size or layout the library does not handle         */
} sv_status_t;

typedef enum { SV_DTYPE_BF16 = 0, SV_DTYPE_F32 = 1 } sv_dtype_t;

/* Per-position / per-row status bits. */
enum {
    SV_ROW_NONFINITE = 1,    /* NaN or +inf logit in a row that is read            */
    SV_ROW_EMPTY = 2,        /* sampling row whose logits are all -inf             */
    SV_ROW_BAD_TOKEN = 4,    /* draft token outside [0, vocab)                     */
    SV_ROW_BAD_PARAM = 8,    /* invalid temperature / top_p for the request        */
    SV_ROW_BAD_LAYOUT = 16,  /* ragged window does not match qo_indptr / bucket    */
    SV_ROW_Q_ZERO = 32,      /* informational: q(d) == 0 at a tested position      */
    SV_ROW_RESID_ZERO = 64,  /* informational: empty residual, sampled from p      */
    SV_ROW_UNSUPPORTED = 128, /* combination the library refuses (sv_verify_*)  */
    SV_ROW_TIMEOUT = 256      /* a bounded wait on a bulk copy gave up: rows of the
                                 call were not processed (never seen in practice) */
};
#define SV_ROW_ERROR_MASK (SV_ROW_NONFINITE | SV_ROW_EMPTY | SV_ROW_BAD_TOKEN | SV_ROW_BAD_PARAM | \
                           SV_ROW_BAD_LAYOUT | SV_ROW_UNSUPPORTED | SV_ROW_TIMEOUT)

/* Host-side promises about a batch's sampling parameters (sv_sampling_t.flags).
 *   SV_SAMPLING_SMALL_TOPK  every request is greedy (T == 0) or keeps at most
 *       32 tokens by top-k (1 <= top_k <= 32).  The verify and row calls then
 *       launch only their prep, the one-pass row kernel and the chain (or row
 *       output) kernels: the full-vocabulary histogram kernels and the
 *       full-row resample, which such a batch never needs, are not launched.
 *       A request that breaks the promise is refused: SV_ROW_UNSUPPORTED (at
 *       position 0 of a verify request, accept_len = num_emitted = 0; in the
 *       row's descriptor for sv_build_target_probs); the other requests are
 *       not affected.  sv_estimator_predict ignores the flag (its features take
 *       greedy requests at T = 1 over the whole row), and so does
 *       sv_verify_block (it keeps its full launch sequence). */
enum { SV_SAMPLING_SMALL_TOPK = 1 };

typedef struct {
    const float* temperature; /* (device) [n_req]; required                       */
    const int32_t* top_k;     /* (device) [n_req] or NULL                         */
    const float* top_p;       /* (device) [n_req] or NULL                         */
    int32_t flags;            /* (host) SV_SAMPLING_* promises, 0 for none        */
} sv_sampling_t;

/* Descriptor of one row's distribution (32 bytes).  With T = temperature,
 * p(x) = exp((l_x - max_logit) / T - log_norm) if x is kept, else 0, where x
 * is kept iff l_x > cutoff_logit, or l_x == cutoff_logit and fewer than
 * cutoff_ties tokens with that logit precede x.  Greedy rows (T == 0) have
 * kept = 1, cutoff = max_logit, p one-hot at argmax. */
typedef struct {
    float max_logit;     /* m = max logit                                     */
    float log_norm;      /* ln of sum over kept tokens of exp((l - m) / T)    */
    float cutoff_logit;  /* logit of the last kept token in sorted order      */
    int32_t cutoff_ties; /* kept tokens whose logit equals cutoff_logit       */
    int32_t kept;        /* number of kept tokens                             */
    int32_t argmax;      /* lowest index holding m                            */
    int32_t status;      /* SV_ROW_* bits of this row                         */
    float temperature;   /* T the row was built with                          */
} sv_row_desc_t;

/* Workspace bytes for a verify call with n_req requests, at most k_max drafted
 * positions each, and this vocabulary; for sv_build_target_probs pass
 * (rows, 0, vocab); for sv_plan_budget pass (n_req, K, 0).  0 on overflow. */
size_t sv_workspace_size(int n_req, int k_max, int vocab);

/* Workspace bytes for sv_verify_block (it keeps up to k_max + 1 full-row jobs
 * per request and each request's weights and residual sums); 0 for sizes
 * the library does not handle. */
size_t sv_workspace_size_block(int n_req, int k_max, int vocab);

/* Human-readable name of a status code (static string). */
const char* sv_status_string(sv_status_t status);

/*
 * Confidence-scheduled verify-budget planner ([P4] "Scheduler", "Ragged").
 *   conf        (device) fp32 [n_req, ld_conf]: c_{r,i} = chance that drafted
 *               position i of request r survives verification; NaN -> 0,
 *               clamped to [0, 1].
 *   draft_len   (device) [n_req] drafted positions per request, or NULL (= K);
 *               values outside [0, K] are clamped and reported in *status.
 *   Survival s_{r,i} = prod_{l <= i} c_{r,l}, in fp32, left to right.  The
 *   N_sel = min(budget_tokens - n_req, sum_r K_r) candidates (r, i) ranked
 *   first by (s desc, i asc, r asc) are verified; verify_lens[r] counts r's
 *   (a per-request prefix); each request submits verify_lens[r] + 1 tokens
 *   (one anchor / bonus row).  qo_indptr [n_req + 1] is the exclusive prefix
 *   sum of the windows, *total_tokens = qo_indptr[n_req] <= budget_tokens;
 *   rows [total_tokens, bucket_tokens) are padding.
 *   Outputs verify_lens [n_req], qo_indptr [n_req + 1], total_tokens [1],
 *   status [1] (device; status may be NULL).
 *   Errors: SV_ERR_INVALID_ARG if n_req < 1, K < 0, ld_conf < K,
 *   budget_tokens < n_req or bucket_tokens < budget_tokens.
 */
sv_status_t sv_plan_budget(const float* conf, int ld_conf, const int32_t* draft_len, int n_req, int K,
                           int budget_tokens, int bucket_tokens, int32_t* verify_lens, int32_t* qo_indptr,
                           int32_t* total_tokens, int32_t* status, void* ws, size_t ws_bytes,
                           sv_stream_t stream);

/*
 * Target-distribution build for `rows` logits rows ([P2]).
 *   logits        (device) [rows, row_stride] of dtype `dt`.
 *   row_to_req    (device) [rows] request of each row (index into the
 *                 n_req-long sampling arrays), or NULL: row r uses request r
 *                 (then n_req must be >= rows).  An index outside [0, n_req)
 *                 gives the row SV_ROW_BAD_PARAM.
 *   token_per_row (device) [rows] or NULL; prob_of_token (device) [rows] fp32
 *                 receives p(token) for rows with a token (may be NULL).
 *   desc          (device) [rows] descriptors (may be NULL).
 *   dense_probs   (device) [rows, vocab] fp32 or NULL: the full distribution
 *                 (a test aid; it writes rows * vocab floats).
 */
sv_status_t sv_build_target_probs(const void* logits, sv_dtype_t dt, int64_t row_stride, int rows, int vocab,
                                  const int32_t* row_to_req, int n_req, sv_sampling_t sp, const int32_t* token_per_row,
                                  float* prob_of_token, sv_row_desc_t* desc, float* dense_probs, void* ws,
                                  size_t ws_bytes, sv_stream_t stream);

/*
 * Verify in the uniform layout ([P3] acceptance, [P2] cap and bonus).
 *   target_logits (device) [n_req, K + 1, vocab]; draft_logits (device)
 *   [n_req, K, vocab] (may be NULL when every request is greedy); both row
 *   stride = vocab.  draft_tokens (device) [n_req, K].  verify_len (device)
 *   [n_req] or NULL (= K): request r tests positions j < v_r only (the
 *   "cap-accept" mode: the dense window is read, acceptance stops at v_r).
 *   For j < v_r: greedy accepts iff d_j == argmax_j; otherwise accepts iff
 *   u(r, j, 0) < p_j(d_j) / q_j(d_j) (q == 0: accept iff p > 0).  a = first
 *   rejection or v_r.  Emitted token t: greedy -> argmax_a; sampling, a < v_r
 *   -> inverse CDF (index order) of max(0, p_a - q_a) with u(r, a, 1) (of p_a
 *   if that mass is zero); a == v_r -> inverse CDF of p_{v_r} with u(r, a, 1).
 *   Outputs (device): accept_len [n_req] = a; out_tokens [n_req, K + 1] =
 *   d_0 .. d_{a-1}, t, then -1; num_emitted [n_req] = a + 1; row_status
 *   [n_req, K + 1] or NULL: OR of the position's target row, draft row and
 *   token bits.
 *   bf16 and fp32 logits take every sampling combination: kept sets of up to
 *   32 tokens are listed by the one-pass row kernel, larger ones (bf16) by
 *   exact per-value histograms or (fp32) by a radix descent on the 32-bit
 *   order keys with exact fixed-point masses, and their tokens are drawn by
 *   a full-row resample.  sp.flags = SV_SAMPLING_SMALL_TOPK skips the
 *   full-vocabulary kernels (see sv_sampling_t); sv_verify_ragged takes it
 *   the same way, sv_verify_block ignores it.
 */
sv_status_t sv_verify_chain(const void* target_logits, const void* draft_logits, sv_dtype_t dt, int n_req, int K,
                            int vocab, const int32_t* draft_tokens, const int32_t* verify_len, sv_sampling_t sp,
                            uint64_t seed, int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                            int32_t* row_status, void* ws, size_t ws_bytes, sv_stream_t stream);

/*
 * Block verification over the uniform layout (local-inference-lab/rtx6kpro
 * dspark-upstream-consolidation.md: rejection_sample_method "block", joint
 * block acceptance with residual-mass reweighting; the steps are those of
 * Sun et al., "Block Verification Accelerates Speculative Decoding", 2024).
 * Arguments, layouts, outputs and errors as sv_verify_chain.  Greedy
 * requests take the chain's rule (the two agree at temperature 0).  For a
 * sampling request with window v and drafts d_j (p_j, q_j its rows'
 * distributions, u(r, j, k) its Philox uniforms):
 *   w_0 = 1, w_j = min(w_{j-1} p_{j-1}(d_{j-1}) / q_{j-1}(d_{j-1}), 1);
 *   H_j = sum_x max(w_j p_j(x) - q_j(x), 0), h_j = H_j / (H_j + 1 - w_j)
 *   (1 when the denominator is 0) for j < v, h_v = w_v;
 *   accept_len = the largest j in 1..v with u(r, j-1, 0) < h_j, else 0;
 *   the emitted token after the accepted drafts is drawn by inverse CDF in
 *   index order with u(r, accept_len, 1) from max(w_a p_a - q_a, 0) (a =
 *   accept_len < v; an empty residual falls back to p_a with
 *   SV_ROW_RESID_ZERO) or from p_v.  q(d) == 0 makes the ratio +inf if
 *   p(d) > 0, else 0 (SV_ROW_Q_ZERO).  With v = 1 this is exactly
 *   sv_verify_chain.  Kept sets of any size: for sampling requests whose kept
 *   sets are not listed (more than 32 tokens) the sums H_j and the draw run
 *   over whole rows in exact 62-bit fixed point, with w p floored as a 64-bit
 *   fraction.  The workspace must hold sv_workspace_size_block(n_req, K,
 *   vocab) bytes.  fp32 logits: as sv_verify_chain.
 */
sv_status_t sv_verify_block(const void* target_logits, const void* draft_logits, sv_dtype_t dt, int n_req, int K,
                            int vocab, const int32_t* draft_tokens, const int32_t* verify_len, sv_sampling_t sp,
                            uint64_t seed, int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                            int32_t* row_status, void* ws, size_t ws_bytes, sv_stream_t stream);

/*
 * Verify in the ragged layout ([P4] "Ragged (per-request) verification",
 * `_rejection_buffers_valid`).  Request r's target rows are rows
 * qo_indptr[r] .. qo_indptr[r] + verify_lens[r] of target_logits (device,
 * [bucket_tokens, vocab]); rows past the last window are padding and never
 * read.  Draft logits stay in the drafted block layout (device, [n_req,
 * K_max, vocab]; NULL if every request is greedy): the block is drafted in
 * full and only the number of verified positions changes.  draft_tokens
 * (device) [n_req, K_max].  A window that is not qo_indptr[r + 1] -
 * qo_indptr[r] == verify_lens[r] + 1 rows wide, or leaves [0,
 * bucket_tokens), gets SV_ROW_BAD_LAYOUT.  Everything else as
 * sv_verify_chain with v_r = verify_lens[r]; outputs are [n_req, K_max + 1].
 */
sv_status_t sv_verify_ragged(const void* target_logits, const void* draft_logits, sv_dtype_t dt, int n_req,
                             int K_max, int vocab, int bucket_tokens, const int32_t* qo_indptr,
                             const int32_t* verify_lens, const int32_t* draft_tokens, sv_sampling_t sp,
                             uint64_t seed, int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                             int32_t* row_status, void* ws, size_t ws_bytes, sv_stream_t stream);

/*
 * Verify budget from a profiled step-cost table, then the plan for it
 * ([P4] description, "What is here / Planner": the budget is the argmax of
 * tau / cost over a profiled step-cost table, a global argmax because the cost
 * curve is a staircase; review commit, "Cost model": the table is indexed by
 * tokens submitted, bs * (verify_len + 1), and carries a fixed per-step
 * overhead and an optional batch-size staircase).  Everything stays on the
 * device: the chosen budget feeds the planner without a host readback.
 *   conf, ld_conf, draft_len, n_req, K: as sv_plan_budget.
 *   cost_tokens (device) int32 [n_cost], strictly ascending: shelf j holds
 *               steps that submit up to cost_tokens[j] tokens ...
 *   cost_ms     (device) fp32 [n_cost]: ... and such a step costs cost_ms[j].
 *   fixed_overhead_ms: per-step cost that does not depend on the budget.
 *   batch_sizes (device) int32 [n_batch] ascending, batch_overhead_ms (device)
 *               fp32 [n_batch]: the overhead of a batch of n_req requests is
 *               that of the first entry with batch_sizes >= n_req (the last
 *               entry above them all).  n_batch may be 0 (pointers NULL).
 *   tau(B) = n_req + the sum of the B - n_req largest survivals (the expected
 *   tokens a step that submits B tokens emits); cost(B) = cost_ms of the first
 *   shelf with cost_tokens >= B, plus the fixed and batch overheads.  The
 *   budget B in [n_req, n_req + min(sum K_r, bucket_tokens - n_req)] with the
 *   largest tau(B) / cost(B) is chosen, the larger B on ties.  n_cost == 0 or
 *   no shelf that holds n_req tokens: no trimming (the largest B), bit 2 of
 *   *budget_status; a table that is not strictly ascending or has a negative
 *   or non-finite cost or overhead: no trimming, bit 4; bit 1: a draft
 *   length was clamped.
 *   Outputs budget_out [1] (device, the chosen budget), budget_status [1]
 *   (device, may be NULL), and the plan for that budget exactly as
 *   sv_plan_budget writes it.  Workspace: sv_workspace_size(n_req, K, 0).
 *   Errors: SV_ERR_INVALID_ARG for the sv_plan_budget argument errors (with
 *   bucket_tokens < n_req in place of the budget checks), a NULL budget_out or
 *   a NULL table array of nonzero length; SV_ERR_UNSUPPORTED for n_req * K >
 *   16384 candidates or more than 4096 shelves or batch entries.
 */
sv_status_t sv_plan_budget_cost(const float* conf, int ld_conf, const int32_t* draft_len, int n_req, int K,
                                const int32_t* cost_tokens, const float* cost_ms, int n_cost, float fixed_overhead_ms,
                                const int32_t* batch_sizes, const float* batch_overhead_ms, int n_batch,
                                int bucket_tokens, int32_t* budget_out, int32_t* budget_status, int32_t* verify_lens,
                                int32_t* qo_indptr, int32_t* total_tokens, int32_t* status, void* ws, size_t ws_bytes,
                                sv_stream_t stream);

/*
 * Acceptance against trimming for one verify step ([P4], the commit that
 * adds trim_regret_rate): a trimmed request (verify_lens[r] < K_r) that
 * accepted its whole window was still alive at the cut, so the cut cost
 * acceptance; one that stopped inside its window lost nothing.
 *   accept_len, num_emitted (device) [n_req]: a verify call's outputs;
 *   requests with num_emitted == 0 (errors) are not counted.
 *   verify_lens (device) [n_req] or NULL (every window K_r: nothing trimmed).
 *   draft_len   (device) [n_req] or NULL (= K); clamped to [0, K].
 *   out (device) int64 [4]: tokens emitted sum(accept_len + 1), tokens
 *   submitted sum(verify_lens + 1), requests trimmed, trimmed requests that
 *   accepted their whole window.
 *   Errors: SV_ERR_INVALID_ARG if n_req < 1, K < 0, or a required pointer is
 *   NULL.
 */
sv_status_t sv_verify_stats(const int32_t* accept_len, const int32_t* num_emitted, const int32_t* verify_lens,
                            const int32_t* draft_len, int n_req, int K, int64_t* out, sv_stream_t stream);

/*
 * Online acceptance estimator (jianc99/sglang PR #8, DFLASH adaptive-
 * verification commits): the confidence source of the planner for drafts
 * without a confidence head.  p_k = sigmoid(slope * x_k + bias_k), x_k =
 * logit(q_max) of the draft distribution at position k, clamped to +-40.
 * q is the request's transform (temperature, top-k, top-p) of draft row k --
 * the q verification uses -- at temperature 1 for greedy requests; q_max = 1/z
 * (z the kept mass relative to the top token), so x = -ln(z - 1).
 * The state is caller-owned device memory of sv_estimator_state_bytes(K)
 * bytes, doubles laid out as [0] slope, [1..K] bias, then the Newton
 * statistics (g_a, H_aa, g_k x K, H_ak x K, H_kk x K, observations, calls).
 * Everything runs on the stream without host synchronisation.
 */
size_t sv_estimator_state_bytes(int K);                          /* 0 unless 1 <= K <= 63 */

/* slope 0.5, every bias -0.2, statistics cleared. */
sv_status_t sv_estimator_init(double* state, int K, sv_stream_t stream);

/*
 * Features and predictions for draft logits (device, [n_req, K, vocab], bf16
 * or fp32): x_out, p_out (device) fp32 [n_req, K].
 * p_out is the planner's conf input (sv_plan_budget / sv_plan_budget_cost).
 * A row with an error gives x = p = NaN (the planner reads NaN as 0).
 * Workspace: sv_workspace_size(n_req * K, 0, vocab).
 */
sv_status_t sv_estimator_predict(const void* draft_logits, sv_dtype_t dt, int n_req, int K, int vocab,
                                 sv_sampling_t sp, const double* state, float* x_out, float* p_out, void* ws,
                                 size_t ws_bytes, sv_stream_t stream);

/*
 * Bytes of the draft-row results sv_estimator_predict_q leaves for
 * sv_verify_chain_q: n_req * K records of the library's row result (0 for
 * sizes outside 1 <= K <= 63, n_req * K <= 2^22).
 */
size_t sv_q_rows_bytes(int n_req, int K);

/*
 * sv_estimator_predict that also keeps what it computed for the verify that
 * follows (jianc99/sglang PR #8, DFLASH adaptive-verification commits: the
 * feature logit(q_max) is a by-product of the draft distribution).  Besides
 * x_out and p_out it writes, for every draft row (r, j), the row's
 * distribution under request r's parameters (greedy requests at T = 1) and
 * q of draft token draft_tokens[r, j] into q_rows (device, 16-byte aligned,
 * sv_q_rows_bytes(n_req, K) bytes).  draft_tokens (device) [n_req, K].
 * Workspace as sv_estimator_predict.
 */
sv_status_t sv_estimator_predict_q(const void* draft_logits, sv_dtype_t dt, int n_req, int K, int vocab,
                                   sv_sampling_t sp, const double* state, const int32_t* draft_tokens, float* x_out,
                                   float* p_out, void* q_rows, void* ws, size_t ws_bytes, sv_stream_t stream);

/*
 * sv_verify_chain with the draft rows' distributions taken from q_rows, made
 * by sv_estimator_predict_q from the same draft logits, draft tokens and
 * sampling parameters (for sampling requests the two transforms are the
 * same): only the target rows are streamed.  draft_logits is still required
 * for sampling requests -- the full-row resample of a request whose kept set
 * is not listed reads its draft row at the emitted position.  Everything
 * else, outputs included, as sv_verify_chain (K >= 1).
 */
sv_status_t sv_verify_chain_q(const void* target_logits, const void* draft_logits, sv_dtype_t dt, int n_req, int K,
                              int vocab, const int32_t* draft_tokens, const int32_t* verify_len, sv_sampling_t sp,
                              uint64_t seed, const void* q_rows, int32_t* accept_len, int32_t* out_tokens,
                              int32_t* num_emitted, int32_t* row_status, void* ws, size_t ws_bytes,
                              sv_stream_t stream);

/*
 * After a verify call: request r's positions 0 .. min(accept_len[r],
 * v_r - 1) are observed (label 1 below accept_len, 0 for the first rejected
 * one; v_r = verify_lens[r], or K when NULL); requests with num_emitted == 0
 * and non-finite features are skipped.  The Newton statistics at the current
 * coefficients accumulate in the state; every refit_every calls (0: never)
 * one ridge (1e-3) Newton step on the arrowhead system, damped by n / (n + 50)
 * for n observations, updates the coefficients: a slope step that would make
 * the slope negative is halved up to 8 times and dropped if it still does;
 * the intercepts step given the slope step taken; non-finite steps are
 * dropped; the statistics are then cleared.  One CTA reduces in a fixed
 * order, so identical inputs give identical coefficients.
 */
sv_status_t sv_estimator_observe(double* state, const float* x, const int32_t* accept_len, const int32_t* num_emitted,
                                 const int32_t* verify_lens, int n_req, int K, int refit_every, sv_stream_t stream);

/*
 * sv_verify_chain without a workspace argument.  The pages have no
 * counterpart: this is for callers that cannot allocate device memory where
 * they verify -- code running while a CUDA graph is captured (cudaMalloc is
 * refused in a global-mode capture), serving runtimes whose device memory is
 * one pool reserved at start-up with no allocation allowed on the decode path,
 * and plugins inside a host engine that owns all memory.  Arguments, outputs
 * and results are those of sv_verify_chain; the scratch is a static 32 MiB
 * device array in the library, resident on each GPU that loads it until the
 * process exits.  Sizes whose sv_workspace_size(n_req, K, vocab) exceeds
 * 32 MiB return SV_ERR_UNSUPPORTED before any launch (the benchmark's
 * 128 x 8 x 248,320 batch needs about 6 MiB).  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  All calls share
 * the array: calls that overlap on the GPU race, so serialise them.  Nothing
 * is allocated or freed.
 */
sv_status_t sv_verify_chain_noalloc(const void* target_logits, const void* draft_logits, sv_dtype_t dt, int n_req,
                                    int K, int vocab, const int32_t* draft_tokens, const int32_t* verify_len,
                                    sv_sampling_t sp, uint64_t seed, int32_t* accept_len, int32_t* out_tokens,
                                    int32_t* num_emitted, int32_t* row_status, sv_stream_t stream);

/*
 * Vocabulary-sharded verify (jianc99/sglang PR #8, DFLASH adaptive-
 * verification commit: the compact scatter works on a vocabulary shard and
 * the target-verify gather is deferred).  The logits of a step may live split
 * along the vocabulary, each shard [v0, v1) on its own device (tensor-parallel
 * lm heads).  Each shard reduces its slice of every row of the window to one
 * fixed-width record; the records of all shards are exchanged once (any
 * collective that gathers equal-sized buffers, e.g. an all-gather: the size
 * depends only on n_req and K, never on the data); every rank then merges
 * them and finishes the step exactly as sv_verify_chain would on the whole
 * rows -- the same accepted lengths, tokens and statuses.  Served: greedy
 * requests and requests whose kept set is listed (top-k <= 32, with or
 * without top-p); a request with a larger kept set gets SV_ROW_UNSUPPORTED
 * (nothing accepted or emitted).
 *
 * sv_shard_record_bytes: bytes of one record (264): its row's top-32
 * composite keys (logit order key above, whole-vocabulary index inverted
 * below, descending) with their count and status bits.
 */
size_t sv_shard_record_bytes(void);

/*
 * One shard's records.  target_shard (device) [n_req, K + 1, v1 - v0] and
 * draft_shard (device) [n_req, K, v1 - v0] (NULL if every request is greedy):
 * columns v0 .. v1 - 1 of the rows sv_verify_chain takes, row stride v1 - v0;
 * 0 <= v0 < v1 <= vocab.  draft_tokens, verify_len and sp as sv_verify_chain
 * (tokens and top_k refer to the whole vocabulary).  records (device,
 * 16-byte aligned) [n_req * (2K + 1)] records of sv_shard_record_bytes(), one
 * per target position 0..K and draft position 0..K-1 of each request (slot
 * r (2K + 1) + j, then r (2K + 1) + K + 1 + j); slots outside a request's
 * window are left as they are and never read.  Workspace:
 * sv_workspace_size(n_req, K, v1 - v0).  Errors: SV_ERR_INVALID_ARG for NULL
 * pointers, sizes, a slice outside [0, vocab), a misaligned records buffer.
 */
sv_status_t sv_verify_chain_shard_rows(const void* target_shard, const void* draft_shard, sv_dtype_t dt, int n_req,
                                       int K, int vocab, int v0, int v1, const int32_t* draft_tokens,
                                       const int32_t* verify_len, sv_sampling_t sp, void* records, void* ws,
                                       size_t ws_bytes, sv_stream_t stream);

/*
 * The merge: records (device, 16-byte aligned) [n_shards][n_req * (2K + 1)]
 * records, the shards' sv_verify_chain_shard_rows outputs in any shard order
 * (shards must cover [0, vocab) without overlap).  The other arguments and
 * the outputs are those of sv_verify_chain.  Workspace: sv_workspace_size(
 * n_req, K, 1).
 */
sv_status_t sv_verify_chain_shard_merge(const void* records, int n_shards, int n_req, int K, int vocab,
                                        const int32_t* draft_tokens, const int32_t* verify_len, sv_sampling_t sp,
                                        uint64_t seed, int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                                        int32_t* row_status, void* ws, size_t ws_bytes, sv_stream_t stream);

/*
 * Measurement aid (not part of the method): when both are non-NULL, every
 * later sv_verify_chain / sv_verify_ragged / sv_build_target_probs call
 * records start_event (a cudaEvent_t) on its stream immediately before the
 * one-pass row-selection kernel and stop_event immediately after it, so a
 * caller can time that kernel alone with cudaEventElapsedTime.  Pass NULLs to
 * stop.  Process-wide; not for calls issued concurrently from several host
 * threads.  Always returns SV_OK.
 */
sv_status_t sv_set_timing_events(void* start_event, void* stop_event);

/*
 * Measurement aid (not part of the method), as sv_set_timing_events but
 * around the exact-histogram row kernels (rows whose kept set can exceed 32
 * tokens: the one-CTA-per-row kernel and the cluster kernel that takes the
 * rows it hands on), recorded on bf16 calls.  Pass NULLs to stop.
 * Process-wide; not for calls issued concurrently from several host
 * threads.  Always returns SV_OK.
 */
sv_status_t sv_set_hist_timing_events(void* start_event, void* stop_event);

#ifdef __cplusplus
}
#endif

#endif /* SV_H */
