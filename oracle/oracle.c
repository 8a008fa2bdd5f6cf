/*
 * oracle.c -- plain CPU definition of the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE.  This file is the checker the CUDA library is compared
 * against.  Only the tests, the package smoke check and the benchmark's CPU
 * baseline leg load it; no product code path calls it, and it shares no code,
 * header, table or constant generator with the CUDA sources.
 *
 * Everything is single-threaded, in double precision, in the order the
 * definition states: no blocking, no fusion, no reordering.  The steps and
 * where they come from (pages cited by title and section):
 *
 *  - Target distribution (temperature, top-k, top-p, normalise): jianc99/sglang
 *    PR #8, commit "build_speculative_verify_target_probs ..." -- top-k on the
 *    raw logits commutes with a positive temperature, the tie choice at the
 *    top-k boundary is deterministic, the probabilities are unchanged.
 *  - Acceptance: local-inference-lab/rtx6kpro dspark-upstream-consolidation.md,
 *    section "Identical rejection scheme" -- greedy accepts iff the draft equals
 *    the target argmax, temperature > 0 runs the Leviathan ratio test.
 *  - Residual resample / bonus from the last verified row: same page
 *    ("residual-mass reweighting") and jianc99/sglang PR #8, the DFLASH
 *    adaptive-verification commit ("The bonus comes from the last verified
 *    row"; accept paths stop at the planned verify length).
 *  - Planner: NVIDIA/TensorRT-LLM PR #17056, description section
 *    "What is here / Scheduler" (cumulative product survival, global survival
 *    rank, value-independent tie-break) and "Ragged (per-request)
 *    verification" (qo_indptr, token bucket); review commit, section
 *    "Cost model" (tokens submitted = bs * (verify_len + 1)).
 *  - Ragged rejection: NVIDIA/TensorRT-LLM PR #17056, the
 *    `_rejection_buffers_valid` commit (padding rows can never be accepted,
 *    accepted count clamped to verify_lens).
 *  - Uniforms: Philox4x32-10, Salmon, Moraes, Dror, Shaw, "Parallel random
 *    numbers: as easy as 1, 2, 3", SC'11.
 *
 * Where the pages are silent, the reading taken is stated at the function
 * that takes it.
 */
#include <math.h>
#include <stdint.h>

/* ORC_PLANT selects a deliberate mistake for the tests that show each pin
 * catches one (0 = the oracle as defined; the tests build the others as
 * separate libraries):
 *   1 residual max(0, q - p) instead of max(0, p - q)
 *   2 top-p keeps the prefix before the crossing token
 *   3 argmax keeps the last occurrence of the maximum
 *   4 planner tie-break by request before position
 *   5 resample reuses the acceptance draw (draw 0)
 *   6 cost table looked up by drafted tokens only (the bonus row left out)
 *   7 budget by first descent of tau / cost instead of the global argmax
 *   8 trim regret counts requests that stopped inside their window
 *   9 block verification: residual and stopping masses without the weight
 *  10 estimator: every position of the window observed, not only up to the
 *     first rejection
 *  11 estimator: a slope step that crosses zero is dropped, not halved     */
#ifndef ORC_PLANT
#define ORC_PLANT 0
#endif
#include <stdlib.h>
#include <string.h>

/* Row / position status bits.  Bits 0..4 and 6 make a request an error. */
#define ORC_NONFINITE   1   /* NaN or +inf logit in a row that is read        */
#define ORC_EMPTY       2   /* sampling row whose logits are all -inf         */
#define ORC_BAD_TOKEN   4   /* draft token outside [0, vocab)                 */
#define ORC_BAD_PARAM   8   /* T < 0 or not finite; top_p NaN or <= 0        */
#define ORC_BAD_LAYOUT 16   /* ragged window inconsistent with the bucket     */
#define ORC_Q_ZERO     32   /* q(d) == 0 at a tested position (informational) */
#define ORC_RESID_ZERO 64   /* residual mass zero, sampled from p (informat.) */
#define ORC_ERROR_MASK (ORC_NONFINITE | ORC_EMPTY | ORC_BAD_TOKEN | ORC_BAD_PARAM | ORC_BAD_LAYOUT)

/* Near-tie flags per request: a decision whose margin is below the bound is
 * reported, and everything downstream of it in that request goes unchecked. */
#define ORC_FLAG_RATIO   1  /* |u - p/q| < 1e-6 (the bound the task states)   */
#define ORC_FLAG_CUTOFF  2  /* top-p prefix mass within 1e-9*Z1 of top_p*Z1   */
#define ORC_FLAG_INVCDF  4  /* u*W within 1e-9*W of a cumulative boundary     */
#define ORC_FLAG_RESID   8  /* residual mass W below 1e-9                     */

static const double RATIO_MARGIN = 1e-6;
static const double CUTOFF_MARGIN = 1e-9;
static const double INVCDF_MARGIN = 1e-9;
static const double RESID_MIN = 1e-9;

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 (Salmon et al., SC'11): ten rounds of two 32x32->64 products */
/* with the Weyl key schedule.                                               */
/* ------------------------------------------------------------------------- */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Uniform for (request, position, draw): key = seed split in two 32-bit
 * halves, counter = (request, position, draw, 0); u = (word0 >> 8) * 2^-24,
 * which is exact in fp32.  draw 0 = acceptance test, draw 1 = resample/bonus. */
double orc_uniform(uint64_t seed, uint32_t req, uint32_t pos, uint32_t draw)
{
    uint32_t ctr[4] = { req, pos, draw, 0u };
    uint32_t key[2] = { (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32) };
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------- */
/* C1: decode a logit to double.  dtype 0 = bf16 (upper half of an fp32),    */
/* dtype 1 = fp32.                                                           */
/* ------------------------------------------------------------------------- */
static double decode(const void* row, int dtype, int64_t i)
{
    if (dtype == 0) {
        uint16_t h = ((const uint16_t*)row)[i];
        uint32_t bits = (uint32_t)h << 16;
        float f;
        memcpy(&f, &bits, 4);
        return (double)f;
    }
    return (double)((const float*)row)[i];
}

typedef struct {
    double value;
    int64_t index;
} orc_entry_t;

/* Order tokens by (logit desc, index asc).  Doubles compare -0 == +0. */
static int cmp_entry(const void* a, const void* b)
{
    const orc_entry_t* x = (const orc_entry_t*)a;
    const orc_entry_t* y = (const orc_entry_t*)b;
    if (x->value > y->value) return -1;
    if (x->value < y->value) return 1;
    if (x->index < y->index) return -1;
    if (x->index > y->index) return 1;
    return 0;
}

typedef struct {
    double max_logit;    /* m                                                */
    double log_norm;     /* ln of sum over kept tokens of exp((l - m) / T)   */
    double cutoff_logit; /* logit of the last kept token in sorted order     */
    int32_t cutoff_ties; /* kept tokens whose logit equals cutoff_logit      */
    int32_t kept;        /* number of kept tokens                            */
    int32_t argmax;      /* smallest index holding m                         */
    int32_t status;      /* ORC_* bits                                       */
    double cut_margin;   /* top-p decision margin / Z1 (inf when top-p off)  */
    double z_rest;       /* kept mass after the first kept token, sum of     */
                         /* exp((l - m) / T) over kept tokens 2..kept        */
    int64_t next_index;  /* first token the final cut leaves out, in sorted  */
                         /* order, among the top-k kept ones (-1: none)     */
} orc_row_t;

static int bad_params(float T, float top_p)
{
    if (!(T >= 0.0f) || isinf(T)) return 1;     /* NaN, negative or +inf     */
    if (T == 0.0f) return 0;                    /* greedy ignores top-k/p    */
    if (!(top_p > 0.0f)) return 1;              /* NaN or <= 0               */
    return 0;
}

/*
 * C2 / C3: one row's target distribution.
 *   T == 0: greedy.  argmax = smallest index x with l_x = max; p is one-hot
 *           there (the T -> 0 limit).
 *   T  > 0: order tokens by (l desc, index asc); keep the first k if
 *           0 < k < V; e_x = exp((l_x - m) / T) over the kept tokens; Z1 = sum;
 *           if top_p < 1 keep the shortest prefix whose cumulative sum is
 *           >= top_p * Z1 (the token that crosses is kept, at least one token);
 *           p(x) = e_x / (sum over the final kept set).
 * probs (nullable, length V) receives p.  Returns the status bits.
 */
int orc_row_transform(const void* row, int dtype, int64_t vocab, float T, int32_t top_k, float top_p,
                      orc_row_t* out, double* probs)
{
    memset(out, 0, sizeof(*out));
    out->cut_margin = INFINITY;
    out->next_index = -1;
    if (probs)
        for (int64_t i = 0; i < vocab; ++i) probs[i] = 0.0;
    if (bad_params(T, top_p)) {
        out->status = ORC_BAD_PARAM;
        return out->status;
    }
    /* C1: NaN / +inf make the row an error; -inf is probability zero. */
    double m = -INFINITY;
    int64_t amax = 0;
    int found = 0;
    for (int64_t i = 0; i < vocab; ++i) {
        double l = decode(row, dtype, i);
        if (isnan(l) || (isinf(l) && l > 0)) {
            out->status |= ORC_NONFINITE;
            return out->status;
        }
        if (!found || l > m || (ORC_PLANT == 3 && l == m)) {
            m = l;
            amax = i;
            found = 1;
        }
    }
    out->max_logit = m;
    out->argmax = (int32_t)amax;
    if (T == 0.0f) {
        out->log_norm = 0.0;
        out->cutoff_logit = m;
        out->cutoff_ties = 1;
        out->kept = 1;
        if (probs) probs[amax] = 1.0;
        return out->status;
    }
    if (isinf(m)) {                 /* every logit is -inf: no distribution */
        out->status |= ORC_EMPTY;
        return out->status;
    }
    orc_entry_t* ord = (orc_entry_t*)malloc((size_t)vocab * sizeof(orc_entry_t));
    double* e = (double*)malloc((size_t)vocab * sizeof(double));
    for (int64_t i = 0; i < vocab; ++i) {
        ord[i].value = decode(row, dtype, i);
        ord[i].index = i;
    }
    qsort(ord, (size_t)vocab, sizeof(orc_entry_t), cmp_entry);
    int64_t kk = (top_k > 0 && (int64_t)top_k < vocab) ? (int64_t)top_k : vocab;
    double Td = (double)T;
    double z1 = 0.0;
    for (int64_t i = 0; i < kk; ++i) {
        e[i] = exp((ord[i].value - m) / Td);
        z1 += e[i];
    }
    int64_t kept = kk;
    if (top_p < 1.0f) {
        double target = (double)top_p * z1;
        double cum = 0.0, prev = 0.0;
        for (int64_t i = 0; i < kk; ++i) {
            prev = cum;
            cum += e[i];
            if (cum >= target) {
                kept = (ORC_PLANT == 2 && i > 0) ? i : i + 1;
                double below = target - prev;   /* > 0: prev did not reach  */
                double above = cum - target;    /* >= 0: cum reached        */
                out->cut_margin = (below < above ? below : above) / z1;
                break;
            }
        }
    }
    double z = 0.0;
    for (int64_t i = 0; i < kept; ++i) z += e[i];
    out->log_norm = log(z);
    for (int64_t i = 1; i < kept; ++i) out->z_rest += e[i];
    out->kept = (int32_t)kept;
    out->cutoff_logit = ord[kept - 1].value;
    int32_t ties = 0;
    for (int64_t i = 0; i < kept; ++i)
        if (ord[i].value == out->cutoff_logit) ++ties;
    out->cutoff_ties = ties;
    out->next_index = kept < kk ? ord[kept].index : -1;
    if (probs)
        for (int64_t i = 0; i < kept; ++i) probs[ord[i].index] = e[i] / z;
    free(ord);
    free(e);
    return out->status;
}

/*
 * C7: inverse CDF over weights w in index order.  W = sum of w in index
 * order; the result is the smallest x with cumulative > u * W; if rounding
 * leaves no such x, the largest x with w_x > 0.  *margin receives the
 * distance of u * W to the nearest cumulative boundary, divided by W.
 */
static int64_t inv_cdf(const double* w, int64_t n, double u, double* margin)
{
    double W = 0.0;
    int64_t last_pos = -1;
    for (int64_t x = 0; x < n; ++x) {
        W += w[x];
        if (w[x] > 0.0) last_pos = x;
    }
    double target = u * W;
    double cum = 0.0;
    for (int64_t x = 0; x < n; ++x) {
        double before = cum;
        cum += w[x];
        if (cum > target) {
            double a = target - before, b = cum - target;
            *margin = (a < b ? a : b) / W;
            return x;
        }
    }
    *margin = 0.0;
    return last_pos;
}

/*
 * Block verification (local-inference-lab/rtx6kpro dspark-upstream-
 * consolidation.md: rejection_sample_method "block", joint block acceptance
 * with residual-mass reweighting).  The pages name the method and measure
 * it; the steps are those of the published algorithm (Sun, Mendlovic,
 * Leviathan, Aharoni, Beirami, Ro, Suresh, "Block Verification Accelerates
 * Speculative Decoding", 2024), in this file's notation:
 *   w_0 = 1,  w_j = min(w_{j-1} * p_{j-1}(d_{j-1}) / q_{j-1}(d_{j-1}), 1)  (j = 1..v)
 *   H_j = sum_x max(w_j p_j(x) - q_j(x), 0),  h_j = H_j / (H_j + 1 - w_j)  (j < v)
 *   h_v = w_v;  accept length a = the largest j with eta_j < h_j (a >= 0)
 *   eta_j = u(r, j - 1, 0) (the acceptance draw of draft j - 1)
 *   next token: inverse CDF (index order, u(r, a, 1)) of max(w_a p_a - q_a, 0)
 *   when a < v, of p_v when a = v.
 * Readings: q(d) == 0 gives the ratio +inf when p(d) > 0 and 0 otherwise
 * (SV_ROW_Q_ZERO), a zero weight stays zero; a zero denominator gives h = 1;
 * eta_j < h_j is strict so that v = 1 is exactly the chain's test u < p / q;
 * an empty residual falls back to p_a (SV_ROW_RESID_ZERO).  Flags: an
 * |eta_j - h_j| below the ratio margin at a decided j, the residual and
 * inverse-CDF margins as in the chain.
 */
static int block_accept(double* const* P, double* const* Q, const int32_t* d, int v, int64_t vocab, uint64_t seed,
                        uint32_t req, int32_t* pos_status, int32_t* flags, double* p_tok, double* q_tok, int64_t* tok)
{
    double* wgt = (double*)malloc((size_t)(v + 1) * sizeof(double));
    double* h = (double*)malloc((size_t)(v + 1) * sizeof(double));
    wgt[0] = 1.0;
    for (int j = 1; j <= v; ++j) {
        const double p = P[j - 1][d[j - 1]], q = Q[j - 1][d[j - 1]];
        p_tok[j - 1] = p;
        q_tok[j - 1] = q;
        double r;
        if (q > 0.0) {
            r = p / q;
        } else {
            pos_status[j - 1] |= ORC_Q_ZERO;
            r = p > 0.0 ? INFINITY : 0.0;
        }
        const double x = wgt[j - 1] > 0.0 ? wgt[j - 1] * r : 0.0;
        wgt[j] = x < 1.0 ? x : 1.0;
    }
    for (int j = 0; j < v; ++j) {
#if ORC_PLANT == 9
        const double wj = 1.0;
#else
        const double wj = wgt[j];
#endif
        double H = 0.0;
        for (int64_t x = 0; x < vocab; ++x) {
            const double m = wj * P[j][x] - Q[j][x];
            H += m > 0.0 ? m : 0.0;
        }
        const double den = H + 1.0 - wgt[j];
        h[j] = den > 0.0 ? H / den : 1.0;
    }
    h[v] = wgt[v];
    int a = 0;
    for (int j = v; j >= 1; --j) {
        const double eta = orc_uniform(seed, req, (uint32_t)(j - 1), 0u);
        if (fabs(eta - h[j]) < RATIO_MARGIN) *flags |= ORC_FLAG_RATIO;
        if (eta < h[j]) {
            a = j;
            break;
        }
    }
    double* w = (double*)malloc((size_t)vocab * sizeof(double));
    if (a < v) {
#if ORC_PLANT == 9
        const double wa = 1.0;
#else
        const double wa = wgt[a];
#endif
        double W = 0.0;
        for (int64_t x = 0; x < vocab; ++x) {
            const double m = wa * P[a][x] - Q[a][x];
            w[x] = m > 0.0 ? m : 0.0;
            W += w[x];
        }
        if (W < RESID_MIN) *flags |= ORC_FLAG_RESID;
        if (!(W > 0.0)) {
            pos_status[a] |= ORC_RESID_ZERO;
            for (int64_t x = 0; x < vocab; ++x) w[x] = P[a][x];
        }
    } else {
        for (int64_t x = 0; x < vocab; ++x) w[x] = P[a][x];
    }
    double margin;
    *tok = inv_cdf(w, vocab, orc_uniform(seed, req, (uint32_t)a, 1u), &margin);
    if (margin < INVCDF_MARGIN) *flags |= ORC_FLAG_INVCDF;
    free(w);
    free(h);
    free(wgt);
    return a;
}

/*
 * Alternative outcomes of near-tie decisions (a test aid, computed beside the
 * outputs above and never feeding them).  A decision inside its margin may
 * go either way on another machine's rounding: the ratio test (|u - p/q| <
 * 1e-6, the bound the task states; block verification: |eta_j - h_j|), a
 * top-p cut (its prefix mass within 1e-9 of top_p * Z1, so the kept set may
 * hold one token more or less, which renormalises every probability of the
 * row), an inverse-CDF draw (u * W within 1e-9 * W of a cumulative
 * boundary), an empty-looking residual (W below 1e-9).  For every position
 * j of a request the oracle states the decision there and whether it is
 * ambiguous, and the token the request would emit if its chain stopped at j,
 * with the neighbours a near boundary admits.  A verify result is then valid
 * iff it is one of the outcomes these decisions allow.
 */
#define ORC_ALT_ACCEPT    1  /* chain: the test at j accepts (j < v);          */
                             /* block: eta_j < h_j (1 <= j <= v)               */
#define ORC_ALT_AMBIG     2  /* that decision lies inside its margin          */
#define ORC_ALT_DRAW_NEAR 4  /* the draw at j sits near a boundary: the       */
                             /* tokens in draw_alt are valid too              */
#define ORC_ALT_DRAW_ROW  8  /* the distribution drawn from at j is itself    */
                             /* uncertain (a near top-p cut of a row it uses, */
                             /* or a residual below 1e-9): any token of p_j's */
                             /* support, or the token its cut leaves out next */

typedef struct {
    int32_t* dec;       /* [n, K+1] ORC_ALT_* bits per position               */
    int32_t* draw;      /* [n, K+1] token emitted if the chain stops at j     */
    int32_t* draw_alt;  /* [n, K+1, 2] tokens across a near boundary, or -1   */
    int32_t* n_flag;    /* [n] decisions of the oracle's own path that are    */
                        /* inside their margins                               */
    int32_t* n_dec;     /* [n] decisions of the oracle's own path             */
} orc_alt_t;

/* inv_cdf (C7) with the tokens across a boundary that u * W lies within
 * INVCDF_MARGIN * W of: alt[0] below (the last positive weight before the
 * token), alt[1] above (the first positive weight after it); -1 where the
 * boundary is not near or no such token exists.  Returns 1 if either is near. */
static int inv_cdf_near(const double* w, int64_t n, double u, int64_t* tok, int32_t alt[2])
{
    double margin;
    *tok = inv_cdf(w, n, u, &margin);
    alt[0] = alt[1] = -1;
    if (!(margin < INVCDF_MARGIN)) return 0;
    double W = 0.0;
    for (int64_t x = 0; x < n; ++x) W += w[x];
    const double target = u * W;
    double before = 0.0;
    for (int64_t x = 0; x < *tok; ++x) before += w[x];
    const double cum = before + (*tok >= 0 ? w[*tok] : 0.0);
    if (*tok < 0 || target - before < INVCDF_MARGIN * W)
        for (int64_t y = (*tok < 0 ? n : *tok) - 1; y >= 0; --y)
            if (w[y] > 0.0) { alt[0] = (int32_t)y; break; }
    if (*tok >= 0 && cum - target < INVCDF_MARGIN * W)
        for (int64_t y = *tok + 1; y < n; ++y)
            if (w[y] > 0.0) { alt[1] = (int32_t)y; break; }
    return 1;
}

/* The alternatives of one request whose rows are all valid (see above).
 * P, Q: dense rows; tr: target row records; qcm: the draft rows' cut
 * margins; a_orc: the oracle's accepted length.  Writes dec, draw, draw_alt
 * ([K+1] slots of this request) and the request's decision counts. */
static void alternatives(double* const* P, double* const* Q, const orc_row_t* tr, const double* qcm, const int32_t* d,
                         int v, int64_t vocab, int greedy, int block, int topp_on, uint64_t seed, uint32_t req,
                         int a_orc, int32_t* dec, int32_t* draw, int32_t* draw_alt, int32_t* n_flag, int32_t* n_dec)
{
    int nf = 0, nd = 0;
    /* near top-p cuts: per position, of the target row and of the draft row */
    int* cut_t = (int*)calloc((size_t)(v + 1), sizeof(int));
    int* cut_q = (int*)calloc((size_t)(v + 1), sizeof(int));
    for (int j = 0; j <= v && !greedy; ++j) {
        cut_t[j] = tr[j].cut_margin < CUTOFF_MARGIN;
        cut_q[j] = j < v && qcm[j] < CUTOFF_MARGIN;
        if (topp_on) nd += 1 + (j < v);
        nf += cut_t[j] + cut_q[j];
    }
    double* wgt = (double*)malloc((size_t)(v + 1) * sizeof(double));
    wgt[0] = 1.0;
    if (greedy) {
        /* greedy requests keep the chain's rule in both modes; in block mode
         * the bits say it as stop tests: j passes iff drafts 0..j-1 all match */
        int match = 1;
        for (int j = 0; j < v; ++j) {
            const int ok = d[j] == tr[j].argmax;
            if (block) {
                match = match && ok;
                dec[j + 1] = match ? ORC_ALT_ACCEPT : 0;
            } else {
                dec[j] = ok ? ORC_ALT_ACCEPT : 0;
            }
        }
        nd += a_orc < v ? a_orc + 1 : v;
    } else if (!block) {
        for (int j = 0; j < v; ++j) {
            const double p = P[j][d[j]], q = Q[j][d[j]];
            const double u = orc_uniform(seed, req, (uint32_t)j, 0u);
            int acc, amb = cut_t[j] || cut_q[j];
            if (q > 0.0) {
                acc = u < p / q;
                if (fabs(u - p / q) < RATIO_MARGIN) {
                    amb = 1;
                    if (j <= a_orc) ++nf;
                }
            } else {
                acc = p > 0.0;
            }
            dec[j] = (acc ? ORC_ALT_ACCEPT : 0) | (amb ? ORC_ALT_AMBIG : 0);
        }
        nd += a_orc < v ? a_orc + 1 : v;
    } else {
        /* block verification: the weights, then stop decisions at 1..v; a
         * near cut of any row up to j moves w_j or H_j */
        int cut_upto = 0;
        for (int j = 1; j <= v; ++j) {
            const double p = P[j - 1][d[j - 1]], q = Q[j - 1][d[j - 1]];
            const double r = q > 0.0 ? p / q : (p > 0.0 ? INFINITY : 0.0);
            const double x = wgt[j - 1] > 0.0 ? wgt[j - 1] * r : 0.0;
            wgt[j] = x < 1.0 ? x : 1.0;
        }
        for (int j = 1; j <= v; ++j) {
            cut_upto |= cut_t[j - 1] || cut_q[j - 1];
            double h = wgt[j];
            if (j < v) {
                double H = 0.0;
                for (int64_t x = 0; x < vocab; ++x) {
                    const double m = wgt[j] * P[j][x] - Q[j][x];
                    H += m > 0.0 ? m : 0.0;
                }
                const double den = H + 1.0 - wgt[j];
                h = den > 0.0 ? H / den : 1.0;
            }
            const double eta = orc_uniform(seed, req, (uint32_t)(j - 1), 0u);
            const int near = fabs(eta - h) < RATIO_MARGIN;
            const int amb = near || cut_upto || cut_t[j] || (j < v && cut_q[j]);
            dec[j] = (eta < h ? ORC_ALT_ACCEPT : 0) | (amb ? ORC_ALT_AMBIG : 0);
            nf += near;
        }
        nd += v;
    }
    /* the token emitted if the chain stops at j */
    double* w = (double*)malloc((size_t)vocab * sizeof(double));
    int cut_upto = 0;
    for (int j = 0; j <= v; ++j) {
        draw_alt[2 * j] = draw_alt[2 * j + 1] = -1;
        if (greedy) {
            draw[j] = tr[j].argmax;
            continue;
        }
        if (j > 0) cut_upto |= cut_t[j - 1] || cut_q[j - 1];
        int bits = 0;
        if (cut_t[j] || (j < v && cut_q[j]) || (block && cut_upto)) bits |= ORC_ALT_DRAW_ROW;
        if (j < v) {
            const double wj = block ? wgt[j] : 1.0;
            double W = 0.0;
            for (int64_t x = 0; x < vocab; ++x) {
                const double m = wj * P[j][x] - Q[j][x];
                w[x] = m > 0.0 ? m : 0.0;
                W += w[x];
            }
            if (W < RESID_MIN) bits |= ORC_ALT_DRAW_ROW;
            if (!(W > 0.0))
                for (int64_t x = 0; x < vocab; ++x) w[x] = P[j][x];
        } else {
            for (int64_t x = 0; x < vocab; ++x) w[x] = P[j][x];
        }
        int64_t t;
        if (inv_cdf_near(w, vocab, orc_uniform(seed, req, (uint32_t)j, 1u), &t, draw_alt + 2 * j))
            bits |= ORC_ALT_DRAW_NEAR;
        draw[j] = (int32_t)t;
        dec[j] |= bits;
        if (j == a_orc) nf += (bits & (ORC_ALT_DRAW_NEAR | ORC_ALT_DRAW_ROW)) != 0;
    }
    nd += 1;   /* the emitted token */
    *n_flag = nf;
    *n_dec = nd;
    free(w);
    free(wgt);
    free(cut_t);
    free(cut_q);
}

/*
 * One request's chain (C5, C6).  tgt_rows[j] (j <= v) and drf_rows[j]
 * (j < v) point at the logits rows of the window; d[j] are the drafts.
 * Outputs follow the library's layout: out_tokens has K+1 slots, -1 filled.
 */
static void verify_request(const void* const* tgt_rows, const void* const* drf_rows, int dtype, int64_t vocab,
                           int v, int K, const int32_t* d, float T, int32_t top_k, float top_p,
                           uint64_t seed, uint32_t req, int32_t layout_bad, int block,
                           int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                           int32_t* pos_status, int32_t* flags, double* p_tok, double* q_tok, const orc_alt_t* alt,
                           size_t alt_off)
{
    *flags = 0;
    for (int j = 0; j <= K; ++j) {
        out_tokens[j] = -1;
        pos_status[j] = 0;
        p_tok[j] = NAN;
        q_tok[j] = NAN;
        if (alt) {
            alt->dec[alt_off + j] = 0;
            alt->draw[alt_off + j] = -1;
            alt->draw_alt[2 * (alt_off + j)] = alt->draw_alt[2 * (alt_off + j) + 1] = -1;
        }
    }
    if (alt) {
        alt->n_flag[alt_off / (size_t)(K + 1)] = 0;
        alt->n_dec[alt_off / (size_t)(K + 1)] = 0;
    }
    *accept_len = 0;
    *num_emitted = 0;
    if (layout_bad) {
        pos_status[0] |= ORC_BAD_LAYOUT;
        return;
    }
    const int greedy = (T == 0.0f);
    int err = 0;
    if (bad_params(T, top_p)) {
        pos_status[0] |= ORC_BAD_PARAM;
        return;
    }
    double** P = (double**)calloc((size_t)(v + 1), sizeof(double*));
    double** Q = (double**)calloc((size_t)(v + 1), sizeof(double*));
    orc_row_t* tr = (orc_row_t*)calloc((size_t)(v + 1), sizeof(orc_row_t));
    orc_row_t qr;
    double* qcm = (double*)malloc((size_t)(v + 1) * sizeof(double));
    for (int j = 0; j <= v; ++j) {
        qcm[j] = INFINITY;
        P[j] = (double*)malloc((size_t)vocab * sizeof(double));
        pos_status[j] |= orc_row_transform(tgt_rows[j], dtype, vocab, T, top_k, top_p, &tr[j], P[j]);
        if (!greedy && tr[j].cut_margin < CUTOFF_MARGIN) *flags |= ORC_FLAG_CUTOFF;
        if (j < v) {
            if (d[j] < 0 || (int64_t)d[j] >= vocab) pos_status[j] |= ORC_BAD_TOKEN;
            if (!greedy) {
                Q[j] = (double*)malloc((size_t)vocab * sizeof(double));
                pos_status[j] |= orc_row_transform(drf_rows[j], dtype, vocab, T, top_k, top_p, &qr, Q[j]);
                if (qr.cut_margin < CUTOFF_MARGIN) *flags |= ORC_FLAG_CUTOFF;
                qcm[j] = qr.cut_margin;
            }
        }
        if (pos_status[j] & ORC_ERROR_MASK) err = 1;
    }
    if (!err) {
        int a = v;
        int64_t t = -1;
        if (greedy) {
            for (int j = 0; j < v; ++j)
                if (d[j] != tr[j].argmax) { a = j; break; }
            t = tr[a].argmax;
        } else if (block) {
            a = block_accept(P, Q, d, v, vocab, seed, req, pos_status, flags, p_tok, q_tok, &t);
        } else {
            for (int j = 0; j < v; ++j) {
                double p = P[j][d[j]], q = Q[j][d[j]];
                p_tok[j] = p;
                q_tok[j] = q;
                double u = orc_uniform(seed, req, (uint32_t)j, 0u);
                int accept;
                if (q > 0.0) {
                    double ratio = p / q;
                    accept = (u < ratio);
                    if (fabs(u - ratio) < RATIO_MARGIN) *flags |= ORC_FLAG_RATIO;
                } else {
                    /* q(d) == 0: the ratio is +inf when p > 0 and 0/0 when
                     * p == 0 (reading: accept only in the first case). */
                    pos_status[j] |= ORC_Q_ZERO;
                    accept = (p > 0.0);
                }
                if (!accept) { a = j; break; }
            }
            double* w = (double*)malloc((size_t)vocab * sizeof(double));
            if (a < v) {
                double W = 0.0;
                for (int64_t x = 0; x < vocab; ++x) {
                    double r = ORC_PLANT == 1 ? Q[a][x] - P[a][x] : P[a][x] - Q[a][x];
                    w[x] = r > 0.0 ? r : 0.0;
                    W += w[x];
                }
                if (W < RESID_MIN) *flags |= ORC_FLAG_RESID;
                if (!(W > 0.0)) {
                    /* reading: an empty residual falls back to p itself */
                    pos_status[a] |= ORC_RESID_ZERO;
                    for (int64_t x = 0; x < vocab; ++x) w[x] = P[a][x];
                }
            } else {
                for (int64_t x = 0; x < vocab; ++x) w[x] = P[a][x];
            }
            double margin;
            t = inv_cdf(w, vocab, orc_uniform(seed, req, (uint32_t)a, ORC_PLANT == 5 ? 0u : 1u), &margin);
            if (margin < INVCDF_MARGIN) *flags |= ORC_FLAG_INVCDF;
            free(w);
        }
        for (int j = 0; j < a; ++j) out_tokens[j] = d[j];
        out_tokens[a] = (int32_t)t;
        *accept_len = a;
        *num_emitted = a + 1;
        if (alt) {
            const size_t r = alt_off / (size_t)(K + 1);
            alternatives(P, Q, tr, qcm, d, v, vocab, greedy, block, top_p < 1.0f, seed, req, a, alt->dec + alt_off,
                         alt->draw + alt_off, alt->draw_alt + 2 * alt_off, alt->n_flag + r, alt->n_dec + r);
        }
    }
    for (int j = 0; j <= v; ++j) {
        free(P[j]);
        if (Q[j]) free(Q[j]);
    }
    free(P);
    free(Q);
    free(tr);
    free(qcm);
}

static const void* row_ptr(const void* base, int dtype, int64_t row, int64_t stride)
{
    size_t esz = dtype == 0 ? 2 : 4;
    return (const void*)((const char*)base + (size_t)row * (size_t)stride * esz);
}

/*
 * Uniform layout (C5-C7): target [n, K+1, V], draft [n, K, V], row stride
 * = vocab.  verify_len (nullable => K) caps each request's window.  The
 * requests are requests first_req .. first_req + n - 1 of a larger batch (their
 * uniforms are keyed by that index).
 * p_tok / q_tok ([n, K+1]) receive p_j(d_j) and q_j(d_j) where tested.
 */
static void verify_uniform(const void* target, const void* draft, int dtype, int n, int K, int64_t vocab,
                           const int32_t* draft_tokens, const int32_t* verify_len, const float* T,
                           const int32_t* top_k, const float* top_p, uint64_t seed, int first_req, int block,
                           int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted, int32_t* pos_status,
                           int32_t* flags, double* p_tok, double* q_tok, const orc_alt_t* alt)
{
    const void** tr = (const void**)malloc((size_t)(K + 1) * sizeof(void*));
    const void** dr = (const void**)malloc((size_t)(K + 1) * sizeof(void*));
    for (int r = 0; r < n; ++r) {
        int v = verify_len ? verify_len[r] : K;
        int bad = (v < 0 || v > K);
        if (bad) v = 0;
        for (int j = 0; j <= v; ++j) {
            tr[j] = row_ptr(target, dtype, (int64_t)r * (K + 1) + j, vocab);
            dr[j] = (j < v && draft) ? row_ptr(draft, dtype, (int64_t)r * K + j, vocab) : NULL;
        }
        verify_request(tr, dr, dtype, vocab, v, K, draft_tokens + (size_t)r * K, T[r],
                       top_k ? top_k[r] : 0, top_p ? top_p[r] : 1.0f, seed, (uint32_t)(first_req + r), bad, block,
                       accept_len + r, out_tokens + (size_t)r * (K + 1), num_emitted + r,
                       pos_status + (size_t)r * (K + 1), flags + r,
                       p_tok + (size_t)r * (K + 1), q_tok + (size_t)r * (K + 1), alt, (size_t)r * (K + 1));
    }
    free(tr);
    free(dr);
}

void orc_verify_chain(const void* target, const void* draft, int dtype, int n, int K, int64_t vocab,
                      const int32_t* draft_tokens, const int32_t* verify_len,
                      const float* T, const int32_t* top_k, const float* top_p, uint64_t seed, int first_req,
                      int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                      int32_t* pos_status, int32_t* flags, double* p_tok, double* q_tok, const orc_alt_t* alt)
{
    verify_uniform(target, draft, dtype, n, K, vocab, draft_tokens, verify_len, T, top_k, top_p, seed, first_req, 0,
                   accept_len, out_tokens, num_emitted, pos_status, flags, p_tok, q_tok, alt);
}

/* Block verification over the uniform layout (see block_accept); arguments
 * and outputs as orc_verify_chain; greedy requests take the chain's rule. */
void orc_verify_block(const void* target, const void* draft, int dtype, int n, int K, int64_t vocab,
                      const int32_t* draft_tokens, const int32_t* verify_len,
                      const float* T, const int32_t* top_k, const float* top_p, uint64_t seed, int first_req,
                      int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                      int32_t* pos_status, int32_t* flags, double* p_tok, double* q_tok, const orc_alt_t* alt)
{
    verify_uniform(target, draft, dtype, n, K, vocab, draft_tokens, verify_len, T, top_k, top_p, seed, first_req, 1,
                   accept_len, out_tokens, num_emitted, pos_status, flags, p_tok, q_tok, alt);
}

/*
 * Ragged layout (C9): target rows packed on a flat token axis, request r's
 * row j at qo_indptr[r] + j (j <= verify_lens[r]), rows past the last window
 * up to the bucket are padding and never read.  Draft rows stay in the
 * drafted block layout [n, K_max, V] (the block is drafted in full; only the
 * verified positions change).  A window that is not qo_indptr[r+1] -
 * qo_indptr[r] == verify_lens[r] + 1 wide, or leaves [0, bucket), is a
 * layout error for that request.
 */
void orc_verify_ragged(const void* target, const void* draft, int dtype, int n, int K_max, int64_t vocab,
                       int64_t bucket, const int32_t* qo_indptr, const int32_t* verify_lens,
                       const int32_t* draft_tokens, const float* T, const int32_t* top_k, const float* top_p,
                       uint64_t seed, int first_req, int32_t* accept_len, int32_t* out_tokens, int32_t* num_emitted,
                       int32_t* pos_status, int32_t* flags, double* p_tok, double* q_tok, const orc_alt_t* alt)
{
    const void** tr = (const void**)malloc((size_t)(K_max + 1) * sizeof(void*));
    const void** dr = (const void**)malloc((size_t)(K_max + 1) * sizeof(void*));
    for (int r = 0; r < n; ++r) {
        int v = verify_lens[r];
        int64_t start = qo_indptr[r], end = qo_indptr[r + 1];
        int bad = (v < 0 || v > K_max || start < 0 || end - start != (int64_t)v + 1 || end > bucket);
        if (bad) v = 0;
        for (int j = 0; j <= v; ++j) {
            tr[j] = bad ? NULL : row_ptr(target, dtype, start + j, vocab);
            dr[j] = (!bad && j < v && draft) ? row_ptr(draft, dtype, (int64_t)r * K_max + j, vocab) : NULL;
        }
        verify_request(tr, dr, dtype, vocab, v, K_max, draft_tokens + (size_t)r * K_max, T[r],
                       top_k ? top_k[r] : 0, top_p ? top_p[r] : 1.0f, seed, (uint32_t)(first_req + r), bad, 0,
                       accept_len + r, out_tokens + (size_t)r * (K_max + 1), num_emitted + r,
                       pos_status + (size_t)r * (K_max + 1), flags + r,
                       p_tok + (size_t)r * (K_max + 1), q_tok + (size_t)r * (K_max + 1), alt,
                       (size_t)r * (K_max + 1));
    }
    free(tr);
    free(dr);
}

/* ------------------------------------------------------------------------- */
/* C8: confidence-scheduled budget planner.                                  */
/* ------------------------------------------------------------------------- */
typedef struct {
    float s;
    int32_t i;
    int32_t r;
} orc_cand_t;

/* Global survival rank: s desc, then position asc, then request asc.  The
 * tie-break uses no values, and position before request keeps each
 * request's selection a prefix even when c == 1 makes survivals tie. */
static int cmp_cand(const void* a, const void* b)
{
    const orc_cand_t* x = (const orc_cand_t*)a;
    const orc_cand_t* y = (const orc_cand_t*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
#if ORC_PLANT == 4
    if (x->r != y->r) return x->r < y->r ? -1 : 1;
#endif
    if (x->i != y->i) return x->i < y->i ? -1 : 1;
    if (x->r != y->r) return x->r < y->r ? -1 : 1;
    return 0;
}

/*
 * c_{r,i} = conf[r * ld + i], NaN -> 0, clamped to [0, 1].  Survival
 * s_{r,i} = s_{r,i-1} * c_{r,i} in fp32, left to right, s_{r,-1} = 1 (fp32 so
 * that the device planner can reach the same bits).  Candidates are (r, i)
 * for i < K_r (K_r = draft_len[r], or K; outside [0, K] is clamped and
 * reported in *status).  N_sel = min(budget - n, sum K_r) candidates are
 * taken in rank order; v_r counts r's; each request submits v_r + 1 tokens
 * (one anchor/bonus row), qo_indptr is the exclusive prefix sum of the
 * windows and total = qo_indptr[n].  Returns 0, or -1 for bad arguments.
 */
int orc_plan_budget(const float* conf, int ld, const int32_t* draft_len, int n, int K,
                    int budget, int bucket, int32_t* verify_lens, int32_t* qo_indptr,
                    int32_t* total, int32_t* status)
{
    if (n <= 0 || K < 0 || ld < K || budget < n || bucket < budget) return -1;
    *status = 0;
    orc_cand_t* cand = (orc_cand_t*)malloc((size_t)n * (size_t)(K > 0 ? K : 1) * sizeof(orc_cand_t));
    int64_t nc = 0;
    for (int r = 0; r < n; ++r) {
        int kr = draft_len ? draft_len[r] : K;
        if (kr < 0 || kr > K) {
            *status |= 1;
            kr = kr < 0 ? 0 : K;
        }
        float s = 1.0f;
        for (int i = 0; i < kr; ++i) {
            float c = conf[(size_t)r * (size_t)ld + (size_t)i];
            if (isnan(c)) c = 0.0f;
            if (c < 0.0f) c = 0.0f;
            if (c > 1.0f) c = 1.0f;
            volatile float prod = s * c;   /* one fp32 rounding per step */
            s = prod;
            cand[nc].s = s;
            cand[nc].i = i;
            cand[nc].r = r;
            ++nc;
        }
    }
    int64_t nsel = (int64_t)budget - n;
    if (nsel > nc) nsel = nc;
    qsort(cand, (size_t)nc, sizeof(orc_cand_t), cmp_cand);
    for (int r = 0; r < n; ++r) verify_lens[r] = 0;
    for (int64_t t = 0; t < nsel; ++t) verify_lens[cand[t].r] += 1;
    qo_indptr[0] = 0;
    for (int r = 0; r < n; ++r) qo_indptr[r + 1] = qo_indptr[r] + verify_lens[r] + 1;
    *total = qo_indptr[n];
    free(cand);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* NEXT-1: verify budget from a profiled step-cost table.                    */
/* ------------------------------------------------------------------------- */
/*
 * NVIDIA/TensorRT-LLM PR #17056, description "What is here / Planner": the
 * budget is the argmax of tau / cost over a profiled step-cost table, a global
 * argmax because the cost curve is a staircase and Theta = tau / T is not
 * unimodal on it; without a profiled table the planner does not trim.  Review
 * commit, section "Cost model": the table is indexed by tokens submitted to the
 * target, bs * (verify_len + 1), the bonus token included; a fixed per-step
 * overhead and an optional batch-size staircase of overheads are added (they
 * do not cancel in the ratio).
 *
 * Readings:
 *  - tau(B) = expected tokens a step that submits B tokens emits: n (one
 *    anchor / bonus token per request) plus the survivals s_{r,i} of the
 *    B - n candidates the planner selects, i.e. the B - n largest survivals
 *    (ties in s do not change the sum).  Survivals as in orc_plan_budget.
 *  - A step submitting B tokens runs on the first shelf j with
 *    cost_tokens[j] >= B (shelves ascending) and costs cost_ms[j]; B above the
 *    last shelf is not available.
 *  - The batch overhead of n requests is batch_overhead_ms of the first entry
 *    with batch_sizes >= n, or of the last entry when n exceeds them all.
 *  - Candidates: B = n .. B_max, B_max = n + min(sum K_r, bucket - n).
 *    Theta(B) = tau(B) / (cost(B) + fixed_overhead_ms + batch overhead); the
 *    largest Theta wins; among equal Theta the larger B (same throughput,
 *    more tokens per step).
 *  - No table, or no shelf that holds B = n: B = B_max (no trimming), status
 *    bit 2.  A table whose shelves are not strictly ascending, or with a cost
 *    or overhead that is negative or not finite: B = B_max, status bit 4.
 *    Status bit 1: a draft length outside [0, K] was clamped.
 *  - *margin = (Theta_best - Theta_second) / Theta_best over candidates with
 *    distinct Theta (1 when there is only one): how close the choice was.
 */
static int cmp_desc_float(const void* a, const void* b)
{
    const float x = *(const float*)a, y = *(const float*)b;
    return x > y ? -1 : (x < y ? 1 : 0);
}

int orc_choose_budget(const float* conf, int ld, const int32_t* draft_len, int n, int K,
                      const int32_t* cost_tokens, const float* cost_ms, int n_cost, float fixed_overhead_ms,
                      const int32_t* batch_sizes, const float* batch_overhead_ms, int n_batch, int bucket,
                      int32_t* budget, double* theta_best, double* margin, int32_t* status)
{
    if (n <= 0 || K < 0 || ld < K || bucket < n || n_cost < 0 || n_batch < 0) return -1;
    *status = 0;
    float* sv = (float*)malloc((size_t)n * (size_t)(K > 0 ? K : 1) * sizeof(float));
    int64_t nc = 0;
    for (int r = 0; r < n; ++r) {
        int kr = draft_len ? draft_len[r] : K;
        if (kr < 0 || kr > K) {
            *status |= 1;
            kr = kr < 0 ? 0 : K;
        }
        float s = 1.0f;
        for (int i = 0; i < kr; ++i) {
            float c = conf[(size_t)r * (size_t)ld + (size_t)i];
            if (isnan(c)) c = 0.0f;
            if (c < 0.0f) c = 0.0f;
            if (c > 1.0f) c = 1.0f;
            volatile float prod = s * c;
            s = prod;
            sv[nc++] = s;
        }
    }
    qsort(sv, (size_t)nc, sizeof(float), cmp_desc_float);
    int64_t m_max = nc < (int64_t)(bucket - n) ? nc : (int64_t)(bucket - n);
    const int64_t b_max = n + m_max;
    /* tau for every B: prefix sums of the sorted survivals, sequential */
    double* tau = (double*)malloc((size_t)(m_max + 1) * sizeof(double));
    tau[0] = (double)n;
    for (int64_t m = 1; m <= m_max; ++m) tau[m] = tau[m - 1] + (double)sv[m - 1];
    double batch_oh = 0.0;
    if (n_batch > 0) {
        int j = 0;
        while (j < n_batch - 1 && batch_sizes[j] < n) ++j;
        batch_oh = (double)batch_overhead_ms[j];
    }
    int table_ok = isfinite(fixed_overhead_ms) && fixed_overhead_ms >= 0.0f && isfinite(batch_oh) && batch_oh >= 0.0;
    for (int j = 0; j < n_cost; ++j)
        if (!(isfinite(cost_ms[j]) && cost_ms[j] >= 0.0f) || (j > 0 && cost_tokens[j] <= cost_tokens[j - 1]))
            table_ok = 0;
    for (int j = 0; j < n_batch; ++j)
        if (!(isfinite(batch_overhead_ms[j]) && batch_overhead_ms[j] >= 0.0f)) table_ok = 0;
    if (!table_ok) *status |= 4;
    double best = -1.0, second = -1.0;
    int64_t best_b = -1;
    int shelf = 0;
    for (int64_t b = n; b <= b_max && n_cost > 0 && table_ok; ++b) {
#if ORC_PLANT == 6
        const int64_t looked_up = b - n;
#else
        const int64_t looked_up = b;
#endif
        while (shelf < n_cost && cost_tokens[shelf] < looked_up) ++shelf;
        if (shelf == n_cost) break;   /* above the last shelf */
        const double th = tau[b - n] / ((double)cost_ms[shelf] + (double)fixed_overhead_ms + batch_oh);
#if ORC_PLANT == 7
        if (best_b >= 0 && th < best) break;   /* first descent */
#endif
        if (th >= best) {
            if (th > best) second = best;
            best = th;
            best_b = b;
        } else if (th > second) {
            second = th;
        }
    }
    if (best_b < 0) {
        if (table_ok) *status |= 2;
        best_b = b_max;
        best = tau[m_max];
        second = -1.0;
    }
    *budget = (int32_t)best_b;
    *theta_best = best;
    *margin = (second < 0.0 || best <= 0.0) ? 1.0 : (best - second) / best;
    free(tau);
    free(sv);
    return 0;
}

/*
 * Acceptance against trimming (NVIDIA/TensorRT-LLM PR #17056, the commit that
 * adds trim_regret_rate): per step, tokens emitted sum(accept_len + 1), tokens
 * submitted sum(v_r + 1), requests trimmed (v_r < K_r), and trimmed requests
 * that accepted their whole window (accept_len == v_r: still alive at the
 * cut, so the cut cost acceptance).  Requests with an error (accept_len < 0
 * or num_emitted == 0) count in none of them.  out[4] as listed.
 */
void orc_verify_stats(const int32_t* accept_len, const int32_t* num_emitted, const int32_t* verify_lens,
                      const int32_t* draft_len, int n, int K, int64_t* out)
{
    out[0] = out[1] = out[2] = out[3] = 0;
    for (int r = 0; r < n; ++r) {
        if (num_emitted[r] == 0 || accept_len[r] < 0) continue;
        int kr = draft_len ? draft_len[r] : K;
        kr = kr < 0 ? 0 : (kr > K ? K : kr);
        const int v = verify_lens ? verify_lens[r] : kr;
        out[0] += accept_len[r] + 1;
        out[1] += v + 1;
        if (v < kr) {
            out[2] += 1;
#if ORC_PLANT == 8
            if (accept_len[r] < v) out[3] += 1;
#else
            if (accept_len[r] == v) out[3] += 1;
#endif
        }
    }
}

/* ------------------------------------------------------------------------- */
/* NEXT-3: online acceptance estimator.                                      */
/* ------------------------------------------------------------------------- */
/*
 * jianc99/sglang PR #8, the DFLASH adaptive-verification commits: a logistic
 * model calibrated while serving, p_k = sigmoid(slope * x_k + bias_k), x_k =
 * logit(q_max) of the temperature-scaled draft distribution at position k
 * (greedy rows at T = 1), clamped to +-40; one slope shared by all positions,
 * one intercept per position, starting from 0.5 and -0.2; observe() labels the
 * accepted drafts and the first rejected one and adds them to the Newton
 * (IRLS) statistics; every 100 calls the arrowhead system is solved with ridge
 * 1e-3, each update is damped by n / (n + 50), non-finite steps are dropped,
 * and a slope step that would make the slope negative is halved up to 8 times
 * and dropped only if it still crosses zero; the intercepts take their Newton
 * step given the slope step actually taken; the statistics are then cleared.
 *
 * Readings:
 *  - q is the distribution the draft token is drawn from, the request's
 *    transform (temperature, top-k, top-p) of the draft row -- the same q the
 *    verification uses -- at T = 1 for greedy requests.  q_max = 1 / z (the
 *    top token has mass exp(0)), so x = logit(q_max) = -ln(z - 1); z - 1 is the
 *    kept mass after the first kept token (no cancellation).  A row with an
 *    error gives x = NaN; a single kept token gives +40.
 *  - Observed positions of request r: k = 0 .. min(accept_len, v_r - 1); label
 *    1 for k < accept_len, 0 for the first rejected one.  Requests that
 *    emitted nothing (errors) and non-finite features are skipped.
 *  - Newton statistics at the current coefficients: g_a = sum (y - p) x,
 *    g_k = sum_k (y - p), H_aa = sum w x^2, H_ak = sum_k w x, H_kk = sum_k w,
 *    w = p (1 - p), n = observation count.  Refit: with lambda = 1e-3 on the
 *    diagonal, t = (g_a - sum_k H_ak g_k / (H_kk + l)) / (H_aa + l - sum_k
 *    H_ak^2 / (H_kk + l)); d = n / (n + 50); while slope + d t < 0 (at most 8
 *    times) t /= 2; if it is still negative t = 0; intercept steps u_k =
 *    (g_k - H_ak t) / (H_kk + l); if t and every u_k are finite, slope += d t
 *    and bias_k += d u_k.  The statistics are cleared either way.  A refit
 *    with no observations changes nothing.
 *
 * State (doubles): [0] slope, [1..K] bias, [K+1] g_a, [K+2] H_aa,
 * [K+3 ..] g_k (K), H_ak (K), H_kk (K), [4K+3] n, [4K+4] calls.
 */
void orc_est_init(double* state, int K)
{
    for (int i = 0; i < 4 * K + 5; ++i) state[i] = 0.0;
    state[0] = 0.5;
    for (int k = 0; k < K; ++k) state[1 + k] = -0.2;
}

void orc_est_features(const void* draft, int dtype, int n, int K, int64_t vocab, const float* T,
                      const int32_t* top_k, const float* top_p, double* x)
{
    for (int r = 0; r < n; ++r) {
        const float t = T[r] > 0.0f ? T[r] : 1.0f;
        for (int k = 0; k < K; ++k) {
            orc_row_t tr;
            const int st = orc_row_transform(row_ptr(draft, dtype, (int64_t)r * K + k, vocab), dtype, vocab, t,
                                             top_k ? top_k[r] : 0, top_p ? top_p[r] : 1.0f, &tr, NULL);
            double xv;
            if (st & ORC_ERROR_MASK) {
                xv = NAN;
            } else {
                xv = tr.z_rest > 0.0 ? -log(tr.z_rest) : INFINITY;
                xv = xv > 40.0 ? 40.0 : (xv < -40.0 ? -40.0 : xv);
            }
            x[(size_t)r * K + k] = xv;
        }
    }
}

void orc_est_predict(const double* state, const double* x, int n, int K, double* p)
{
    for (int r = 0; r < n; ++r)
        for (int k = 0; k < K; ++k) {
            const double s = state[0] * x[(size_t)r * K + k] + state[1 + k];
            p[(size_t)r * K + k] = 1.0 / (1.0 + exp(-s));
        }
}

static void est_refit(double* st, int K)
{
    double* g_b = st + K + 3;
    double* h_ab = g_b + K;
    double* h_bb = h_ab + K;
    const double lam = 1e-3, n = st[4 * K + 3];
    if (n > 0.0) {
        double num = st[K + 1], den = st[K + 2] + lam;
        for (int k = 0; k < K; ++k) {
            num -= h_ab[k] * g_b[k] / (h_bb[k] + lam);
            den -= h_ab[k] * h_ab[k] / (h_bb[k] + lam);
        }
        double t = num / den;
        const double d = n / (n + 50.0);
#if ORC_PLANT == 11
        if (st[0] + d * t < 0.0) t = 0.0;
#else
        for (int i = 0; i < 8 && st[0] + d * t < 0.0; ++i) t *= 0.5;
        if (st[0] + d * t < 0.0) t = 0.0;
#endif
        int ok = isfinite(t);
        for (int k = 0; k < K; ++k) ok = ok && isfinite((g_b[k] - h_ab[k] * t) / (h_bb[k] + lam));
        if (ok) {
            for (int k = 0; k < K; ++k) st[1 + k] += d * (g_b[k] - h_ab[k] * t) / (h_bb[k] + lam);
            st[0] += d * t;
        }
    }
    for (int i = K + 1; i < 4 * K + 4; ++i) st[i] = 0.0;
}

void orc_est_observe(double* state, const double* x, const int32_t* accept_len, const int32_t* num_emitted,
                     const int32_t* verify_lens, int n, int K, int refit_every)
{
    double* g_b = state + K + 3;
    double* h_ab = g_b + K;
    double* h_bb = h_ab + K;
    for (int r = 0; r < n; ++r) {
        if (num_emitted[r] == 0 || accept_len[r] < 0) continue;
        int v = verify_lens ? verify_lens[r] : K;
        v = v < 0 ? 0 : (v > K ? K : v);
        const int a = accept_len[r];
#if ORC_PLANT == 10
        const int last = v - 1;
#else
        const int last = a < v - 1 ? a : v - 1;
#endif
        for (int k = 0; k <= last; ++k) {
            const double xv = x[(size_t)r * K + k];
            if (!isfinite(xv)) continue;
            const double y = k < a ? 1.0 : 0.0;
            const double p = 1.0 / (1.0 + exp(-(state[0] * xv + state[1 + k])));
            const double w = p * (1.0 - p);
            state[K + 1] += (y - p) * xv;
            state[K + 2] += w * xv * xv;
            g_b[k] += y - p;
            h_ab[k] += w * xv;
            h_bb[k] += w;
            state[4 * K + 3] += 1.0;
        }
    }
    state[4 * K + 4] += 1.0;
    if (refit_every > 0 && fmod(state[4 * K + 4], (double)refit_every) == 0.0) est_refit(state, K);
}
