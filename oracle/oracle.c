/*
 * oracle.c -- plain, slow, fp64 CPU oracle of the target-side verification
 * step of speculative decoding.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The GPU library
 * shares no code, header, table or constant with it and never calls it.
 *
 * Every function follows one of these pages (cited by page title + section):
 *   [LZ] "3.5 Speculative Decoding" (llm-learning-path): "Notation",
 *        "The algorithm (one step)", "Proof that the output distribution is
 *        exactly p", "Tree verification", "Worked example".
 *   [MN] "246 Speculative Decoding" (ai_in_action): 2.2 "The acceptance test
 *        for one token", 3.1 "The acceptance step", 3.3 "The full block loop".
 *   [LB] "Speculative Decoding: Mathematical Foundations, Rejection Sampling
 *        Dynamics, ..." (llms.blog): "The Modified Rejection Sampling
 *        Algorithm", "Acceptance Rate and Total Variation Distance",
 *        "Tree-Based Verification and Custom Attention Masks".
 *   [SS] "Speculative Decoding from First Principles" (theservingstack.com):
 *        "Draft, verify, keep what matches".
 *
 * Where the pages are silent or disagree, the oracle takes these readings:
 *   R1 top-p: the pages name top-p (as part of the pipeline that makes p and
 *      q, [LZ] "Notation", [MN] 6 "Pitfalls") but never define it.  Reading:
 *      the standard nucleus -- tau is the largest probability value such
 *      that the tokens with p >= tau carry total mass >= top_p; every token
 *      with p >= tau is kept (ties at tau all kept), the rest get 0, and the
 *      kept mass is renormalised.  PARITY UNPINNED by the pages: the tests
 *      pin it only to this definition (brute force over upper sets).
 *   R2 accept test: [LZ] writes r < min(1, p/q), [MN] 3.1 and [LB] write
 *      u <= ratio.  Reading: strict, in the division-free form u*Q < P,
 *      which also fixes Q = 0 (accept iff P > 0).
 *   R3 final draw: the residual (or bonus) token is drawn by inverse CDF in
 *      token-index order -- the smallest x with C(x) > u*S, S = sum of the
 *      weights -- with u the (k+1)-th caller-supplied uniform of the
 *      sequence.  The rejecting position's own uniform is never reused: it
 *      is conditioned on the rejection.  If rounding leaves no such x, the
 *      last x with weight > 0 is taken.
 *   R4 residual fallback: if sum max(0, p - q) is 0, the weights are p
 *      ([MN] 3.1 "residual_distribution" falls back to p).
 *   R5 greedy argmax: the first (lowest-index) maximum of the raw logits;
 *      temperature and top-p do not move the argmax.
 *   R6 tree: accept child c of an accepted node n iff token(c) equals the
 *      argmax of n's row; keep the deepest accepted node, ties to the lowest
 *      flattened index ([LZ] "Tree verification", [LB] tree mask).
 *   R7 data errors: a row holding NaN or +inf, a row that is entirely -inf,
 *      a token outside [0, V) or a uniform outside [0, 1) marks the whole
 *      sequence as failed: its tokens and its accepted count are -1.
 *   R10 top-k ([MN] 6 "Pitfalls" names top-k among the processors the
 *      target and draft must share; never defined): keep the tokens whose
 *      logit is at least the K-th largest logit of the row (all ties of the
 *      K-th kept, as in R1), renormalise; applied after temperature (which
 *      does not change the order) and before top-p, which then runs on the
 *      renormalised top-k distribution.  K <= 0 or K >= V: no top-k.
 *   R11 stochastic tree ([LZ] "Tree verification" names SpecInfer's
 *      lossless multi-candidate acceptance rule for sampling without
 *      stating it): the children of a node are candidates drawn
 *      independently from the draft row of that node; they are tried in
 *      flattened order against a target that becomes the normalised
 *      residual max(0, p' - q) after each rejected child (see
 *      oracle_verify_tree_sample).
 *   R8 draft given as probabilities: the step takes the draft "logits (or
 *      probabilities)".  Reading: a probability row is q itself, the
 *      distribution the drafter sampled from -- used as given (no
 *      temperature, no top-p, no renormalisation); only p is processed.
 *      The k gathered values q_i(x~_i) must lie in [0, 1] (R7 otherwise);
 *      the rest of a row is not checked.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* The oracle's own enumerations (deliberately not shared with the GPU
 * library; the tests map names to names). */
enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_STOCHASTIC = 0, ORC_GREEDY = 1 };
enum {
    ORC_OK = 0,
    ORC_BAD_ARGUMENT = -1,
    ORC_ROW_NONFINITE = 1,   /* a NaN or +inf logit                       */
    ORC_ROW_ALL_NEG_INF = 2, /* every logit of the row is -inf            */
    ORC_TOKEN_RANGE = 3,     /* a draft or node token outside [0, V)      */
    ORC_UNIFORM_RANGE = 4,   /* a uniform outside [0, 1)                  */
    ORC_TREE_SHAPE = 5,      /* parents not a rooted tree in topological
                                order, or a node deeper than D            */
    ORC_PROB_RANGE = 6       /* a gathered draft probability not in [0, 1] */
};

/* ---------------------------------------------------------------- input */

/* One logit, upcast exactly to fp64 (fp32 and bf16 both embed in fp64). */
static double logit_at(const void *base, int dtype, size_t i)
{
    if (dtype == ORC_F32)
        return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------- processed row (p/q) */

/* Descending order of probabilities; equal values by index (only to make
 * the sort deterministic -- equal values are always kept or dropped
 * together, R1). */
static const double *g_sort_prob;
static int by_prob_desc(const void *a, const void *b)
{
    int32_t ia = *(const int32_t *)a, ib = *(const int32_t *)b;
    double pa = g_sort_prob[ia], pb = g_sort_prob[ib];
    if (pa > pb) return -1;
    if (pa < pb) return 1;
    return (ia > ib) - (ia < ib);
}

/*
 * Top-p (nucleus) filter of a normalised row, reading R1.
 * Writes info[0] = tau, info[1] = mass of the tokens with p > tau (the
 * cumulative mass just before tau's tie group), info[2] = mass with
 * p >= tau (the cumulative mass that first reaches top_p).
 */
static void nucleus(double *prob, int V, double top_p, double *info)
{
    int32_t *order = (int32_t *)malloc((size_t)V * sizeof *order);
    for (int v = 0; v < V; ++v) order[v] = v;
    g_sort_prob = prob;
    qsort(order, (size_t)V, sizeof *order, by_prob_desc);

    double cum = 0.0, before = 0.0, tau = -1.0;
    int i = 0;
    while (i < V) {
        double value = prob[order[i]];
        double group = 0.0;
        int j = i;
        while (j < V && prob[order[j]] == value) {
            group += prob[order[j]];
            ++j;
        }
        before = cum;
        cum += group;
        if (cum >= top_p) {
            tau = value;
            break;
        }
        i = j;
    }
    if (tau < 0.0) {
        /* Rounding left the whole row short of top_p: keep every token
         * with p > 0. */
        tau = INFINITY;
        for (int v = 0; v < V; ++v)
            if (prob[v] > 0.0 && prob[v] < tau) tau = prob[v];
        before = cum;
    }
    free(order);

    double kept = 0.0;
    for (int v = 0; v < V; ++v) {
        if (prob[v] < tau) prob[v] = 0.0;
        kept += prob[v];
    }
    for (int v = 0; v < V; ++v) prob[v] /= kept;
    info[0] = tau;
    info[1] = before;
    info[2] = cum;
}

/*
 * The processed distribution of one logit row: temperature, then top-p
 * ([LZ] "Notation": p and q are the distributions after temperature and
 * top-p; [MN] 6 "Pitfalls": the same processing on target and draft).
 *   z = l / T,  p(x) = exp(z(x) - max z) / sum_y exp(z(y) - max z).
 * A -inf logit gets probability 0.  Returns a row status (R7).
 * info (optional, 4 doubles): [0] Z = sum exp((l - max l)/T), the
 * normaliser relative to the row maximum; [1] tau; [2] mass above tau;
 * [3] mass at and above tau (top-p only; tau = 0 and both masses = 1
 * without top-p).
 */
/*
 * Top-k filter of a normalised row, reading R10: the K-th largest value
 * (counting equal values one by one), every token at or above it kept,
 * the kept mass renormalised.  Probability is increasing in the logit
 * (T > 0), so this keeps the K largest logits and their ties.
 */
static void top_k_filter(double *prob, int V, int top_k)
{
    int32_t *order = (int32_t *)malloc((size_t)V * sizeof *order);
    for (int v = 0; v < V; ++v) order[v] = v;
    g_sort_prob = prob;
    qsort(order, (size_t)V, sizeof *order, by_prob_desc);
    const double kth = prob[order[top_k - 1]];
    free(order);
    double kept = 0.0;
    for (int v = 0; v < V; ++v) {
        if (prob[v] < kth) prob[v] = 0.0;
        kept += prob[v];
    }
    for (int v = 0; v < V; ++v) prob[v] /= kept;
}

/* oracle_process_row with top-k (R10) between temperature and top-p. */
int oracle_process_row_k(const void *logits, int dtype, int V, double T,
                         double top_p, int top_k, double *prob, double *info)
{
    if (!logits || !prob || V < 1 || !(T > 0.0) || !(top_p > 0.0))
        return ORC_BAD_ARGUMENT;
    double mx = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double l = logit_at(logits, dtype, (size_t)v);
        if (isnan(l) || l == INFINITY) return ORC_ROW_NONFINITE;
        if (l > mx) mx = l;
    }
    if (mx == -INFINITY) return ORC_ROW_ALL_NEG_INF;

    double Z = 0.0;
    for (int v = 0; v < V; ++v) {
        double l = logit_at(logits, dtype, (size_t)v);
        double e = exp((l - mx) / T); /* exp(-inf) = 0 */
        prob[v] = e;
        Z += e;
    }
    for (int v = 0; v < V; ++v) prob[v] /= Z;
    if (top_k > 0 && top_k < V) top_k_filter(prob, V, top_k);

    double tinfo[3] = {0.0, 1.0, 1.0};
    if (top_p < 1.0) nucleus(prob, V, top_p, tinfo);
    if (info) {
        info[0] = Z;
        info[1] = tinfo[0];
        info[2] = tinfo[1];
        info[3] = tinfo[2];
    }
    return ORC_OK;
}

int oracle_process_row(const void *logits, int dtype, int V, double T,
                       double top_p, double *prob, double *info)
{
    return oracle_process_row_k(logits, dtype, V, T, top_p, 0, prob, info);
}

/* First (lowest-index) maximum of the raw logits, reading R5.  Returns a
 * row status; *arg receives the index. */
int oracle_argmax_row(const void *logits, int dtype, int V, int32_t *arg)
{
    double best = -INFINITY;
    int32_t at = -1;
    for (int v = 0; v < V; ++v) {
        double l = logit_at(logits, dtype, (size_t)v);
        if (isnan(l) || l == INFINITY) return ORC_ROW_NONFINITE;
        if (l > best) {
            best = l;
            at = v;
        }
    }
    if (at < 0) return ORC_ROW_ALL_NEG_INF;
    *arg = at;
    return ORC_OK;
}

/* ----------------------------------------------------------- the draw */

/*
 * Inverse-CDF draw from non-negative weights w (reading R3):
 *   S = sum_x w(x) in index order, C(x) = w(0) + ... + w(x),
 *   token = the smallest x with C(x) > u * S.
 * Optional edges[0..2] = S, C(token - 1), C(token).
 */
int32_t oracle_inverse_cdf(const double *w, int V, double u, double *edges)
{
    double S = 0.0;
    for (int x = 0; x < V; ++x) S += w[x];
    double t = u * S, C = 0.0, Cprev = 0.0;
    int32_t last_positive = -1;
    for (int x = 0; x < V; ++x) {
        Cprev = C;
        C += w[x];
        if (w[x] > 0.0) last_positive = x;
        if (C > t) {
            if (edges) {
                edges[0] = S;
                edges[1] = Cprev;
                edges[2] = C;
            }
            return x;
        }
    }
    if (edges) {
        edges[0] = S;
        edges[1] = S;
        edges[2] = S;
    }
    return last_positive;
}

/* ------------------------------------------------------- chain verify */

static void fail_sequence(int32_t *tok, int width, int32_t *num)
{
    for (int i = 0; i < width; ++i) tok[i] = -1;
    *num = -1;
}

/*
 * The accept scan and the final draw of one sequence whose rows passed
 * every check.  p: the k+1 processed target rows, q: the k draft rows (V
 * doubles each, row-major); xt: the k draft tokens; ub: the k+1 uniforms;
 * w: V doubles of scratch.  Writes the sequence's tokens and j, and (d not
 * NULL) P_1..P_k, Q_1..Q_k, S, C(token-1), C(token).
 */
static void step_sequence(const double *p, const double *q, const int32_t *xt,
                          const float *ub, int k, int V, double *w, double *d,
                          int32_t *ot, int32_t *num)
{
    /* Accept x~_i iff u_i * q_i(x~_i) < p_i(x~_i) (R2), left to right,
     * stopping at the first rejection. */
    int j = k;
    for (int i = 0; i < k; ++i) {
        double P = p[(size_t)i * V + xt[i]];
        double Q = q[(size_t)i * V + xt[i]];
        if (d) {
            d[i] = P;
            d[k + i] = Q;
        }
        if (j == k && !((double)ub[i] * Q < P)) j = i;
    }

    /* Residual max(0, p - q) at the rejecting position ([LZ] step 3,
     * [MN] 2.2, [LB] step 3), or p_{k+1} when all k were accepted
     * ([LZ] step 4 "Bonus token"). */
    const double *p_row = p + (size_t)j * V;
    if (j < k) {
        const double *q_row = q + (size_t)j * V;
        double S = 0.0;
        for (int x = 0; x < V; ++x) {
            double diff = p_row[x] - q_row[x];
            w[x] = diff > 0.0 ? diff : 0.0;
            S += w[x];
        }
        if (!(S > 0.0)) /* R4 */
            memcpy(w, p_row, (size_t)V * sizeof *w);
    } else {
        memcpy(w, p_row, (size_t)V * sizeof *w);
    }
    int32_t drawn = oracle_inverse_cdf(w, V, (double)ub[k], d ? d + 2 * k : NULL);

    for (int i = 0; i < j; ++i) ot[i] = xt[i];
    ot[j] = drawn;
    for (int i = j + 1; i <= k; ++i) ot[i] = -1;
    *num = j;
}

/*
 * One verification step for B independent sequences ([LZ] "The algorithm
 * (one step)"; [MN] 3.3; [LB] "The Modified Rejection Sampling Algorithm").
 *
 * target  [B, k+1, V]  logits of the k+1 target positions (dtype)
 * draft   [B, k,   V]  draft logits (STOCHASTIC only; may be NULL in GREEDY)
 * tokens  [B, k]       draft tokens x~_1..x~_k
 * uniforms[B, k+1]     u_1..u_k for the accept tests, u_{k+1} for the final
 *                      draw (STOCHASTIC only; may be NULL in GREEDY)
 * out_tokens [B, k+1]  emitted tokens, -1 after the last one
 * out_num    [B]       number of accepted drafts j (0..k), -1 on a data error
 * dbg [B, 2k+3] (optional): P_1..P_k, Q_1..Q_k, S, C(token-1), C(token)
 * row_info [B, 2k+1, 4] (optional): oracle_process_row's info per row,
 *                      target rows first, then draft rows
 * Returns ORC_BAD_ARGUMENT, or the OR of (1 << status) over every check
 * that failed in any sequence (a failed sequence is checked completely).
 */
int oracle_verify_sample_k(const void *target, const void *draft, int dtype,
                           const int32_t *tokens, const float *uniforms,
                           int B, int k, int V, double T, double top_p, int top_k,
                           int mode, int32_t *out_tokens, int32_t *out_num,
                           double *dbg, double *row_info)
{
    if (!target || !tokens || !out_tokens || !out_num || B < 0 || k < 1 ||
        V < 1 || (dtype != ORC_F32 && dtype != ORC_BF16) ||
        (mode != ORC_STOCHASTIC && mode != ORC_GREEDY))
        return ORC_BAD_ARGUMENT;
    if (mode == ORC_STOCHASTIC &&
        (!draft || !uniforms || !(T > 0.0) || !(top_p > 0.0) || top_p > 1.0))
        return ORC_BAD_ARGUMENT;

    const size_t esz = dtype == ORC_F32 ? 4 : 2;
    const int R = mode == ORC_STOCHASTIC ? 2 * k + 1 : k + 1;
    double *prob = (double *)malloc((size_t)R * V * sizeof *prob);
    double *w = (double *)malloc((size_t)V * sizeof *w);
    int32_t *g = (int32_t *)malloc((size_t)(k + 1) * sizeof *g);
    int errors = 0;

    for (int b = 0; b < B; ++b) {
        int32_t *ot = out_tokens + (size_t)b * (k + 1);
        const int32_t *xt = tokens + (size_t)b * k;
        int bad = 0; /* OR of (1 << status) over everything that failed */

        for (int i = 0; i < k; ++i)
            if (xt[i] < 0 || xt[i] >= V) bad |= 1 << ORC_TOKEN_RANGE;

        if (mode == ORC_GREEDY) {
            /* [LZ] proof, last sentence; [SS] "Draft, verify, keep what
             * matches": accept iff the draft equals the target's argmax,
             * else emit the argmax; bonus = argmax of row k+1. */
            for (int i = 0; i <= k; ++i) {
                const char *row = (const char *)target +
                                  ((size_t)b * (k + 1) + i) * V * esz;
                int status = oracle_argmax_row(row, dtype, V, &g[i]);
                if (status != ORC_OK) bad |= 1 << status;
            }
            if (bad) {
                errors |= bad;
                fail_sequence(ot, k + 1, &out_num[b]);
                continue;
            }
            int j = 0;
            while (j < k && xt[j] == g[j]) ++j;
            for (int i = 0; i < j; ++i) ot[i] = xt[i];
            ot[j] = g[j];
            for (int i = j + 1; i <= k; ++i) ot[i] = -1;
            out_num[b] = j;
            continue;
        }

        const float *ub = uniforms + (size_t)b * (k + 1);
        for (int i = 0; i <= k; ++i)
            if (!(ub[i] >= 0.0f && ub[i] < 1.0f)) bad |= 1 << ORC_UNIFORM_RANGE;

        /* p_1..p_{k+1} (rows 0..k), then q_1..q_k (rows k+1..2k). */
        for (int r = 0; r < R; ++r) {
            const char *row =
                r <= k ? (const char *)target +
                             ((size_t)b * (k + 1) + r) * V * esz
                       : (const char *)draft +
                             ((size_t)b * k + (r - k - 1)) * V * esz;
            double *info = row_info ? row_info + ((size_t)b * R + r) * 4 : NULL;
            int status = oracle_process_row_k(row, dtype, V, T, top_p, top_k,
                                              prob + (size_t)r * V, info);
            if (status != ORC_OK) bad |= 1 << status;
        }
        if (bad) {
            errors |= bad;
            fail_sequence(ot, k + 1, &out_num[b]);
            continue;
        }

        step_sequence(prob, prob + (size_t)(k + 1) * V, xt, ub, k, V, w,
                      dbg ? dbg + (size_t)b * (2 * k + 3) : NULL, ot, &out_num[b]);
    }
    free(prob);
    free(w);
    free(g);
    return errors;
}

/*
 * oracle_verify_sample (STOCHASTIC) with the draft given as probabilities
 * (R8): draft_probs [B, k, V] fp32 is q_1..q_k as given; the target rows
 * are processed as usual.  Same outputs; row_info [B, k+1, 4] (optional)
 * covers the target rows only.
 */
int oracle_verify_sample_probs_k(const void *target, const float *draft_probs,
                                 int dtype, const int32_t *tokens,
                                 const float *uniforms, int B, int k, int V,
                                 double T, double top_p, int top_k, int32_t *out_tokens,
                                 int32_t *out_num, double *dbg, double *row_info)
{
    if (!target || !draft_probs || !tokens || !uniforms || !out_tokens ||
        !out_num || B < 0 || k < 1 || V < 1 ||
        (dtype != ORC_F32 && dtype != ORC_BF16) || !(T > 0.0) ||
        !(top_p > 0.0) || top_p > 1.0)
        return ORC_BAD_ARGUMENT;
    const size_t esz = dtype == ORC_F32 ? 4 : 2;
    double *p = (double *)malloc((size_t)(k + 1) * V * sizeof *p);
    double *q = (double *)malloc((size_t)k * V * sizeof *q);
    double *w = (double *)malloc((size_t)V * sizeof *w);
    int errors = 0;
    for (int b = 0; b < B; ++b) {
        int32_t *ot = out_tokens + (size_t)b * (k + 1);
        const int32_t *xt = tokens + (size_t)b * k;
        const float *ub = uniforms + (size_t)b * (k + 1);
        const float *qb = draft_probs + (size_t)b * k * V;
        int bad = 0;
        for (int i = 0; i < k; ++i) {
            if (xt[i] < 0 || xt[i] >= V) {
                bad |= 1 << ORC_TOKEN_RANGE;
                continue;
            }
            float g = qb[(size_t)i * V + xt[i]];
            if (!(g >= 0.0f && g <= 1.0f)) bad |= 1 << ORC_PROB_RANGE;
        }
        for (int i = 0; i <= k; ++i)
            if (!(ub[i] >= 0.0f && ub[i] < 1.0f)) bad |= 1 << ORC_UNIFORM_RANGE;
        for (int r = 0; r <= k; ++r) {
            const char *row = (const char *)target + ((size_t)b * (k + 1) + r) * V * esz;
            double *info = row_info ? row_info + ((size_t)b * (k + 1) + r) * 4 : NULL;
            int status = oracle_process_row_k(row, dtype, V, T, top_p, top_k,
                                              p + (size_t)r * V, info);
            if (status != ORC_OK) bad |= 1 << status;
        }
        if (bad) {
            errors |= bad;
            fail_sequence(ot, k + 1, &out_num[b]);
            continue;
        }
        for (size_t e = 0; e < (size_t)k * V; ++e) q[e] = (double)qb[e];
        step_sequence(p, q, xt, ub, k, V, w, dbg ? dbg + (size_t)b * (2 * k + 3) : NULL,
                      ot, &out_num[b]);
    }
    free(p);
    free(q);
    free(w);
    return errors;
}

/* ------------------------------------------------------ acceptance rate */

/*
 * Per-position acceptance rate and total-variation distance of one
 * verification batch.  [LZ] "Proof that the output distribution is exactly
 * p": the chance that position i accepts (given that it is tested) is
 * beta_i = sum_x min(p_i(x), q_i(x)), one minus the total-variation
 * distance; [LB] "Acceptance Rate and Total Variation Distance" defines
 * TV(p, q) = (1/2) sum_x |p(x) - q(x)|; [MN] 3.2 measures the rate as
 * sum_t min(p_t, q_t).  Both sums are taken here straight from their
 * definitions, in token order, over p_i and q_i processed exactly as in
 * oracle_verify_sample; neither is derived from the other.
 *
 * target [B, k+1, V] (rows 0..k-1 used), draft [B, k, V]
 * beta [B, k], tv [B, k] (tv may be NULL): NaN where either row of the pair
 *      has a data error (R7)
 * Returns ORC_BAD_ARGUMENT, or the OR of (1 << status) over failed rows.
 */
int oracle_acceptance_k(const void *target, const void *draft, int dtype,
                        int B, int k, int V, double T, double top_p, int top_k,
                        double *beta, double *tv)
{
    if (!target || !draft || !beta || B < 0 || k < 1 || V < 1 ||
        (dtype != ORC_F32 && dtype != ORC_BF16) || !(T > 0.0) ||
        !(top_p > 0.0) || top_p > 1.0)
        return ORC_BAD_ARGUMENT;
    const size_t esz = dtype == ORC_F32 ? 4 : 2;
    double *p = (double *)malloc((size_t)V * sizeof *p);
    double *q = (double *)malloc((size_t)V * sizeof *q);
    int errors = 0;
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < k; ++i) {
            const char *prow = (const char *)target + ((size_t)b * (k + 1) + i) * V * esz;
            const char *qrow = (const char *)draft + ((size_t)b * k + i) * V * esz;
            int sp = oracle_process_row_k(prow, dtype, V, T, top_p, top_k, p, NULL);
            int sq = oracle_process_row_k(qrow, dtype, V, T, top_p, top_k, q, NULL);
            double overlap = NAN, dist = NAN;
            if (sp != ORC_OK) errors |= 1 << sp;
            if (sq != ORC_OK) errors |= 1 << sq;
            if (sp == ORC_OK && sq == ORC_OK) {
                overlap = 0.0;
                dist = 0.0;
                for (int x = 0; x < V; ++x) {
                    overlap += p[x] < q[x] ? p[x] : q[x];
                    dist += fabs(p[x] - q[x]);
                }
                dist *= 0.5;
            }
            beta[(size_t)b * k + i] = overlap;
            if (tv) tv[(size_t)b * k + i] = dist;
        }
    }
    free(p);
    free(q);
    return errors;
}

/* The same three entry points without top-k. */
int oracle_verify_sample(const void *target, const void *draft, int dtype,
                         const int32_t *tokens, const float *uniforms,
                         int B, int k, int V, double T, double top_p,
                         int mode, int32_t *out_tokens, int32_t *out_num,
                         double *dbg, double *row_info)
{
    return oracle_verify_sample_k(target, draft, dtype, tokens, uniforms, B, k, V, T, top_p,
                                  0, mode, out_tokens, out_num, dbg, row_info);
}

int oracle_verify_sample_probs(const void *target, const float *draft_probs,
                               int dtype, const int32_t *tokens,
                               const float *uniforms, int B, int k, int V,
                               double T, double top_p, int32_t *out_tokens,
                               int32_t *out_num, double *dbg, double *row_info)
{
    return oracle_verify_sample_probs_k(target, draft_probs, dtype, tokens, uniforms, B, k, V,
                                        T, top_p, 0, out_tokens, out_num, dbg, row_info);
}

int oracle_acceptance(const void *target, const void *draft, int dtype,
                      int B, int k, int V, double T, double top_p,
                      double *beta, double *tv)
{
    return oracle_acceptance_k(target, draft, dtype, B, k, V, T, top_p, 0, beta, tv);
}

/* -------------------------------------------------------- tree verify */

/*
 * Depth of every node of a flattened tree; parents[0] = -1 (the root, the
 * last committed token) and 0 <= parents[n] < n otherwise (a topological,
 * e.g. breadth-first, flattening).  Returns 0, or ORC_TREE_SHAPE.
 */
static int tree_depths(const int32_t *parents, int N, int32_t *depth)
{
    if (N < 1 || parents[0] != -1) return ORC_TREE_SHAPE;
    depth[0] = 0;
    for (int n = 1; n < N; ++n) {
        if (parents[n] < 0 || parents[n] >= n) return ORC_TREE_SHAPE;
        depth[n] = depth[parents[n]] + 1;
    }
    return ORC_OK;
}

/*
 * Ancestor relation of the flattened tree: mask[i*N + j] = 1 iff j == i or
 * j is an ancestor of i -- the "may attend" entries of the tree attention
 * mask of [LZ] "Tree verification" and [LB] (M_ij = 0 there, -inf
 * elsewhere).  Returns 0 or ORC_TREE_SHAPE.
 */
int oracle_ancestor_mask(const int32_t *parents, int N, uint8_t *mask)
{
    int32_t *depth = (int32_t *)malloc((size_t)N * sizeof *depth);
    int status = tree_depths(parents, N, depth);
    free(depth);
    if (status != ORC_OK) return status;
    memset(mask, 0, (size_t)N * N);
    for (int i = 0; i < N; ++i)
        for (int a = i; a >= 0; a = parents[a]) mask[(size_t)i * N + a] = 1;
    return ORC_OK;
}

/*
 * Tree attention inputs for B candidate trees (the step just before the
 * target pass that verify reads): [LZ] "Tree verification" -- every node
 * attends to the context and to its own ancestors only, and nodes at the
 * same depth get the same position index (for RoPE); [LB] "Tree-Based
 * Verification and Custom Attention Masks": M_ij = 0 where j is an
 * ancestor of i, -inf elsewhere.
 *
 * parents [B, N]  each sequence's tree, as for oracle_verify_tree
 * pos0    [B]     position index of each tree's root (NULL: all 0)
 * mask    [B, N, N] (optional): 1 iff j == i or j is an ancestor of i
 * pos     [B, N]  (optional): pos0[b] + depth(n)
 * A sequence whose parents are not a rooted tree in topological order gets
 * an all-zero mask and positions -1.  Returns ORC_BAD_ARGUMENT, or the OR
 * of (1 << ORC_TREE_SHAPE) if any tree failed.
 */
int oracle_tree_mask(const int32_t *parents, const int32_t *pos0, int B, int N,
                     uint8_t *mask, int32_t *pos)
{
    if (!parents || B < 0 || N < 1) return ORC_BAD_ARGUMENT;
    int32_t *depth = (int32_t *)malloc((size_t)N * sizeof *depth);
    int errors = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parents + (size_t)b * N;
        uint8_t *m = mask ? mask + (size_t)b * N * N : NULL;
        int32_t *pb = pos ? pos + (size_t)b * N : NULL;
        int status = tree_depths(par, N, depth);
        if (status != ORC_OK) {
            errors |= 1 << status;
            if (m) memset(m, 0, (size_t)N * N);
            if (pb)
                for (int n = 0; n < N; ++n) pb[n] = -1;
            continue;
        }
        if (m) {
            memset(m, 0, (size_t)N * N);
            for (int i = 0; i < N; ++i)
                for (int a = i; a >= 0; a = par[a]) m[(size_t)i * N + a] = 1;
        }
        if (pb)
            for (int n = 0; n < N; ++n) pb[n] = (pos0 ? pos0[b] : 0) + depth[n];
    }
    free(depth);
    return errors;
}

/*
 * Greedy tree verification ([LZ] "Tree verification": keep the longest
 * accepted root-to-leaf path; [LB] "Tree-Based Verification"), reading R6.
 *
 * target      [B, N, V]  logits of every flattened node
 * parents     [N]        parents[0] = -1, 0 <= parents[n] < n
 * node_tokens [B, N]     candidate token of each node (the root's ignored)
 * D                      the tree's depth bound: every node has depth <= D
 * out_tokens  [B, D+1]   accepted path tokens, then the bonus argmax, -1 pad
 * out_num     [B]        accepted depth d (0..D), -1 on a data error
 * out_path    [B, D+1]   node ids root, n_1, ..., n_d, -1 pad (optional)
 * Returns ORC_BAD_ARGUMENT, or the OR of (1 << status) over failures.
 */
int oracle_verify_tree(const void *target, int dtype, const int32_t *parents,
                       const int32_t *node_tokens, int B, int N, int V, int D,
                       int32_t *out_tokens, int32_t *out_num,
                       int32_t *out_path)
{
    if (!target || !parents || !node_tokens || !out_tokens || !out_num ||
        B < 0 || N < 1 || V < 1 || D < 0 ||
        (dtype != ORC_F32 && dtype != ORC_BF16))
        return ORC_BAD_ARGUMENT;
    const size_t esz = dtype == ORC_F32 ? 4 : 2;
    const int W = D + 1;
    int32_t *depth = (int32_t *)malloc((size_t)N * sizeof *depth);
    int32_t *g = (int32_t *)malloc((size_t)N * sizeof *g);
    uint8_t *acc = (uint8_t *)malloc((size_t)N);
    int32_t *path = (int32_t *)malloc((size_t)N * sizeof *path);
    int errors = 0;

    int shape = tree_depths(parents, N, depth);
    for (int n = 0; n < N && shape == ORC_OK; ++n)
        if (depth[n] > D) shape = ORC_TREE_SHAPE;

    for (int b = 0; b < B; ++b) {
        int32_t *ot = out_tokens + (size_t)b * W;
        int32_t *op = out_path ? out_path + (size_t)b * W : NULL;
        const int32_t *tok = node_tokens + (size_t)b * N;
        int bad = shape != ORC_OK ? 1 << shape : 0;
        for (int n = 1; n < N; ++n)
            if (tok[n] < 0 || tok[n] >= V) bad |= 1 << ORC_TOKEN_RANGE;
        for (int n = 0; n < N; ++n) {
            const char *row = (const char *)target + ((size_t)b * N + n) * V * esz;
            int status = oracle_argmax_row(row, dtype, V, &g[n]);
            if (status != ORC_OK) bad |= 1 << status;
        }
        if (bad) {
            errors |= bad;
            fail_sequence(ot, W, &out_num[b]);
            if (op)
                for (int i = 0; i < W; ++i) op[i] = -1;
            continue;
        }

        int best = 0;
        acc[0] = 1;
        for (int n = 1; n < N; ++n) {
            int par = parents[n];
            acc[n] = acc[par] && tok[n] == g[par];
            if (acc[n] && depth[n] > depth[best]) best = n;
        }
        int d = depth[best];
        for (int n = best, i = d; i >= 0; n = parents[n], --i) path[i] = n;

        for (int i = 0; i < W; ++i) ot[i] = -1;
        for (int i = 0; i < d; ++i) ot[i] = tok[path[i + 1]];
        ot[d] = g[best];
        if (op) {
            for (int i = 0; i < W; ++i) op[i] = -1;
            for (int i = 0; i <= d; ++i) op[i] = path[i];
        }
        out_num[b] = d;
    }
    free(depth);
    free(g);
    free(acc);
    free(path);
    return errors;
}

/*
 * Stochastic tree verification, reading R11.  [LZ] "Tree verification"
 * names SpecInfer's lossless multi-candidate acceptance rule for sampling
 * without stating it.  Reading: the children of node n are candidates
 * drawn independently from q_n (draft row n).  At the current node the
 * children are tried in flattened order; child c is accepted iff
 *   u_c * q_n(x_c) < p'(x_c)
 * where p' starts as p_n (target row n) and, after each rejected child,
 * becomes the residual max(0, p' - q_n) normalised (kept when that residual
 * is zero everywhere, R4).  An accepted child becomes the current node; when
 * every child is rejected, or the node has none, the final token is drawn
 * from p' by inverse CDF (R3) with the final uniform.  Each try is the
 * one-token rule against target p', so every emitted position follows p.
 *
 * target [B, N, V], draft [B, N, V] (row n: the law node n's children were
 * drawn from), parents [N] (as oracle_verify_tree), node_tokens [B, N],
 * uniforms [B, N]: entry c >= 1 for node c's test, entry 0 for the final
 * draw.  T, top_p, top_k process target and draft rows alike.
 * out_tokens [B, D+1] (path tokens, drawn token, -1), out_num [B] (depth,
 * -1 on a data error), out_path [B, D+1] (optional),
 * margin [B] (optional): the smallest distance of a uniform used to its
 * decision boundary (|u - p'/q| over the tests run with q > 0, |u - C/S| at
 * the drawn token's two CDF edges).
 */
int oracle_verify_tree_sample(const void *target, const void *draft, int dtype,
                              const int32_t *parents, const int32_t *node_tokens,
                              const float *uniforms, int B, int N, int V, int D,
                              double T, double top_p, int top_k, int32_t *out_tokens,
                              int32_t *out_num, int32_t *out_path, double *margin)
{
    if (!target || !draft || !parents || !node_tokens || !uniforms || !out_tokens ||
        !out_num || B < 0 || N < 1 || V < 1 || D < 0 ||
        (dtype != ORC_F32 && dtype != ORC_BF16) || !(T > 0.0) || !(top_p > 0.0) ||
        top_p > 1.0)
        return ORC_BAD_ARGUMENT;
    const size_t esz = dtype == ORC_F32 ? 4 : 2;
    const int W = D + 1;
    int32_t *depth = (int32_t *)malloc((size_t)N * sizeof *depth);
    int32_t *path = (int32_t *)malloc((size_t)W * sizeof *path);
    double *p = (double *)malloc((size_t)N * V * sizeof *p);
    double *q = (double *)malloc((size_t)N * V * sizeof *q);
    double *pr = (double *)malloc((size_t)V * sizeof *pr);
    int errors = 0;

    int shape = tree_depths(parents, N, depth);
    for (int n = 0; n < N && shape == ORC_OK; ++n)
        if (depth[n] > D) shape = ORC_TREE_SHAPE;

    for (int b = 0; b < B; ++b) {
        int32_t *ot = out_tokens + (size_t)b * W;
        int32_t *op = out_path ? out_path + (size_t)b * W : NULL;
        const int32_t *tok = node_tokens + (size_t)b * N;
        const float *ub = uniforms + (size_t)b * N;
        int bad = shape != ORC_OK ? 1 << shape : 0;
        for (int n = 1; n < N; ++n)
            if (tok[n] < 0 || tok[n] >= V) bad |= 1 << ORC_TOKEN_RANGE;
        for (int n = 0; n < N; ++n)
            if (!(ub[n] >= 0.0f && ub[n] < 1.0f)) bad |= 1 << ORC_UNIFORM_RANGE;
        for (int n = 0; n < N; ++n) {
            const char *trow = (const char *)target + ((size_t)b * N + n) * V * esz;
            const char *drow = (const char *)draft + ((size_t)b * N + n) * V * esz;
            int s1 = oracle_process_row_k(trow, dtype, V, T, top_p, top_k, p + (size_t)n * V, NULL);
            int s2 = oracle_process_row_k(drow, dtype, V, T, top_p, top_k, q + (size_t)n * V, NULL);
            if (s1 != ORC_OK) bad |= 1 << s1;
            if (s2 != ORC_OK) bad |= 1 << s2;
        }
        if (margin) margin[b] = INFINITY;
        if (bad) {
            errors |= bad;
            fail_sequence(ot, W, &out_num[b]);
            if (op)
                for (int i = 0; i < W; ++i) op[i] = -1;
            continue;
        }

        double mg = INFINITY;
        int cur = 0, d = 0;
        path[0] = 0;
        int32_t drawn = -1;
        for (;;) {
            const double *qn = q + (size_t)cur * V;
            memcpy(pr, p + (size_t)cur * V, (size_t)V * sizeof *pr);
            int next = -1;
            for (int c = 1; c < N && next < 0; ++c) {
                if (parents[c] != cur) continue;
                const double P = pr[tok[c]], Q = qn[tok[c]];
                if (Q > 0.0 && fabs((double)ub[c] - P / Q) < mg) mg = fabs((double)ub[c] - P / Q);
                if ((double)ub[c] * Q < P) {
                    next = c;
                    break;
                }
                double S = 0.0;
                for (int x = 0; x < V; ++x) {
                    double r = pr[x] - qn[x];
                    S += r > 0.0 ? r : 0.0;
                }
                if (S > 0.0)
                    for (int x = 0; x < V; ++x) {
                        double r = pr[x] - qn[x];
                        pr[x] = r > 0.0 ? r / S : 0.0;
                    }
            }
            if (next < 0) {
                double edges[3];
                drawn = oracle_inverse_cdf(pr, V, (double)ub[0], edges);
                double e0 = fabs((double)ub[0] - edges[1] / edges[0]);
                double e1 = fabs((double)ub[0] - edges[2] / edges[0]);
                if (e0 < mg) mg = e0;
                if (e1 < mg) mg = e1;
                break;
            }
            cur = next;
            path[++d] = next;
        }
        for (int i = 0; i < W; ++i) ot[i] = -1;
        for (int i = 0; i < d; ++i) ot[i] = tok[path[i + 1]];
        ot[d] = drawn;
        if (op) {
            for (int i = 0; i < W; ++i) op[i] = -1;
            for (int i = 0; i <= d; ++i) op[i] = path[i];
        }
        out_num[b] = d;
        if (margin) margin[b] = mg;
    }
    free(depth);
    free(path);
    free(p);
    free(q);
    free(pr);
    return errors;
}
