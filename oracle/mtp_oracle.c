/*
 * Oracle for the centroid-masked sparse LM head of the Gemma4 MTP drafter.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library.  It shares no code, header, table or
 * helper with the CUDA library; both read their inputs from the seeded
 * generator and nothing else.
 *
 * What it follows: "Add Gemma4 MTP speculative decoding with centroids masking"
 * (vLLM compare view), file vllm/model_executor/models/gemma4_mtp.py, class
 * Gemma4MTPMaskedEmbedder:
 *   - __init__: vocab_size_per_centroid = vocab_size // num_centroids; the
 *     centroid table is a bias-free Linear(hidden_size -> num_centroids), so it
 *     is stored [C, H]; token_ordering is a [V] buffer viewed as [C, V/C].
 *   - _select_and_score: centroid scores = Linear(h); top-K centroid indices;
 *     selected = token_ordering.view(C, V/C)[topk] (ordered position -> token
 *     id); candidate rows = lm_head_weight[selected] (token-id order); sparse
 *     logits = per-row dot products with the candidate rows.
 *   - get_top_tokens: the token id of the largest sparse logit.
 *   - forward: full-vocabulary row, selected tokens get their logit, every
 *     other token gets -inf (the docstring's reading; see below).
 *
 * Readings where the page is silent or inconsistent (each is listed in the
 * design notes with its reason):
 *   - scores, logits and all sums are fp64 from the exact bf16 inputs;
 *   - top-K ties: lower centroid index wins; the selected list is ordered by
 *     (score desc, index asc), like a sorted topk;
 *   - argmax ties: lower token id wins;
 *   - fill value: -inf (the docstring), not the dtype's finite minimum;
 *   - variable clusters: cluster c owns ordered positions [off[c], off[c+1]);
 *     off == NULL means uniform clusters of V/C positions (the page's view());
 *   - a row whose selected clusters are all empty has no candidate: its token
 *     is -1 and its max logit -inf.
 *
 * Reference-fidelity options (the `flags` argument; 0 is the reading above):
 *   ORC_FLAG_FILL_FINFO_MIN  forward fills with bf16's finite minimum, the
 *                            value the page's code uses (finfo(dtype).min);
 *   ORC_FLAG_BF16_SCORES     the selection uses the centroid scores rounded to
 *                            bf16, as the page's bf16 Linear returns them;
 *   ORC_FLAG_BF16_LOGITS     the sparse (and dense) logits are rounded to bf16,
 *                            as the page's bf16 einsum returns them, before the
 *                            argmax and the scatter.
 * The dense comparator can also apply the final logit softcap of the page's
 * dense path (Gemma4MTP.compute_logits through the logits processor):
 * cap * tanh(logit / cap) for cap > 0, before any bf16 rounding.
 * Rounding to bf16 is round-to-nearest-even of the exact fp64 value to 8
 * significant bits (bf16's exponent range, its subnormals included).
 *
 * Parity pins live in tests/test_oracle_pins.py (hand-worked example, brute
 * force top-K by subset enumeration, K=C and C=1 dense identities, integer
 * exact cases, invariants).
 *
 * Plain C99, no threads, no intrinsics; compiled with gcc -O2 (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_NOMEM -2

#define ORC_FLAG_FILL_FINFO_MIN 1
#define ORC_FLAG_BF16_SCORES 2
#define ORC_FLAG_BF16_LOGITS 4

/* bf16's largest finite value, (2 - 2^-7) * 2^127. */
#define ORC_BF16_MAX 3.3895313892515355e38

/* x rounded to the nearest bf16 value, ties to even: 8 significant bits while
 * |x| >= 2^-126, a fixed quantum of 2^-133 below (bf16 subnormals), infinity
 * beyond ORC_BF16_MAX after rounding. */
double orc_round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x))
        return x;
    int e;
    frexp(x, &e);                 /* |x| in [2^(e-1), 2^e) */
    int q = e - 8;                /* exponent of the last of 8 significant bits */
    if (q < -133)
        q = -133;
    double r = ldexp(nearbyint(ldexp(x, -q)), q);   /* nearbyint: nearest, ties even */
    if (fabs(r) > ORC_BF16_MAX)
        return r > 0 ? INFINITY : -INFINITY;
    return r;
}

/* bf16 bit pattern -> exact double. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Dot product of a bf16 row of the hidden states with a bf16 table row. */
static double dot_bf16(const uint16_t *x, const uint16_t *w, int64_t n)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i)
        s += bf16_value(x[i]) * bf16_value(w[i]);
    return s;
}

/* First and one-past-last ordered position owned by centroid c. */
static void cluster_range(int64_t c, int64_t V, int64_t C, const int32_t *off,
                          int64_t *lo, int64_t *hi)
{
    if (off) {
        *lo = off[c];
        *hi = off[c + 1];
    } else {
        int64_t s = V / C;
        *lo = c * s;
        *hi = (c + 1) * s;
    }
}

/* Step 1 (Linear centroid projection): scores[b, c] = sum_h h[b,h] Wc[c,h]
 * for rows b in [b0, b1); scores is indexed by absolute row. */
int orc_centroid_scores(const uint16_t *hidden, int64_t b0, int64_t b1, int64_t H,
                        const uint16_t *centroid_w, int64_t C, double *scores)
{
    if (!hidden || !centroid_w || !scores || H <= 0 || C <= 0 || b0 < 0 || b1 < b0)
        return ORC_ERR_ARG;
    for (int64_t b = b0; b < b1; ++b)
        for (int64_t c = 0; c < C; ++c)
            scores[b * C + c] = dot_bf16(hidden + b * H, centroid_w + c * H, H);
    return ORC_OK;
}

typedef struct {
    double score;
    int32_t index;
} scored_index;

/* Sort order of the selection: larger score first, lower index on ties. */
static int by_score_desc_index_asc(const void *pa, const void *pb)
{
    const scored_index *a = (const scored_index *)pa;
    const scored_index *b = (const scored_index *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->index > b->index) - (a->index < b->index);
}

/* Step 2 (topk over centroid scores) for one row: sel[0..K) ordered by
 * (score desc, index asc).  margin = score of the K-th pick minus score of the
 * (K+1)-th (INFINITY when K == C). */
int orc_topk_row(const double *scores, int64_t C, int64_t K, int32_t *sel, double *margin)
{
    if (!scores || !sel || K <= 0 || K > C)
        return ORC_ERR_ARG;
    scored_index *all = (scored_index *)malloc((size_t)C * sizeof *all);
    if (!all)
        return ORC_ERR_NOMEM;
    for (int64_t c = 0; c < C; ++c) {
        all[c].score = scores[c];
        all[c].index = (int32_t)c;
    }
    qsort(all, (size_t)C, sizeof *all, by_score_desc_index_asc);
    for (int64_t k = 0; k < K; ++k)
        sel[k] = all[k].index;
    if (margin)
        *margin = (K < C) ? all[K - 1].score - all[K].score : INFINITY;
    free(all);
    return ORC_OK;
}

/* Number of candidate tokens of a selection (sum of the selected cluster sizes). */
static int64_t candidate_count(const int32_t *sel, int64_t K, int64_t V, int64_t C,
                               const int32_t *off)
{
    int64_t n = 0;
    for (int64_t k = 0; k < K; ++k) {
        int64_t lo, hi;
        cluster_range(sel[k], V, C, off, &lo, &hi);
        n += hi - lo;
    }
    return n;
}

/* Steps 3-4 (cluster -> token ids through token_ordering, gather of the
 * candidate lm_head rows, sparse dot products) for one row.  Candidates are
 * listed in selection order, then position order inside each cluster, which is
 * the order of the page's `selected` tensor.  tokens/logits hold at least
 * candidate_count() entries. */
static void select_and_score_row(const uint16_t *h_row, int64_t H,
                                 const uint16_t *embed_w, int64_t ld_embed,
                                 const int32_t *ordering, const int32_t *off,
                                 int64_t V, int64_t C, const int32_t *sel, int64_t K,
                                 int32_t *tokens, double *logits, int64_t flags)
{
    int64_t j = 0;
    for (int64_t k = 0; k < K; ++k) {
        int64_t lo, hi;
        cluster_range(sel[k], V, C, off, &lo, &hi);
        for (int64_t p = lo; p < hi; ++p) {
            int32_t t = ordering[p];
            tokens[j] = t;
            logits[j] = dot_bf16(h_row, embed_w + (int64_t)t * ld_embed, H);
            if (flags & ORC_FLAG_BF16_LOGITS)
                logits[j] = orc_round_bf16(logits[j]);
            ++j;
        }
    }
}

/* Step 5a (get_top_tokens) plus the margins used to keep test inputs away
 * from near-ties.  For rows [b0, b1):
 *   tokens[b]        token id of the largest sparse logit (lower id on ties),
 *                    -1 if the row has no candidate;
 *   max_logit[b]     that logit (-INFINITY if none);
 *   score_margin[b]  K-th minus (K+1)-th centroid score;
 *   logit_margin[b]  top-1 minus top-2 sparse logit (INFINITY if < 2 candidates);
 *   sel[b*K + k]     the selected centroids (optional);
 *   n_cand[b]        number of candidates (optional).
 * Output arrays are indexed by absolute row. */
int orc_masked_topk_tokens(const uint16_t *hidden, int64_t b0, int64_t b1, int64_t H,
                           const uint16_t *centroid_w, int64_t C, int64_t K,
                           const uint16_t *embed_w, int64_t ld_embed, int64_t V,
                           const int32_t *ordering, const int32_t *off,
                           int32_t *tokens, double *max_logit, double *score_margin,
                           double *logit_margin, int32_t *sel_out, int64_t *n_cand, int64_t flags)
{
    if (!hidden || !centroid_w || !embed_w || !ordering || !tokens || H <= 0 || C <= 0 ||
        K <= 0 || K > C || V <= 0 || ld_embed < H || b0 < 0 || b1 < b0)
        return ORC_ERR_ARG;
    if (!off && V % C != 0)
        return ORC_ERR_ARG;
    double *scores = (double *)malloc((size_t)C * sizeof *scores);
    int32_t *sel = (int32_t *)malloc((size_t)K * sizeof *sel);
    if (!scores || !sel) {
        free(scores);
        free(sel);
        return ORC_ERR_NOMEM;
    }
    int rc = ORC_OK;
    for (int64_t b = b0; b < b1 && rc == ORC_OK; ++b) {
        const uint16_t *h_row = hidden + b * H;
        for (int64_t c = 0; c < C; ++c) {
            scores[c] = dot_bf16(h_row, centroid_w + c * H, H);
            if (flags & ORC_FLAG_BF16_SCORES)
                scores[c] = orc_round_bf16(scores[c]);
        }
        double smargin;
        rc = orc_topk_row(scores, C, K, sel, &smargin);
        if (rc != ORC_OK)
            break;
        int64_t n = candidate_count(sel, K, V, C, off);
        int32_t *cand_tok = (int32_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof *cand_tok);
        double *cand_log = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof *cand_log);
        if (!cand_tok || !cand_log) {
            free(cand_tok);
            free(cand_log);
            rc = ORC_ERR_NOMEM;
            break;
        }
        select_and_score_row(h_row, H, embed_w, ld_embed, ordering, off, V, C, sel, K,
                             cand_tok, cand_log, flags);
        int32_t best_t = -1;
        double best = -INFINITY, second = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            double v = cand_log[j];
            int32_t t = cand_tok[j];
            if (best_t < 0 || v > best || (v == best && t < best_t)) {
                if (best_t >= 0)
                    second = best;
                best = v;
                best_t = t;
            } else if (v > second) {
                second = v;
            }
        }
        tokens[b] = best_t;
        if (max_logit)
            max_logit[b] = best;
        if (score_margin)
            score_margin[b] = smargin;
        if (logit_margin)
            logit_margin[b] = (n >= 2) ? best - second : INFINITY;
        if (sel_out)
            memcpy(sel_out + b * K, sel, (size_t)K * sizeof *sel);
        if (n_cand)
            n_cand[b] = n;
        free(cand_tok);
        free(cand_log);
    }
    free(scores);
    free(sel);
    return rc;
}

/* Step 5b (forward): full-vocabulary rows [b0, b1) of out[b, V]: the sparse
 * logit at each selected token id, -INFINITY everywhere else. */
int orc_masked_scatter_logits(const uint16_t *hidden, int64_t b0, int64_t b1, int64_t H,
                              const uint16_t *centroid_w, int64_t C, int64_t K,
                              const uint16_t *embed_w, int64_t ld_embed, int64_t V,
                              const int32_t *ordering, const int32_t *off, double *out,
                              int64_t flags)
{
    if (!hidden || !centroid_w || !embed_w || !ordering || !out || H <= 0 || C <= 0 ||
        K <= 0 || K > C || V <= 0 || ld_embed < H || b0 < 0 || b1 < b0)
        return ORC_ERR_ARG;
    if (!off && V % C != 0)
        return ORC_ERR_ARG;
    double *scores = (double *)malloc((size_t)C * sizeof *scores);
    int32_t *sel = (int32_t *)malloc((size_t)K * sizeof *sel);
    if (!scores || !sel) {
        free(scores);
        free(sel);
        return ORC_ERR_NOMEM;
    }
    int rc = ORC_OK;
    for (int64_t b = b0; b < b1 && rc == ORC_OK; ++b) {
        const uint16_t *h_row = hidden + b * H;
        double *row = out + b * V;
        const double fill = (flags & ORC_FLAG_FILL_FINFO_MIN) ? -ORC_BF16_MAX : -INFINITY;
        for (int64_t t = 0; t < V; ++t)
            row[t] = fill;
        for (int64_t c = 0; c < C; ++c) {
            scores[c] = dot_bf16(h_row, centroid_w + c * H, H);
            if (flags & ORC_FLAG_BF16_SCORES)
                scores[c] = orc_round_bf16(scores[c]);
        }
        rc = orc_topk_row(scores, C, K, sel, NULL);
        if (rc != ORC_OK)
            break;
        int64_t n = candidate_count(sel, K, V, C, off);
        int32_t *cand_tok = (int32_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof *cand_tok);
        double *cand_log = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof *cand_log);
        if (!cand_tok || !cand_log) {
            free(cand_tok);
            free(cand_log);
            rc = ORC_ERR_NOMEM;
            break;
        }
        select_and_score_row(h_row, H, embed_w, ld_embed, ordering, off, V, C, sel, K,
                             cand_tok, cand_log, flags);
        for (int64_t j = 0; j < n; ++j)
            row[cand_tok[j]] = cand_log[j];
        free(cand_tok);
        free(cand_log);
    }
    free(scores);
    free(sel);
    return rc;
}

/* The sparse pair of _select_and_score for one row b: logits and token ids of
 * the candidates in the page's order (selection order, then position order).
 * cap = capacity of the two arrays; *n receives the candidate count (the call
 * fails with ORC_ERR_ARG if it exceeds cap). */
int orc_select_and_score_row(const uint16_t *hidden, int64_t b, int64_t H,
                             const uint16_t *centroid_w, int64_t C, int64_t K,
                             const uint16_t *embed_w, int64_t ld_embed, int64_t V,
                             const int32_t *ordering, const int32_t *off,
                             int32_t *tokens, double *logits, int64_t cap, int64_t *n,
                             int64_t flags)
{
    if (!hidden || !centroid_w || !embed_w || !ordering || !tokens || !logits || !n ||
        K <= 0 || K > C || (!off && V % C != 0))
        return ORC_ERR_ARG;
    double *scores = (double *)malloc((size_t)C * sizeof *scores);
    int32_t *sel = (int32_t *)malloc((size_t)K * sizeof *sel);
    if (!scores || !sel) {
        free(scores);
        free(sel);
        return ORC_ERR_NOMEM;
    }
    const uint16_t *h_row = hidden + b * H;
    for (int64_t c = 0; c < C; ++c) {
        scores[c] = dot_bf16(h_row, centroid_w + c * H, H);
        if (flags & ORC_FLAG_BF16_SCORES)
            scores[c] = orc_round_bf16(scores[c]);
    }
    int rc = orc_topk_row(scores, C, K, sel, NULL);
    if (rc == ORC_OK) {
        *n = candidate_count(sel, K, V, C, off);
        if (*n > cap)
            rc = ORC_ERR_ARG;
        else
            select_and_score_row(h_row, H, embed_w, ld_embed, ordering, off, V, C, sel, K,
                                 tokens, logits, flags);
    }
    free(scores);
    free(sel);
    return rc;
}

/* Dense comparator (the LogitsProcessor path without softcapping): out[b, t]
 * = sum_h h[b,h] E[t,h] for rows [b0, b1) and every token t < V. */
int orc_dense_logits(const uint16_t *hidden, int64_t b0, int64_t b1, int64_t H,
                     const uint16_t *embed_w, int64_t ld_embed, int64_t V, double *out,
                     int64_t flags, double softcap)
{
    if (!hidden || !embed_w || !out || H <= 0 || V <= 0 || ld_embed < H || b0 < 0 || b1 < b0)
        return ORC_ERR_ARG;
    for (int64_t b = b0; b < b1; ++b)
        for (int64_t t = 0; t < V; ++t)
        {
            out[b * V + t] = dot_bf16(hidden + b * H, embed_w + t * ld_embed, H);
            if (softcap > 0.0)
                out[b * V + t] = softcap * tanh(out[b * V + t] / softcap);
            if (flags & ORC_FLAG_BF16_LOGITS)
                out[b * V + t] = orc_round_bf16(out[b * V + t]);
        }
    return ORC_OK;
}

/* Dense logits at n sampled (row, token) pairs: out[i] = h[rows[i]] . E[tokens[i]]. */
int orc_dense_logits_at(const uint16_t *hidden, int64_t H, const uint16_t *embed_w,
                        int64_t ld_embed, const int64_t *rows, const int64_t *tokens, int64_t n,
                        double *out)
{
    if (!hidden || !embed_w || !rows || !tokens || !out || H <= 0 || ld_embed < H || n < 0)
        return ORC_ERR_ARG;
    for (int64_t i = 0; i < n; ++i)
        out[i] = dot_bf16(hidden + rows[i] * H, embed_w + tokens[i] * ld_embed, H);
    return ORC_OK;
}

/* 1 if ordering is a permutation of 0..V-1 (a precondition, not checked by
 * the CUDA library), else 0. */
int orc_is_permutation(const int32_t *ordering, int64_t V)
{
    if (!ordering || V <= 0)
        return 0;
    unsigned char *seen = (unsigned char *)calloc((size_t)V, 1);
    if (!seen)
        return 0;
    int ok = 1;
    for (int64_t p = 0; p < V && ok; ++p) {
        int32_t t = ordering[p];
        if (t < 0 || t >= V || seen[t])
            ok = 0;
        else
            seen[t] = 1;
    }
    free(seen);
    return ok;
}
