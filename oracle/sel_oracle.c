/*
 * sel_oracle.c -- plain, slow CPU oracle for decode-step token selection.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The product path (the CUDA library
 * and its Python binding) never loads, links or calls it, and the two share
 * no code, header, table or helper: this file includes only the C standard
 * library.
 *
 * Arithmetic is double precision throughout. The inputs are the same fp32
 * logits and fp32 uniforms the GPU path reads; each is widened to double on
 * load. Every routine is a direct statement of its definition: linear scans,
 * a full stable sort, sums taken in a fixed order. Nothing is blocked, fused
 * or reordered.
 *
 * Sources (page -- section):
 *  [Ch21]  "Ch 21 -- Sampling, argmax, and grammar" (Muser book chapter)
 *          21.3 / Figure 21.1: argmax compares with strict '>', so a tie keeps
 *               the lower index;
 *          21.4: the greedy serving variant latches any NaN/Inf logit and the
 *               reduction then returns 0xffffffff (fail closed);
 *          21.6: the CPU first-maximum scan and the finite check that refuses
 *               a row with a nonfinite entry;
 *          21.7: the sampler chain filters top-k before top-p;
 *          21.9: speculative acceptance: accept with probability min(p/q, 1),
 *               q <= 0 accepts; on the first rejection draw from the
 *               normalised residual max(p - q, 0), or from p when the
 *               residual total is <= 0; if all are accepted draw from the
 *               last target row.
 *  [Spec]  "Speculative-decoding acceptance rules" (mlxcel docs)
 *          "Argmax-against-argmax": accept iff the draft equals the target
 *               argmax, emit the argmax on a mismatch;
 *          "Modified rejection sampling": accept iff u*q(t) <= p(t); on the
 *               first rejection draw from normalize(relu(p - q)) and stop; if
 *               every draft is accepted draw a bonus token from p;
 *          "RNG dependency": one uniform per tested position, one per draw;
 *               temperature 0 is the argmax rule and draws nothing.
 *  [PR49]  "llama.cpp pull 49" (on-device logits top-k)
 *          "Change": each row yields its k largest logits with their token
 *               ids; a chain with top-k first needs only those k candidates,
 *               and top-p / min-p then act on them.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - sampling applies temperature first (z = x / T), then top-k on z, softmax
 *    over the candidates, top-p, min-p, renormalise, and draws by inverse CDF
 *    with the candidates in (probability desc, id asc) order; the
 *    temperature-last order filters with T = 1 probabilities and draws from
 *    the tempered ones;
 *  - top-p keeps the shortest prefix whose cumulative mass reaches top_p
 *    (the crossing token included, at least one token); min-p keeps
 *    P_i >= min_p * P_max;
 *  - the residual and bonus draws of speculative acceptance walk the
 *    vocabulary in ascending token id;
 *  - a uniform outside [0, 1) or a nonfinite logit makes the row (sequence)
 *    invalid: every output id is 0xFFFFFFFF;
 *  - temperature 0 means greedy: sampling returns the argmax with
 *    probability 1; speculative acceptance uses the argmax rule.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_INVALID 0xFFFFFFFFu

/* ----------------------------------------------------------------------- */
/* helpers                                                                 */
/* ----------------------------------------------------------------------- */

/* [Ch21] 21.6: a row with any NaN or +-Inf entry is refused outright. */
static int row_is_finite(const float *x, uint32_t n)
{
    for (uint32_t i = 0; i < n; ++i)
        if (!isfinite(x[i]))
            return 0;
    return 1;
}

static int uniform_is_valid(float u)
{
    return u >= 0.0f && u < 1.0f; /* false for NaN as well */
}

/*
 * Stable merge sort of ids[0..n) by key[id] descending. Stability keeps the
 * lower id first among equal keys because ids start in ascending order.
 * Bottom-up: runs of width 1, 2, 4, ... are merged from ids into tmp and back.
 */
static void stable_sort_desc(uint32_t *ids, uint32_t *tmp, const double *key,
                             size_t n)
{
    uint32_t *src = ids, *dst = tmp;
    for (size_t width = 1; width < n; width *= 2) {
        for (size_t lo = 0; lo < n; lo += 2 * width) {
            size_t mid = lo + width < n ? lo + width : n;
            size_t hi = lo + 2 * width < n ? lo + 2 * width : n;
            size_t a = lo, b = mid, o = lo;
            while (a < mid && b < hi) {
                /* take from the right run only if strictly greater */
                if (key[src[b]] > key[src[a]])
                    dst[o++] = src[b++];
                else
                    dst[o++] = src[a++];
            }
            while (a < mid)
                dst[o++] = src[a++];
            while (b < hi)
                dst[o++] = src[b++];
        }
        uint32_t *t = src;
        src = dst;
        dst = t;
    }
    if (src != ids)
        memcpy(ids, src, n * sizeof(uint32_t));
}

/* ids[0..n) sorted by x descending, ties by lower id. Caller frees. */
static uint32_t *sorted_ids_desc(const double *key, uint32_t n)
{
    uint32_t *ids = (uint32_t *)malloc((size_t)n * sizeof(uint32_t));
    uint32_t *tmp = (uint32_t *)malloc((size_t)n * sizeof(uint32_t));
    for (uint32_t i = 0; i < n; ++i)
        ids[i] = i;
    stable_sort_desc(ids, tmp, key, n);
    free(tmp);
    return ids;
}

/* p[i] = exp(x[i]/T - max_j x[j]/T) / sum_j exp(...), summed in id order. */
static void softmax_row(const float *x, uint32_t V, double T, double *p)
{
    double m = -INFINITY;
    for (uint32_t i = 0; i < V; ++i) {
        double z = (double)x[i] / T;
        if (z > m)
            m = z;
    }
    double s = 0.0;
    for (uint32_t i = 0; i < V; ++i) {
        p[i] = exp((double)x[i] / T - m);
        s += p[i];
    }
    for (uint32_t i = 0; i < V; ++i)
        p[i] /= s;
}

/*
 * Inverse-CDF draw over w[0..n) (non-negative weights, visited in index
 * order): C_i = (w_0 + ... + w_i) / W, return the first i with u < C_i; if
 * rounding leaves none, the last i with w_i > 0. *margin receives
 * min_i |u - C_i| over every boundary except the final one (which is 1).
 */
static int cmp_u64(const void *a, const void *b)
{
    uint64_t x = *(const uint64_t *)a, y = *(const uint64_t *)b;
    return x < y ? -1 : (x > y ? 1 : 0);
}

static uint32_t inverse_cdf(const double *w, uint32_t n, double u,
                            double *margin)
{
    double W = 0.0;
    for (uint32_t i = 0; i < n; ++i)
        W += w[i];
    double c = 0.0, best_margin = INFINITY;
    uint32_t pick = ORC_INVALID, last_pos = ORC_INVALID;
    for (uint32_t i = 0; i < n; ++i) {
        if (w[i] > 0.0)
            last_pos = i;
        c += w[i];
        double C = c / W;
        if (pick == ORC_INVALID && u < C)
            pick = i;
    }
    /* boundaries strictly before the last positive weight */
    c = 0.0;
    for (uint32_t i = 0; i < n; ++i) {
        c += w[i];
        if (last_pos != ORC_INVALID && i >= last_pos)
            break;
        if (w[i] > 0.0) {
            double d = fabs(u - c / W);
            if (d < best_margin)
                best_margin = d;
        }
    }
    if (margin)
        *margin = best_margin;
    if (pick == ORC_INVALID || (last_pos != ORC_INVALID && pick > last_pos))
        pick = last_pos;
    return pick;
}

/* ----------------------------------------------------------------------- */
/* argmax                                                                  */
/* ----------------------------------------------------------------------- */

/*
 * [Ch21] 21.3, 21.6: first-maximum scan with strict '>', so the lowest index
 * attaining the maximum wins. [Ch21] 21.4: any nonfinite entry -> 0xFFFFFFFF.
 */
uint32_t orc_argmax_row(const float *x, uint32_t V)
{
    if (V == 0 || !row_is_finite(x, V))
        return ORC_INVALID;
    uint32_t best = 0;
    for (uint32_t i = 1; i < V; ++i)
        if ((double)x[i] > (double)x[best])
            best = i;
    return best;
}

void orc_argmax(const float *logits, uint32_t rows, uint32_t V,
                uint32_t *out_ids)
{
    for (uint32_t r = 0; r < rows; ++r)
        out_ids[r] = orc_argmax_row(logits + (size_t)r * V, V);
}

/*
 * [Ch21] 21.4, the greedy serving variant: a request's end-of-generation ids
 * are masked out inside the reduction only (the logits themselves stay
 * untouched), and the NaN/Inf latch still covers every logit of the row.
 * Definition used: the first maximum (strict '>') over the ids that are not
 * in `excluded`; ids >= V in the set are ignored; duplicates do not matter.
 * A nonfinite logit anywhere in the row (excluded or not), or a row whose ids
 * are all excluded, gives 0xFFFFFFFF.
 */
uint32_t orc_argmax_excluding_row(const float *x, uint32_t V,
                                  const uint32_t *excluded, uint32_t n_excluded)
{
    if (V == 0 || !row_is_finite(x, V))
        return ORC_INVALID;
    uint32_t best = ORC_INVALID;
    for (uint32_t i = 0; i < V; ++i) {
        int is_excluded = 0;
        for (uint32_t e = 0; e < n_excluded; ++e)
            if (excluded[e] == i)
                is_excluded = 1;
        if (is_excluded)
            continue;
        if (best == ORC_INVALID || (double)x[i] > (double)x[best])
            best = i;
    }
    return best;
}

void orc_argmax_excluding(const float *logits, uint32_t rows, uint32_t V,
                          const uint32_t *excluded, uint32_t n_excluded,
                          uint32_t *out_ids)
{
    for (uint32_t r = 0; r < rows; ++r)
        out_ids[r] = orc_argmax_excluding_row(logits + (size_t)r * V, V,
                                              excluded, n_excluded);
}

/* ----------------------------------------------------------------------- */
/* top-k                                                                   */
/* ----------------------------------------------------------------------- */

/*
 * [PR49] "Change": the k largest logits of each row with their token ids.
 * Definition used: sort all ids by value descending with a stable sort (ties
 * keep the lower id, the [Ch21] 21.3 convention), take the first k.
 * A nonfinite row gives ids 0xFFFFFFFF and values NaN.
 */
void orc_topk(const float *logits, uint32_t rows, uint32_t V, uint32_t k,
              float *out_vals, uint32_t *out_ids)
{
    double *key = (double *)malloc((size_t)V * sizeof(double));
    for (uint32_t r = 0; r < rows; ++r) {
        const float *x = logits + (size_t)r * V;
        float *ov = out_vals + (size_t)r * k;
        uint32_t *oi = out_ids + (size_t)r * k;
        if (!row_is_finite(x, V)) {
            for (uint32_t j = 0; j < k; ++j) {
                ov[j] = NAN;
                oi[j] = ORC_INVALID;
            }
            continue;
        }
        for (uint32_t i = 0; i < V; ++i)
            key[i] = (double)x[i];
        uint32_t *ids = sorted_ids_desc(key, V);
        for (uint32_t j = 0; j < k; ++j) {
            oi[j] = ids[j];
            ov[j] = x[ids[j]];
        }
        free(ids);
    }
    free(key);
}

/* ----------------------------------------------------------------------- */
/* filtered sampling                                                       */
/* ----------------------------------------------------------------------- */

/*
 * One row of filtered sampling. Steps, in order (the chain of [Ch21] 21.7:
 * top_n_sigma, top-k, typical_p, top-p; then min-p):
 *  1. z_i = x_i / T                     (T == 0: greedy, prob 1)
 *  2. top_n_sigma > 0: only ids with x_i >= max(x) - top_n_sigma * sigma
 *     remain, sigma the population standard deviation of the row's logits
 *     (a mask against the max; it does not depend on T)
 *     candidates C: the top_k of the remaining ids by the top-k definition
 *     above (top_k == 0: all of them), in (z desc, id asc) order
 *  3. w_i = exp(z_i - z_max), P_i = w_i / sum_C w       (softmax over C)
 *  3b. 0 < typical_p < 1 (locally typical sampling): H = -sum_C P ln P,
 *     score_i = |-ln P_i - H|; in (score asc, then C's order) keep the
 *     shortest prefix with cumulative P >= typical_p (at least one); the
 *     kept ids stay in C's order and P is renormalised over them
 *  4. top_p < 1: keep the shortest prefix of C with cumulative P >= top_p
 *  5. min_p > 0: keep survivors with P_i >= min_p * P_max
 *  6. Q_i = w_i / sum_survivors w ; draw by inverse CDF in the same order
 *     (full-row sampling, top_k == 0: in ascending id among the survivors)
 * temp_last != 0: steps 3-5 use T = 1 probabilities (filter on the
 * untempered distribution) and step 6 uses the tempered weights.
 * *margin = distance of the nearest decision to its threshold: |u - C_i|,
 * |cum_i - top_p|, |P_i / P_max - min_p|, |cum - typical_p| and the score gap
 * at the typical cut, and |x - (max - n sigma)| / max(|max - n sigma|, 1).
 */
static uint32_t sample_row(const float *x, uint32_t V, double T,
                           uint32_t top_k, double top_p, double min_p,
                           int temp_last, double top_n_sigma,
                           double typical_p, float u_f, double *prob,
                           double *margin)
{
    *margin = INFINITY;
    if (!row_is_finite(x, V) || !uniform_is_valid(u_f)) {
        *prob = NAN;
        return ORC_INVALID;
    }
    if (T == 0.0) {
        *prob = 1.0;
        return orc_argmax_row(x, V);
    }
    double u = (double)u_f;

    /* 1-2. tempered scores and the candidate set, in (z desc, id asc) */
    double *z = (double *)malloc((size_t)V * sizeof(double));
    for (uint32_t i = 0; i < V; ++i)
        z[i] = (double)x[i] / T;
    uint32_t *order = sorted_ids_desc(z, V);
    uint32_t nc = (top_k == 0 || top_k > V) ? V : top_k;

    /* 2. top-n-sigma: the ids at or above max - n sigma are a prefix of the
     *    order (z = x / T orders like x) */
    if (top_n_sigma > 0.0) {
        double mean = 0.0;
        for (uint32_t i = 0; i < V; ++i)
            mean += (double)x[i];
        mean /= (double)V;
        double var = 0.0;
        for (uint32_t i = 0; i < V; ++i)
            var += ((double)x[i] - mean) * ((double)x[i] - mean);
        double sigma = sqrt(var / (double)V);
        double thr = (double)x[order[0]] - top_n_sigma * sigma;
        double scale = fabs(thr) > 1.0 ? fabs(thr) : 1.0;
        uint32_t m = 0;
        while (m < V && (double)x[order[m]] >= thr)
            ++m;
        if (m > 0) {
            double d = fabs((double)x[order[m - 1]] - thr) / scale;
            if (d < *margin)
                *margin = d;
        }
        if (m < V) {
            double d = fabs((double)x[order[m]] - thr) / scale;
            if (d < *margin)
                *margin = d;
        }
        if (m < nc)
            nc = m;
    }

    /* 3. softmax over the candidates (filter distribution and draw weights) */
    double Tf = temp_last ? 1.0 : T;
    double *wf = (double *)malloc((size_t)nc * sizeof(double)); /* filter */
    double *wd = (double *)malloc((size_t)nc * sizeof(double)); /* draw */
    double zmax_f = (double)x[order[0]] / Tf, zmax_d = z[order[0]];
    double Sf = 0.0;
    for (uint32_t j = 0; j < nc; ++j) {
        wf[j] = exp((double)x[order[j]] / Tf - zmax_f);
        wd[j] = exp(z[order[j]] - zmax_d);
        Sf += wf[j];
    }

    /* 3b. locally typical: keep the most typical ids up to typical_p mass */
    if (typical_p > 0.0 && typical_p < 1.0 && nc > 1) {
        double H = 0.0;
        for (uint32_t j = 0; j < nc; ++j) {
            double P = wf[j] / Sf;
            if (P > 0.0)
                H -= P * log(P);
        }
        double *score = (double *)malloc((size_t)nc * sizeof(double));
        for (uint32_t j = 0; j < nc; ++j) {
            double P = wf[j] / Sf;
            score[j] = P > 0.0 ? fabs(-log(P) - H) : INFINITY;
        }
        /* (score asc, position asc): a stable sort of the positions by -score */
        double *neg = (double *)malloc((size_t)nc * sizeof(double));
        for (uint32_t j = 0; j < nc; ++j)
            neg[j] = -score[j];
        uint32_t *tord = sorted_ids_desc(neg, nc);
        char *keep = (char *)calloc(nc, 1);
        double cum = 0.0;
        for (uint32_t t = 0; t < nc; ++t) {
            uint32_t j = tord[t];
            keep[j] = 1;
            cum += wf[j] / Sf;
            double d = fabs(cum - typical_p);
            if (d < *margin)
                *margin = d;
            if (cum >= typical_p) {
                if (t + 1 < nc) {
                    double g = fabs(score[tord[t + 1]] - score[j]);
                    double sc = score[j] > 1.0 ? score[j] : 1.0;
                    if (g / sc < *margin)
                        *margin = g / sc;
                }
                break;
            }
        }
        uint32_t n2 = 0;
        double S2 = 0.0;
        for (uint32_t j = 0; j < nc; ++j) {
            if (!keep[j])
                continue;
            order[n2] = order[j];
            wf[n2] = wf[j];
            wd[n2] = wd[j];
            S2 += wf[n2];
            ++n2;
        }
        nc = n2;
        Sf = S2;
        free(keep);
        free(tord);
        free(neg);
        free(score);
    }

    /* 4. top-p: shortest prefix with cumulative mass >= top_p */
    uint32_t ns = nc;
    if (top_p < 1.0) {
        double cum = 0.0;
        for (uint32_t j = 0; j < nc; ++j) {
            cum += wf[j] / Sf;
            double d = fabs(cum - top_p);
            if (d < *margin)
                *margin = d;
            if (cum >= top_p) {
                ns = j + 1;
                break;
            }
        }
    }

    /* 5. min-p against the most probable survivor (always kept) */
    if (min_p > 0.0) {
        double pmax = wf[0] / Sf;
        uint32_t keep = 1;
        for (uint32_t j = 1; j < ns; ++j) {
            double ratio = (wf[j] / Sf) / pmax;
            double d = fabs(ratio - min_p);
            if (d < *margin)
                *margin = d;
            if (ratio >= min_p)
                keep = j + 1; /* P is non-increasing: survivors form a prefix */
        }
        ns = keep;
    }

    /* 6. renormalise over the survivors and draw: in the survivors' order,
     *    or, for full-row sampling (top_k == 0), in ascending id. The pages
     *    fix no CDF order; the distribution is the same either way, and
     *    ascending id needs no sort of V (the residual and bonus draws of
     *    speculative acceptance take the same reading). */
    double Sd = 0.0;
    for (uint32_t j = 0; j < ns; ++j)
        Sd += wd[j];
    double m_draw;
    uint32_t id;
    if (top_k == 0) {
        /* survivors by ascending id: (id << 32 | position), sorted */
        uint64_t *by_id = (uint64_t *)malloc((size_t)ns * sizeof(uint64_t));
        for (uint32_t j = 0; j < ns; ++j)
            by_id[j] = ((uint64_t)order[j] << 32) | j;
        qsort(by_id, ns, sizeof(uint64_t), cmp_u64);
        double *wa = (double *)malloc((size_t)ns * sizeof(double));
        for (uint32_t i = 0; i < ns; ++i)
            wa[i] = wd[(uint32_t)by_id[i]];
        uint32_t pick = inverse_cdf(wa, ns, u, &m_draw);
        id = (uint32_t)(by_id[pick] >> 32);
        *prob = wa[pick] / Sd;
        free(wa);
        free(by_id);
    } else {
        uint32_t pick = inverse_cdf(wd, ns, u, &m_draw);
        id = order[pick];
        *prob = wd[pick] / Sd;
    }
    if (m_draw < *margin)
        *margin = m_draw;

    free(wd);
    free(wf);
    free(order);
    free(z);
    return id;
}

int orc_sample_ex(const float *logits, uint32_t rows, uint32_t V,
                  double temperature, uint32_t top_k, double top_p,
                  double min_p, int temp_last, double top_n_sigma,
                  double typical_p, const float *uniforms, uint32_t *out_ids,
                  double *out_probs, double *out_margin)
{
    for (uint32_t r = 0; r < rows; ++r) {
        double m;
        out_ids[r] = sample_row(logits + (size_t)r * V, V, temperature,
                                top_k, top_p, min_p, temp_last, top_n_sigma,
                                typical_p, uniforms[r], &out_probs[r], &m);
        if (out_margin)
            out_margin[r] = m;
    }
    return 0;
}

int orc_sample(const float *logits, uint32_t rows, uint32_t V,
               double temperature, uint32_t top_k, double top_p,
               double min_p, int temp_last, const float *uniforms,
               uint32_t *out_ids, double *out_probs, double *out_margin)
{
    return orc_sample_ex(logits, rows, V, temperature, top_k, top_p, min_p,
                         temp_last, 0.0, 1.0, uniforms, out_ids, out_probs,
                         out_margin);
}

/* ----------------------------------------------------------------------- */
/* speculative acceptance                                                  */
/* ----------------------------------------------------------------------- */

/*
 * One sequence. target: (K+1) rows of V, draft: K rows of V (unused by the
 * argmax rule), tokens: K draft tokens. Writes accepted count n and
 * emitted[0..K]: t_0 .. t_{n-1}, then the drawn token, then 0xFFFFFFFF.
 *
 * mode 0, modified rejection sampling ([Spec], [Ch21] 21.9):
 *   p_j = softmax(target_j / T), q_j = softmax(draft_j / T);
 *   position j accepts iff u_acc[j] * q_j(t_j) <= p_j(t_j);
 *   first rejection j*: draw with u_fin from normalize(max(p - q, 0)),
 *   falling back to p when the residual total is <= 0;
 *   all accepted: draw with u_fin from p_K (the last target row).
 * mode 1, argmax-against-argmax ([Spec]): a_j = argmax(target_j);
 *   n = first j with t_j != a_j (else K); emit a_n.
 * T == 0 selects mode 1 ([Spec] "RNG dependency": greedy draws nothing).
 */
static void spec_sequence(const float *target, const float *draft,
                          const uint32_t *tokens, uint32_t K, uint32_t V,
                          double T, int mode, const float *u_acc, float u_fin,
                          uint32_t *accepted, uint32_t *emitted,
                          double *margin_accept, double *margin_draw)
{
    *margin_accept = INFINITY;
    *margin_draw = INFINITY;
    for (uint32_t j = 0; j <= K; ++j)
        emitted[j] = ORC_INVALID;
    *accepted = ORC_INVALID;
    if (T == 0.0)
        mode = 1;

    /* fail closed: any nonfinite row, out-of-range token or bad uniform */
    for (uint32_t j = 0; j <= K; ++j)
        if (!row_is_finite(target + (size_t)j * V, V))
            return;
    for (uint32_t j = 0; j < K; ++j)
        if (tokens[j] >= V)
            return;
    if (mode == 0) {
        for (uint32_t j = 0; j < K; ++j)
            if (!row_is_finite(draft + (size_t)j * V, V) ||
                !uniform_is_valid(u_acc[j]))
                return;
        if (!uniform_is_valid(u_fin))
            return;
    }

    if (mode == 1) {
        uint32_t n = 0;
        uint32_t a = 0;
        for (;;) {
            a = orc_argmax_row(target + (size_t)n * V, V);
            if (n == K || tokens[n] != a)
                break;
            ++n;
        }
        for (uint32_t j = 0; j < n; ++j)
            emitted[j] = tokens[j];
        emitted[n] = a;
        *accepted = n;
        return;
    }

    double *p = (double *)malloc((size_t)V * sizeof(double));
    double *q = (double *)malloc((size_t)V * sizeof(double));
    double *r = (double *)malloc((size_t)V * sizeof(double));
    uint32_t n = 0;
    int rejected = 0;
    for (; n < K; ++n) {
        softmax_row(target + (size_t)n * V, V, T, p);
        softmax_row(draft + (size_t)n * V, V, T, q);
        double pt = p[tokens[n]], qt = q[tokens[n]];
        double lhs = (double)u_acc[n] * qt;
        double scale = pt > qt ? pt : qt;
        if (scale > 0.0) {
            double d = fabs(lhs - pt) / scale;
            if (d < *margin_accept)
                *margin_accept = d;
        }
        if (lhs <= pt)
            continue;
        rejected = 1;
        break;
    }
    uint32_t drawn;
    if (rejected) {
        /* residual max(p - q, 0); p again if its total is <= 0 */
        double total = 0.0;
        for (uint32_t i = 0; i < V; ++i) {
            double d = p[i] - q[i];
            r[i] = d > 0.0 ? d : 0.0;
            total += r[i];
        }
        if (!(total > 0.0))
            memcpy(r, p, (size_t)V * sizeof(double));
        drawn = inverse_cdf(r, V, (double)u_fin, margin_draw);
    } else {
        softmax_row(target + (size_t)K * V, V, T, p);
        drawn = inverse_cdf(p, V, (double)u_fin, margin_draw);
    }
    for (uint32_t j = 0; j < n; ++j)
        emitted[j] = tokens[j];
    emitted[n] = drawn;
    *accepted = n;
    free(r);
    free(q);
    free(p);
}

int orc_spec_accept(const float *target, const float *draft,
                    const uint32_t *draft_tokens, uint32_t S, uint32_t K,
                    uint32_t V, double temperature, int mode,
                    const float *u_acc, const float *u_fin,
                    uint32_t *accepted, uint32_t *emitted,
                    double *margin_accept, double *margin_draw)
{
    for (uint32_t s = 0; s < S; ++s) {
        double ma, md;
        spec_sequence(target + (size_t)s * (K + 1) * V,
                      draft ? draft + (size_t)s * K * V : NULL,
                      draft_tokens + (size_t)s * K, K, V, temperature, mode,
                      u_acc ? u_acc + (size_t)s * K : NULL,
                      u_fin ? u_fin[s] : 0.0f, &accepted[s],
                      emitted + (size_t)s * (K + 1), &ma, &md);
        if (margin_accept)
            margin_accept[s] = ma;
        if (margin_draw)
            margin_draw[s] = md;
    }
    return 0;
}

/*
 * [Spec] "Sampler-match (the default at temperature > 0)": position j draws a
 * fresh token from the target's sampler -- here the sampling chain of
 * sample_row with the caller's policy and uniform u[j] -- and accepts the
 * drafted token iff it equals that draw; the first mismatch emits the draw
 * and ends the chain; when all K drafts match, the draw at position K is the
 * bonus token. Every emitted token is a fresh draw from the target sampler.
 * Readings: one uniform per verified position, u[0..K]; the sequence fails
 * closed (every id 0xFFFFFFFF) on a nonfinite target row, a draft token >= V
 * or any of its K + 1 uniforms outside [0, 1); T == 0 is the greedy sampler.
 * *margin = the smallest sampling margin among the draws the chain used.
 */
static void spec_sampler_sequence(const float *target, const uint32_t *tokens,
                                  uint32_t K, uint32_t V, double T,
                                  uint32_t top_k, double top_p, double min_p,
                                  int temp_last, const float *u,
                                  uint32_t *accepted, uint32_t *emitted,
                                  double *margin)
{
    *margin = INFINITY;
    for (uint32_t j = 0; j <= K; ++j)
        emitted[j] = ORC_INVALID;
    *accepted = ORC_INVALID;
    for (uint32_t j = 0; j <= K; ++j)
        if (!row_is_finite(target + (size_t)j * V, V) ||
            !uniform_is_valid(u[j]))
            return;
    for (uint32_t j = 0; j < K; ++j)
        if (tokens[j] >= V)
            return;
    uint32_t n = 0, drawn = 0;
    for (;;) {
        double prob, m;
        drawn = sample_row(target + (size_t)n * V, V, T, top_k, top_p, min_p,
                           temp_last, 0.0, 1.0, u[n], &prob, &m);
        if (m < *margin)
            *margin = m;
        if (n == K || tokens[n] != drawn)
            break;
        ++n;
    }
    for (uint32_t j = 0; j < n; ++j)
        emitted[j] = tokens[j];
    emitted[n] = drawn;
    *accepted = n;
}

int orc_spec_sampler(const float *target, const uint32_t *draft_tokens,
                     uint32_t S, uint32_t K, uint32_t V, double temperature,
                     uint32_t top_k, double top_p, double min_p, int temp_last,
                     const float *u, uint32_t *accepted, uint32_t *emitted,
                     double *margin)
{
    for (uint32_t s = 0; s < S; ++s) {
        double m;
        spec_sampler_sequence(target + (size_t)s * (K + 1) * V,
                              draft_tokens + (size_t)s * K, K, V, temperature,
                              top_k, top_p, min_p, temp_last,
                              u + (size_t)s * (K + 1), &accepted[s],
                              emitted + (size_t)s * (K + 1), &m);
        if (margin)
            margin[s] = m;
    }
    return 0;
}

/*
 * [Spec] "Verifying the gain before trusting a throughput number": per
 * verified position, sum_x min(p(x), q(x)) -- the probability that modified
 * rejection sampling accepts -- and sum_x p(x) q(x) -- the probability that
 * sampler-match accepts -- with p = softmax(target_j / T) and
 * q = softmax(draft_j / T), T > 0 (reading: the tempered distributions the
 * rejection rule here uses, no filters). A position with a nonfinite target
 * or draft row gives NaN for both.
 */
void orc_spec_diagnostics(const float *target, const float *draft, uint32_t S,
                          uint32_t K, uint32_t V, double T, double *sum_min,
                          double *sum_prod)
{
    double *p = (double *)malloc((size_t)V * sizeof(double));
    double *q = (double *)malloc((size_t)V * sizeof(double));
    for (uint32_t s = 0; s < S; ++s) {
        for (uint32_t j = 0; j < K; ++j) {
            const float *t = target + ((size_t)s * (K + 1) + j) * V;
            const float *d = draft + ((size_t)s * K + j) * V;
            double *om = sum_min + (size_t)s * K + j;
            double *op = sum_prod + (size_t)s * K + j;
            if (!row_is_finite(t, V) || !row_is_finite(d, V)) {
                *om = NAN;
                *op = NAN;
                continue;
            }
            softmax_row(t, V, T, p);
            softmax_row(d, V, T, q);
            double a = 0.0, b = 0.0;
            for (uint32_t i = 0; i < V; ++i) {
                a += p[i] < q[i] ? p[i] : q[i];
                b += p[i] * q[i];
            }
            *om = a;
            *op = b;
        }
    }
    free(q);
    free(p);
}

/* Plain softmax of one row in double, exported for tests that need p and q. */
void orc_softmax_row(const float *x, uint32_t V, double T, double *p)
{
    softmax_row(x, V, T, p);
}
