/*
 * ssd_oracle.c -- the CPU oracle for the verify-and-recover step of
 * speculative decoding (SD) and Speculative Speculative Decoding (SSD).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously correct
 * statement of what the GPU path computes.  It shares no code, header, table
 * or constant with the CUDA library; only the tests, the package smoke check
 * and the benchmark's CPU-baseline leg load it.  The product path never calls
 * it and has no CPU fallback.
 *
 * Everything is scalar C in double precision, one batch row b at a time, one
 * logit row at a time, in index order, with sequential summation.  No
 * blocking, fusion or reordering.
 *
 * What it follows:
 *   - "tanishqkumar/ssd" summary page (thehardwarestore.ai), module notes:
 *     the sampler mixes greedy and stochastic sampling by temperature
 *     (temperature 0 = greedy argmax); forked recovery tokens are chosen by
 *     top-k over logits with masking for cache hits.
 *   - "SSD: drafting and verification on separate GPUs" (hysenlabs.com),
 *     section "What changes in SSD": the draft guesses several tokens, the
 *     target verifies them in one forward pass, and the method is exact (it
 *     does not change the output distribution).
 *   - speculative-sampling summary (sourcepulse.org project 1842340),
 *     "How It Works": accept correct tokens and re-generate from the point of
 *     divergence; "Highlighted Details": Google's and DeepMind's algorithms.
 *   - The published speculative-sampling rule those two algorithms share
 *     (Leviathan, Kalman & Matias 2023; Chen et al. 2023): accept x_i with
 *     probability min(1, p_i(x_i)/q_i(x_i)); on the first rejection at
 *     position n draw from norm(max(0, p_n - q_n)); after k accepts draw the
 *     bonus token from p_k.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   R1 the row's temperature T_b applies to target and draft rows alike;
 *   R2 acceptance is the strict compare u < p/q; q(x) == 0 accepts iff p(x)>0;
 *   R3 greedy (T == 0) acceptance is x_i == argmax Z[b,i] (lowest index wins);
 *   R4 inverse CDF: smallest j with C_j > u * C_{V-1}, C the sequential prefix
 *      sum; if rounding leaves none, the last j with w(j) > 0;
 *   R5 an all-zero residual falls back to p_n;
 *   R6 top-f orders by (logit descending, index ascending) over unmasked
 *      tokens; fewer than f candidates pads with (token -1, logit -inf);
 *   R7 sentinels: T < 0 or NaN -> accept_len -1; a draft token outside [0,V)
 *      -> accept_len -2; a NaN logit in any row read (or, for T > 0, a +inf
 *      logit or an all -inf row) -> accept_len -1.  Out tokens are then -1.
 *   R9 top-k / top-p filtered distributions (both the target's and the
 *      draft's, with the same K and top_p): order the tokens by (logit
 *      descending, index ascending); keep the first K; then keep the shortest
 *      prefix of those whose probability mass is >= top_p times their mass;
 *      renormalise over what is kept.  Acceptance, the residual and the bonus
 *      draw then use the filtered p and q; greedy rows are unchanged.
 *   R10 token-tree verification (the summary page's "tree decoding"; the
 *      rule is the multi-step speculative sampling of SpecInfer, Miao et
 *      al. 2024, for children drawn independently from the draft's q at
 *      their parent): per batch row a tree of N nodes, node 0 the root,
 *      parent[j] < j, children tried in increasing node index.  At the
 *      current node with target law r (initially p of that node) each
 *      child token x is accepted when u < r(x)/q(x) (R2 for q(x) == 0); an
 *      accepted child becomes the current node (r = its p); a rejection
 *      replaces r by norm(max(0, r - q)) (kept unchanged if that is all
 *      zero, as R5).  When the children are exhausted the final token is
 *      drawn from r by R4.  Greedy rows accept the first child whose token
 *      is the argmax of the current node's target row and end with that
 *      argmax.  All N target rows are read, and the draft rows of the
 *      nodes that have children (a leaf's q is never used), with R7's
 *      checks; parent[0] != -1, parent[j] outside [0, j) or a token outside
 *      [0, V) gives accept_len -2.
 *   R8 draft-side sampling: the drafter's token at T > 0 is the Gumbel-max
 *      draw argmax_v (z_v / T + G_v), G_v = -ln(-ln u_v), which is exactly a
 *      draw from softmax(z / T); u_v comes from the counter-based generator
 *      Philox4x32-10 (Salmon, Moraes, Dror & Shaw 2011) so that both sides
 *      can regenerate it; ties go to the lowest index; T == 0 takes the
 *      argmax; invalid T or rows give -1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* Status codes of the oracle's own entry points. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* One logit as a double.  bf16 is the upper 16 bits of an IEEE binary32,
 * so widening is a 16-bit shift; float to double is exact. */
static double logit_at(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_BF16) {
        uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

/* Copy one row into a double buffer. */
static void load_row(const void *base, int dtype, int64_t row_start, int64_t V,
                     double *out)
{
    for (int64_t v = 0; v < V; ++v)
        out[v] = logit_at(base, dtype, row_start + v);
}

/* Row validity (reading R7).  greedy rows only reject NaN. */
static int row_is_valid(const double *z, int64_t V, int greedy)
{
    int any_finite_or_neg = 0;
    for (int64_t v = 0; v < V; ++v) {
        if (isnan(z[v]))
            return 0;
        if (!greedy && isinf(z[v]) && z[v] > 0)
            return 0;
        if (!(isinf(z[v]) && z[v] < 0))
            any_finite_or_neg = 1;
    }
    if (!greedy && !any_finite_or_neg)
        return 0; /* all -inf: softmax undefined */
    return 1;
}

/* Argmax with the lowest index winning ties (reading R3). */
static int64_t argmax_lowest(const double *z, int64_t V)
{
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
        if (z[v] > z[best])
            best = v;
    return best;
}

/* Temperature softmax of one row (summary page: temperature-controlled
 * sampler).  m = max z, S = sum_v exp((z_v - m)/T), p_v = exp((z_v - m)/T)/S.
 * p may be NULL.  Requires T > 0 and a valid row. */
static void softmax_temp(const double *z, int64_t V, double T, double *p,
                         double *m_out, double *S_out)
{
    double m = z[0];
    for (int64_t v = 1; v < V; ++v)
        if (z[v] > m)
            m = z[v];
    double S = 0.0;
    for (int64_t v = 0; v < V; ++v)
        S += exp((z[v] - m) / T);
    if (p)
        for (int64_t v = 0; v < V; ++v)
            p[v] = exp((z[v] - m) / T) / S;
    *m_out = m;
    *S_out = S;
}

/* Inverse CDF over nonnegative weights w (reading R4). */
static int64_t inverse_cdf(const double *w, int64_t V, double u)
{
    double total = 0.0;
    for (int64_t v = 0; v < V; ++v)
        total += w[v];
    double target = u * total;
    double C = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        C += w[v];
        if (C > target)
            return v;
    }
    for (int64_t v = V - 1; v >= 0; --v)
        if (w[v] > 0.0)
            return v;
    return V - 1;
}

/*
 * oracle_softmax_temp: per row m, S, argmax and (optionally) p.
 * rows x V logits, contiguous.  T[r] == 0 gives the greedy distribution: a
 * one-hot at the argmax, S = 1.  T < 0 or NaN, or an invalid row (R7), gives
 * m = S = NaN, argmax = -1 and p = NaN.
 */
int oracle_softmax_temp(const void *logits, int dtype, int rows, int64_t V,
                        const float *T, double *probs, double *row_max,
                        double *row_sum, int32_t *row_argmax)
{
    if (!logits || !T || rows < 0 || V < 1)
        return ORACLE_BAD_ARG;
    double *z = (double *)malloc((size_t)V * sizeof(double));
    if (!z)
        return ORACLE_NO_MEMORY;
    for (int r = 0; r < rows; ++r) {
        double t = (double)T[r];
        load_row(logits, dtype, (int64_t)r * V, V, z);
        double *p = probs ? probs + (int64_t)r * V : NULL;
        int greedy = (t == 0.0);
        if (isnan(t) || t < 0.0 || !row_is_valid(z, V, greedy)) {
            row_max[r] = NAN;
            row_sum[r] = NAN;
            row_argmax[r] = -1;
            if (p)
                for (int64_t v = 0; v < V; ++v)
                    p[v] = NAN;
            continue;
        }
        int64_t a = argmax_lowest(z, V);
        row_argmax[r] = (int32_t)a;
        if (greedy) {
            row_max[r] = z[a];
            row_sum[r] = 1.0;
            if (p)
                for (int64_t v = 0; v < V; ++v)
                    p[v] = (v == a) ? 1.0 : 0.0;
        } else {
            softmax_temp(z, V, t, p, &row_max[r], &row_sum[r]);
        }
    }
    free(z);
    return ORACLE_OK;
}

/* One token in the order of readings R6 / R9. */
typedef struct {
    double z;
    int64_t v;
} ranked_t;

/* Logit descending, then index ascending (qsort comparator). */
static int rank_cmp(const void *a, const void *b)
{
    const ranked_t *x = (const ranked_t *)a, *y = (const ranked_t *)b;
    if (x->z > y->z)
        return -1;
    if (x->z < y->z)
        return 1;
    return (x->v < y->v) ? -1 : (x->v > y->v);
}

/* Top-k / top-p filter of one row's probabilities p (reading R9), in
 * place: all V tokens ordered by (z descending, index ascending) -- a sort
 * serves as the step -- then the first K of them, then the shortest prefix
 * of those holding >= top_p of their mass, renormalised; every other token
 * gets 0.  `ord` is scratch for V entries and `taken` for V flags. */
static void filter_topk_topp(const double *z, double *p, int64_t V, int K, double top_p,
                             ranked_t *ord, char *taken)
{
    if (V < 1)
        return;
    for (int64_t v = 0; v < V; ++v) {
        ord[v].z = z[v];
        ord[v].v = v;
    }
    qsort(ord, (size_t)V, sizeof(ranked_t), rank_cmp);
    const int64_t n = (int64_t)K < V ? (int64_t)K : V;
    double mass = 0.0;
    for (int64_t j = 0; j < n; ++j)
        mass += p[ord[j].v];
    int64_t keep = n;
    if (top_p < 1.0) {
        double c = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            c += p[ord[j].v];
            if (c >= top_p * mass) {
                keep = j + 1;
                break;
            }
        }
    }
    double kept = 0.0;
    for (int64_t j = 0; j < keep; ++j)
        kept += p[ord[j].v];
    for (int64_t v = 0; v < V; ++v)
        taken[v] = 0;
    for (int64_t j = 0; j < keep; ++j)
        taken[ord[j].v] = 1;
    for (int64_t v = 0; v < V; ++v)
        p[v] = taken[v] ? p[v] / kept : 0.0;
}

/*
 * verify_core / oracle_verify_recover_f64: one verify-and-recover step for B batch rows,
 * with the uniforms in double precision (the core; the binary32 entry point
 * below widens its uniforms and calls this).
 *
 * Z: target logits, row (b, i) starts at b*z_bstride + i*V, i in 0..k.
 * D: draft logits,  row (b, i) starts at b*d_bstride + i*V, i in 0..k-1.
 * x[b*k + i]: draft tokens; T[b]: temperature; u_acc[b*k + i], u_smp[b]:
 * the supplied uniforms.  Outputs: accept_len[b] (n, or a sentinel),
 * p_at_x / q_at_x [b*k + i] (may be NULL), out_tok[b*(k+1) + j]: the n
 * accepted draft tokens, then the recovery/bonus token, then -1.
 *
 * Step order per b follows the speculative-sampling rule: acceptance per
 * position, first rejection n, then one draw from the residual (n < k) or
 * from the target's last row (n == k).
 */
/* The core; K == 0 filters nothing (R9 otherwise, top_p may be NULL). */
static int verify_core(const void *Z, int64_t z_bstride, const void *D, int64_t d_bstride,
                       int dtype, int B, int k, int64_t V, const int32_t *x, const float *T,
                       int K, const float *top_p, const double *u_acc, const double *u_smp,
                       int32_t *accept_len, double *p_at_x, double *q_at_x, int32_t *out_tok)
{
    if (!Z || !D || !x || !T || !u_acc || !u_smp || !accept_len || !out_tok ||
        B < 0 || k < 1 || V < 1 || K < 0)
        return ORACLE_BAD_ARG;
    double *zrow = (double *)malloc((size_t)V * sizeof(double));
    double *drow = (double *)malloc((size_t)V * sizeof(double));
    double *p = (double *)malloc((size_t)V * sizeof(double));
    double *q = (double *)malloc((size_t)V * sizeof(double));
    double *w = (double *)malloc((size_t)V * sizeof(double));
    int *accepted = (int *)malloc((size_t)k * sizeof(int));
    ranked_t *ord = (ranked_t *)malloc((size_t)(K > 0 ? V : 1) * sizeof(ranked_t));
    char *taken = (char *)malloc((size_t)V);
    if (!zrow || !drow || !p || !q || !w || !accepted || !ord || !taken) {
        free(zrow); free(drow); free(p); free(q); free(w); free(accepted); free(ord);
        free(taken);
        return ORACLE_NO_MEMORY;
    }

    for (int b = 0; b < B; ++b) {
        double t = (double)T[b];
        const double pb = top_p ? (double)top_p[b] : 1.0;
        int32_t *out = out_tok + (int64_t)b * (k + 1);
        for (int j = 0; j <= k; ++j)
            out[j] = -1;
        if (p_at_x)
            for (int i = 0; i < k; ++i) {
                p_at_x[(int64_t)b * k + i] = NAN;
                q_at_x[(int64_t)b * k + i] = NAN;
            }

        /* R7 sentinels, in this order: temperature, token range, rows. */
        if (isnan(t) || t < 0.0) {
            accept_len[b] = -1;
            continue;
        }
        int bad_token = 0;
        for (int i = 0; i < k; ++i)
            if (x[(int64_t)b * k + i] < 0 || x[(int64_t)b * k + i] >= V)
                bad_token = 1;
        if (bad_token) {
            accept_len[b] = -2;
            continue;
        }
        int greedy = (t == 0.0);
        int rows_ok = 1;
        for (int i = 0; i <= k && rows_ok; ++i) {
            load_row(Z, dtype, (int64_t)b * z_bstride + (int64_t)i * V, V, zrow);
            rows_ok = row_is_valid(zrow, V, greedy);
        }
        for (int i = 0; i < k && rows_ok; ++i) {
            load_row(D, dtype, (int64_t)b * d_bstride + (int64_t)i * V, V, drow);
            rows_ok = row_is_valid(drow, V, greedy);
        }
        if (!rows_ok) {
            accept_len[b] = -1;
            continue;
        }

        /* Acceptance at each draft position. */
        for (int i = 0; i < k; ++i) {
            int32_t xi = x[(int64_t)b * k + i];
            load_row(Z, dtype, (int64_t)b * z_bstride + (int64_t)i * V, V, zrow);
            load_row(D, dtype, (int64_t)b * d_bstride + (int64_t)i * V, V, drow);
            double pi, qi;
            if (greedy) {
                /* R3: the greedy distribution is a one-hot at the argmax. */
                pi = (argmax_lowest(zrow, V) == xi) ? 1.0 : 0.0;
                qi = (argmax_lowest(drow, V) == xi) ? 1.0 : 0.0;
                accepted[i] = (pi == 1.0);
            } else {
                double m, S;
                softmax_temp(zrow, V, t, p, &m, &S);
                softmax_temp(drow, V, t, q, &m, &S);
                if (K > 0) {
                    filter_topk_topp(zrow, p, V, K, pb, ord, taken);
                    filter_topk_topp(drow, q, V, K, pb, ord, taken);
                }
                pi = p[xi];
                qi = q[xi];
                /* R2: accept with probability min(1, p/q) against u. */
                if (qi == 0.0)
                    accepted[i] = (pi > 0.0);
                else
                    accepted[i] = (u_acc[(int64_t)b * k + i] < pi / qi);
            }
            if (p_at_x) {
                p_at_x[(int64_t)b * k + i] = pi;
                q_at_x[(int64_t)b * k + i] = qi;
            }
        }

        /* First rejection: the point of divergence. */
        int n = k;
        for (int i = 0; i < k; ++i)
            if (!accepted[i]) {
                n = i;
                break;
            }

        /* Recovery (n < k) or bonus (n == k) token. */
        int64_t tok;
        load_row(Z, dtype, (int64_t)b * z_bstride + (int64_t)n * V, V, zrow);
        if (greedy) {
            tok = argmax_lowest(zrow, V);
        } else {
            double m, S;
            softmax_temp(zrow, V, t, p, &m, &S);
            if (K > 0)
                filter_topk_topp(zrow, p, V, K, pb, ord, taken);
            if (n < k) {
                load_row(D, dtype, (int64_t)b * d_bstride + (int64_t)n * V, V, drow);
                softmax_temp(drow, V, t, q, &m, &S);
                if (K > 0)
                    filter_topk_topp(drow, q, V, K, pb, ord, taken);
                double total = 0.0;
                for (int64_t v = 0; v < V; ++v) {
                    double d = p[v] - q[v];
                    w[v] = d > 0.0 ? d : 0.0;
                    total += w[v];
                }
                if (total == 0.0) /* R5 */
                    for (int64_t v = 0; v < V; ++v)
                        w[v] = p[v];
            } else {
                for (int64_t v = 0; v < V; ++v)
                    w[v] = p[v];
            }
            tok = inverse_cdf(w, V, u_smp[b]);
        }

        accept_len[b] = n;
        for (int i = 0; i < n; ++i)
            out[i] = x[(int64_t)b * k + i];
        out[n] = (int32_t)tok;
    }

    free(zrow); free(drow); free(p); free(q); free(w); free(accepted); free(ord); free(taken);
    return ORACLE_OK;
}

int oracle_verify_recover_f64(const void *Z, int64_t z_bstride, const void *D,
                              int64_t d_bstride, int dtype, int B, int k,
                              int64_t V, const int32_t *x, const float *T,
                              const double *u_acc, const double *u_smp,
                              int32_t *accept_len, double *p_at_x,
                              double *q_at_x, int32_t *out_tok)
{
    return verify_core(Z, z_bstride, D, d_bstride, dtype, B, k, V, x, T, 0, NULL, u_acc,
                       u_smp, accept_len, p_at_x, q_at_x, out_tok);
}

/* The step over top-k / top-p filtered distributions (R9), binary32 or
 * double uniforms (f64 != 0). */
int oracle_verify_recover_filtered(const void *Z, int64_t z_bstride, const void *D,
                                   int64_t d_bstride, int dtype, int B, int k, int64_t V,
                                   const int32_t *x, const float *T, int K, const float *top_p,
                                   const void *u_acc, const void *u_smp, int f64,
                                   int32_t *accept_len, double *p_at_x, double *q_at_x,
                                   int32_t *out_tok)
{
    if (K < 1 || !u_acc || !u_smp)
        return ORACLE_BAD_ARG;
    if (f64)
        return verify_core(Z, z_bstride, D, d_bstride, dtype, B, k, V, x, T, K, top_p,
                           (const double *)u_acc, (const double *)u_smp, accept_len, p_at_x,
                           q_at_x, out_tok);
    double *ua = (double *)malloc((size_t)(B > 0 ? B : 1) * (size_t)k * sizeof(double));
    double *us = (double *)malloc((size_t)(B > 0 ? B : 1) * sizeof(double));
    if (!ua || !us) {
        free(ua); free(us);
        return ORACLE_NO_MEMORY;
    }
    for (int64_t j = 0; j < (int64_t)B * k; ++j)
        ua[j] = (double)((const float *)u_acc)[j];
    for (int b = 0; b < B; ++b)
        us[b] = (double)((const float *)u_smp)[b];
    int rc = verify_core(Z, z_bstride, D, d_bstride, dtype, B, k, V, x, T, K, top_p, ua, us,
                         accept_len, p_at_x, q_at_x, out_tok);
    free(ua); free(us);
    return rc;
}

/* The same step with binary32 uniforms, as the GPU library takes them. */
int oracle_verify_recover(const void *Z, int64_t z_bstride, const void *D,
                          int64_t d_bstride, int dtype, int B, int k, int64_t V,
                          const int32_t *x, const float *T, const float *u_acc,
                          const float *u_smp, int32_t *accept_len,
                          double *p_at_x, double *q_at_x, int32_t *out_tok)
{
    if (!u_acc || !u_smp || B < 0 || k < 1)
        return ORACLE_BAD_ARG;
    double *ua = (double *)malloc(((size_t)B * k + 1) * sizeof(double));
    double *us = (double *)malloc(((size_t)B + 1) * sizeof(double));
    if (!ua || !us) {
        free(ua); free(us);
        return ORACLE_NO_MEMORY;
    }
    for (int64_t i = 0; i < (int64_t)B * k; ++i)
        ua[i] = (double)u_acc[i];
    for (int b = 0; b < B; ++b)
        us[b] = (double)u_smp[b];
    int rc = oracle_verify_recover_f64(Z, z_bstride, D, d_bstride, dtype, B, k,
                                       V, x, T, ua, us, accept_len, p_at_x,
                                       q_at_x, out_tok);
    free(ua);
    free(us);
    return rc;
}

/*
 * oracle_forked_topf: forked recovery tokens (summary page: top-k over logits
 * with masking for cache hits).  For every (b, j), j in 0..P-1, the f largest
 * logits of row L[b*l_bstride + j*V ...] whose token is not listed in
 * mask[(b*P + j)*M + 0..M-1] (entries outside [0,V) list nothing).  Order R6.
 * A row holding a NaN gives tokens -1 and logits NaN.
 *
 * Plain method: mark the masked tokens, then f times pick the best unpicked
 * candidate by a full scan.
 */
int oracle_forked_topf(const void *L, int64_t l_bstride, int dtype, int B,
                       int P, int64_t V, int f, const int32_t *mask, int M,
                       int32_t *fork_tok, double *fork_logit)
{
    if (!L || !fork_tok || !fork_logit || B < 0 || P < 1 || V < 1 || f < 1 ||
        M < 0 || (M > 0 && !mask))
        return ORACLE_BAD_ARG;
    double *z = (double *)malloc((size_t)V * sizeof(double));
    char *taken = (char *)malloc((size_t)V);
    if (!z || !taken) {
        free(z); free(taken);
        return ORACLE_NO_MEMORY;
    }
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < P; ++j) {
            int64_t orow = ((int64_t)b * P + j) * f;
            load_row(L, dtype, (int64_t)b * l_bstride + (int64_t)j * V, V, z);
            int has_nan = 0;
            for (int64_t v = 0; v < V; ++v)
                if (isnan(z[v]))
                    has_nan = 1;
            if (has_nan) {
                for (int r = 0; r < f; ++r) {
                    fork_tok[orow + r] = -1;
                    fork_logit[orow + r] = NAN;
                }
                continue;
            }
            memset(taken, 0, (size_t)V);
            for (int mi = 0; mi < M; ++mi) {
                int32_t t = mask[((int64_t)b * P + j) * M + mi];
                if (t >= 0 && t < V)
                    taken[t] = 1;
            }
            for (int r = 0; r < f; ++r) {
                int64_t best = -1;
                for (int64_t v = 0; v < V; ++v) {
                    if (taken[v])
                        continue;
                    if (best < 0 || z[v] > z[best])
                        best = v;
                }
                if (best < 0) {
                    fork_tok[orow + r] = -1;
                    fork_logit[orow + r] = -INFINITY;
                } else {
                    taken[best] = 1;
                    fork_tok[orow + r] = (int32_t)best;
                    fork_logit[orow + r] = z[best];
                }
            }
        }
    }
    free(z);
    free(taken);
    return ORACLE_OK;
}


/*
 * oracle_verify_tree_f64: token-tree verification (reading R10) for B batch rows
 * of N nodes each.
 *
 * Z, D: target and draft logits, row (b, j) of node j at b*bstride + j*V.
 * parent[b*N + j], tok[b*N + j]: the tree (entry 0 of tok unused).
 * u_acc[b*N + j]: the uniform of node j's acceptance test (entry 0 unused);
 * u_smp[b]: the final draw (double here; oracle_verify_tree below takes
 * binary32 uniforms).  Outputs: accept_len[b] (accepted nodes, or a
 * sentinel), out_tok[b*N + i]: the accepted tokens in path order, then the
 * final token, then -1; out_node[b*N + i] (may be NULL): the accepted node
 * ids, then -1.
 */
int oracle_verify_tree_f64(const void *Z, int64_t z_bstride, const void *D,
                           int64_t d_bstride, int dtype, int B, int N, int64_t V,
                           const int32_t *parent, const int32_t *tok, const float *T,
                           const double *u_acc, const double *u_smp, int32_t *accept_len,
                           int32_t *out_tok, int32_t *out_node)
{
    if (!Z || !D || !parent || !tok || !T || !u_acc || !u_smp || !accept_len || !out_tok ||
        B < 0 || N < 1 || V < 1)
        return ORACLE_BAD_ARG;
    double *zrow = (double *)malloc((size_t)V * sizeof(double));
    double *r = (double *)malloc((size_t)V * sizeof(double));
    double *q = (double *)malloc((size_t)V * sizeof(double));
    double *w = (double *)malloc((size_t)V * sizeof(double));
    if (!zrow || !r || !q || !w) {
        free(zrow); free(r); free(q); free(w);
        return ORACLE_NO_MEMORY;
    }
    for (int b = 0; b < B; ++b) {
        const int32_t *par = parent + (int64_t)b * N;
        const int32_t *tk = tok + (int64_t)b * N;
        int32_t *out = out_tok + (int64_t)b * N;
        int32_t *node = out_node ? out_node + (int64_t)b * N : NULL;
        for (int j = 0; j < N; ++j) {
            out[j] = -1;
            if (node)
                node[j] = -1;
        }
        double t = (double)T[b];
        if (isnan(t) || t < 0.0) {
            accept_len[b] = -1;
            continue;
        }
        int bad_tree = par[0] != -1;
        for (int j = 1; j < N; ++j)
            if (par[j] < 0 || par[j] >= j || tk[j] < 0 || tk[j] >= V)
                bad_tree = 1;
        if (bad_tree) {
            accept_len[b] = -2;
            continue;
        }
        int greedy = (t == 0.0);
        int rows_ok = 1;
        for (int j = 0; j < N && rows_ok; ++j) {
            load_row(Z, dtype, (int64_t)b * z_bstride + (int64_t)j * V, V, zrow);
            rows_ok = row_is_valid(zrow, V, greedy);
            int has_child = 0;
            for (int c = j + 1; c < N; ++c)
                if (par[c] == j)
                    has_child = 1;
            if (has_child && rows_ok) {
                load_row(D, dtype, (int64_t)b * d_bstride + (int64_t)j * V, V, zrow);
                rows_ok = row_is_valid(zrow, V, greedy);
            }
        }
        if (!rows_ok) {
            accept_len[b] = -1;
            continue;
        }

        int cur = 0, depth = 0;
        double m, S;
        load_row(Z, dtype, (int64_t)b * z_bstride, V, zrow);
        if (!greedy)
            softmax_temp(zrow, V, t, r, &m, &S); /* r = p of the root */
        for (;;) {
            /* zrow holds the current node's target row */
            int moved = 0;
            if (greedy) {
                int64_t a = argmax_lowest(zrow, V);
                for (int c = cur + 1; c < N; ++c)
                    if (par[c] == cur && tk[c] == a) {
                        moved = c;
                        break;
                    }
                if (!moved) {
                    out[depth] = (int32_t)a;
                    break;
                }
            } else {
                int have_q = 0;
                for (int c = cur + 1; c < N && !moved; ++c) {
                    if (par[c] != cur)
                        continue;
                    if (!have_q) {
                        load_row(D, dtype, (int64_t)b * d_bstride + (int64_t)cur * V, V, w);
                        softmax_temp(w, V, t, q, &m, &S);
                        have_q = 1;
                    }
                    const int32_t x = tk[c];
                    int acc;
                    if (q[x] == 0.0)
                        acc = r[x] > 0.0;
                    else
                        acc = u_acc[(int64_t)b * N + c] < r[x] / q[x];
                    if (acc) {
                        moved = c;
                    } else {
                        /* the residual: norm(max(0, r - q)), r kept if all zero */
                        double tot = 0.0;
                        for (int64_t v = 0; v < V; ++v) {
                            double d = r[v] - q[v];
                            w[v] = d > 0.0 ? d : 0.0;
                            tot += w[v];
                        }
                        if (tot > 0.0)
                            for (int64_t v = 0; v < V; ++v)
                                r[v] = w[v] / tot;
                    }
                }
                if (!moved) {
                    out[depth] = (int32_t)inverse_cdf(r, V, u_smp[b]);
                    break;
                }
            }
            out[depth] = tk[moved];
            if (node)
                node[depth] = moved;
            ++depth;
            cur = moved;
            load_row(Z, dtype, (int64_t)b * z_bstride + (int64_t)cur * V, V, zrow);
            if (!greedy)
                softmax_temp(zrow, V, t, r, &m, &S);
        }
        accept_len[b] = depth;
    }
    free(zrow); free(r); free(q); free(w);
    return ORACLE_OK;
}

/* The same with binary32 uniforms, as the GPU library takes them. */
int oracle_verify_tree(const void *Z, int64_t z_bstride, const void *D, int64_t d_bstride,
                       int dtype, int B, int N, int64_t V, const int32_t *parent,
                       const int32_t *tok, const float *T, const float *u_acc,
                       const float *u_smp, int32_t *accept_len, int32_t *out_tok,
                       int32_t *out_node)
{
    if (!u_acc || !u_smp || B < 0 || N < 1)
        return ORACLE_BAD_ARG;
    double *ua = (double *)malloc(((size_t)B * N + 1) * sizeof(double));
    double *us = (double *)malloc(((size_t)B + 1) * sizeof(double));
    if (!ua || !us) {
        free(ua); free(us);
        return ORACLE_NO_MEMORY;
    }
    for (int64_t i = 0; i < (int64_t)B * N; ++i)
        ua[i] = (double)u_acc[i];
    for (int b = 0; b < B; ++b)
        us[b] = (double)u_smp[b];
    int rc = oracle_verify_tree_f64(Z, z_bstride, D, d_bstride, dtype, B, N, V, parent, tok,
                                    T, ua, us, accept_len, out_tok, out_node);
    free(ua); free(us);
    return rc;
}

/* ------------------------------------------------------------------------
 * Draft-side sampling (reading R8).
 * ------------------------------------------------------------------------ */

/* Philox4x32-10, from its published definition (Salmon et al. 2011,
 * "Parallel random numbers: as easy as 1, 2, 3"): ten rounds of
 *   (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
 *                        lo(M0 c0))
 * with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key bumped by the Weyl
 * constants (0x9E3779B9, 0xBB67AE85) before every round but the first. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The uniform of element v of draft row i of batch row b: word v mod 4 of
 * Philox4x32-10 at counter (v / 4, i, b, offset), key (seed_lo, seed_hi),
 * mapped to u = (w >> 9 + 1/2) / 2^23 in (0, 1) -- 23 bits, so that u and
 * 1 - u are exact in binary32 as well as here.  Returns 1 - u. */
static double draft_one_minus_u(uint32_t seed_lo, uint32_t seed_hi, uint32_t offset, int b,
                                int i, int64_t v)
{
    uint32_t ctr[4] = {(uint32_t)(v >> 2), (uint32_t)i, (uint32_t)b, offset};
    uint32_t key[2] = {seed_lo, seed_hi};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    uint32_t w = out[v & 3] >> 9;
    return ((double)(8388607u - w) + 0.5) / 8388608.0;
}

/* x[b * x_bstride + (i - row0)] for draft rows i in [row0, row0 + rows) of
 * D [B][Pd][V] (batch stride d_bstride). */
int oracle_draft_sample(const void *D, int64_t d_bstride, int dtype, int B, int Pd, int64_t V,
                        int row0, int rows, const float *T, uint32_t seed_lo, uint32_t seed_hi,
                        uint32_t offset, int32_t *x, int64_t x_bstride)
{
    if (!D || !T || !x || B < 0 || Pd < 1 || V < 1 || row0 < 0 || rows < 0 ||
        row0 + rows > Pd)
        return ORACLE_BAD_ARG;
    double *z = (double *)malloc((size_t)V * sizeof(double));
    if (!z)
        return ORACLE_NO_MEMORY;
    for (int b = 0; b < B; ++b) {
        const double Tb = (double)T[b];
        const int t_bad = isnan(Tb) || Tb < 0.0;
        const int greedy = !(Tb > 0.0);
        for (int i = row0; i < row0 + rows; ++i) {
            int32_t *xo = x + (int64_t)b * x_bstride + (i - row0);
            load_row(D, dtype, (int64_t)b * d_bstride + (int64_t)i * V, V, z);
            if (t_bad || !row_is_valid(z, V, greedy)) {
                *xo = -1;
                continue;
            }
            if (greedy) {
                *xo = (int32_t)argmax_lowest(z, V);
                continue;
            }
            int64_t best = -1;
            double best_y = -INFINITY;
            for (int64_t v = 0; v < V; ++v) {
                if (z[v] == -INFINITY)
                    continue;
                /* E = -ln u = -log1p(-(1 - u)), G = -ln E */
                double e = -log1p(-draft_one_minus_u(seed_lo, seed_hi, offset, b, i, v));
                double y = z[v] / Tb - log(e);
                if (best < 0 || y > best_y) {
                    best = v;
                    best_y = y;
                }
            }
            *xo = (int32_t)best;
        }
    }
    free(z);
    return ORACLE_OK;
}
