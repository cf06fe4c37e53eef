/*
 * oracle.c -- float64 CPU oracle for row-wise softmax and softmax+TopK.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only tests/, __graft_entry__.smoke() and the cpu_baseline /
 * reference legs of bench.py use it.  It shares no code, header, table or
 * constant with the CUDA library; the two meet only at the seeded inputs.
 *
 * Every function is a plain statement of a definition from the source pages,
 * computed in IEEE double with the host libm `exp`:
 *
 *   softmax  : three-pass safe softmax  m = max_j x_j,  d = sum_j e^(x_j - m),
 *              y_i = e^(x_i - m) / d.
 *              ("Online normalizer calculation for softmax" notes, section 2,
 *              safe softmax; "5.2 CUDA Online Softmax", section 1.1;
 *              "CUDA operator optimization (3): Softmax", CPU implementation.)
 *              The online method reaches this same result in exact arithmetic
 *              (the notes' section 3.2 induction proof), so the definition is
 *              the oracle for every kernel.
 *   stats    : the (m, d) pair of a row by the same definition.
 *   online   : the single-pass recurrence m_j = max(m_{j-1}, x_j),
 *              d_j = d_{j-1} e^(m_{j-1} - m_j) + e^(x_j - m_j), element by
 *              element (notes, section 3.1; "5.2 CUDA Online Softmax", 2.1).
 *              Used only by the pin tests that check it against `stats`.
 *   combine  : the binary operator
 *              (m1,d1) (+) (m2,d2) = (max, d1 e^(m1-max) + d2 e^(m2-max))
 *              (notes, section 3.3; "Lesson 7: Online Softmax and associative
 *              state", section 2), with the identity element (-inf, 0) of
 *              Lesson 7, section 3.
 *   topk     : the K largest probabilities and their indices (notes,
 *              section 4, "Softmax and top-k fusion": select on the logits u,
 *              then v = e^(u - m_V) / d_V).  Selection is a full sort of the
 *              row by (x descending, index ascending); the pages leave ties
 *              open, and they go to the lower index.
 *   attention: softmax(scale Q K^T) V and L = m + ln d per query row, with
 *              an optional causal mask (see oracle_attention_f64).
 *
 * Conventions: exp(-inf) = 0 from libm, so a -inf entry contributes nothing to
 * d and gets probability +0.  A row whose entries are all -inf has m = -inf and
 * d = 0; its probabilities are the formula's 0/0 = NaN.  Inputs are assumed
 * free of NaN.
 *
 * Rows are independent; an OpenMP loop over rows (when compiled with
 * -fopenmp) changes no arithmetic inside a row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the row loops from now on (n >= 1); no effect on the arithmetic
 * of a row.  A build without OpenMP always runs one. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* (m, d) of one row by definition: first the maximum, then the shifted sum. */
static void row_stats(const double *x, int64_t n, double *m_out, double *d_out) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (x[j] > m) m = x[j];
    double d = 0.0;
    if (m != -INFINITY)
        for (int64_t j = 0; j < n; ++j)
            d += exp(x[j] - m);
    *m_out = m;
    *d_out = d;
}

void oracle_row_stats_f64(const double *x, double *m, double *d,
                          int64_t rows, int64_t cols) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        row_stats(x + r * cols, cols, &m[r], &d[r]);
}

/* Three-pass safe softmax, one row after another. */
void oracle_softmax_f64(const double *x, double *y, int64_t rows, int64_t cols) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * cols;
        double *yr = y + r * cols;
        double m, d;
        row_stats(xr, cols, &m, &d);
        for (int64_t j = 0; j < cols; ++j)
            yr[j] = exp(xr[j] - m) / d;
    }
}

/* Log-sum-exp of each row, ln sum_j e^(x_j) = m + ln d: the online
 * normalizer's state (m, d) of "Online normalizer calculation for softmax"
 * (notes), section 3, folded into one number ("6.2 FlashAttention V2" keeps it
 * per row).  Rows that are all -inf give -inf. */
void oracle_lse_f64(const double *x, double *lse, int64_t rows, int64_t cols) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double m, d;
        row_stats(x + r * cols, cols, &m, &d);
        lse[r] = m == -INFINITY ? -INFINITY : m + log(d);
    }
}

/* Causal mask: row r keeps columns c <= (r mod period) + offset, the query
 * position r mod period seeing keys up to its own position shifted by
 * `offset` ("6.2 FlashAttention V2", causal masking); the other entries
 * become -inf.  period >= 1. */
void oracle_causal_mask_f64(const double *x, double *out, int64_t rows, int64_t cols,
                            int64_t period, int64_t offset) {
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = c > (r % period) + offset ? -INFINITY : x[r * cols + c];
}

/* Top-K sampling from the K (value, index) pairs of each row (values >= 0),
 * by the inverse of the cumulative distribution of the renormalised values:
 * the smallest k with p_0 + ... + p_k > u (p_0 + ... + p_{K-1}), the partial
 * sums taken in index order in double; when no k qualifies (u >= 1) the last
 * one.  The drawn column idx[r*K + k] goes to out[r].  ("Online normalizer
 * calculation for softmax" (notes), section 4, names sampling from the top-K
 * probabilities as the consumer of the fused pass; the draw itself is this
 * plain definition.) */
void oracle_topk_sample_f64(const double *vals, const int32_t *idx, const double *u,
                            int32_t *out, int64_t rows, int32_t K) {
    for (int64_t r = 0; r < rows; ++r) {
        const double *p = vals + r * K;
        double total = 0.0;
        for (int32_t k = 0; k < K; ++k) total += p[k];
        const double target = u[r] * total;
        int32_t pick = K - 1;
        double run = 0.0;
        for (int32_t k = 0; k < K; ++k) {
            run += p[k];
            if (run > target) {
                pick = k;
                break;
            }
        }
        out[r] = idx[r * K + pick];
    }
}

/* The online normalizer recurrence, one element at a time, from (-inf, 0). */
void oracle_online_stats_f64(const double *x, int64_t n, double *m_out, double *d_out) {
    double m = -INFINITY, d = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double m_new = x[j] > m ? x[j] : m;
        if (m_new == -INFINITY) continue;          /* still the identity state */
        d = d * exp(m - m_new) + exp(x[j] - m_new);
        m = m_new;
    }
    *m_out = m;
    *d_out = d;
}

/* (m1,d1) (+) (m2,d2).  When both maxima are -inf both states are the
 * identity and so is the result; this avoids e^(-inf - (-inf)). */
void oracle_combine_f64(double m1, double d1, double m2, double d2,
                        double *m_out, double *d_out) {
    double m = m1 > m2 ? m1 : m2;
    if (m == -INFINITY) {
        *m_out = -INFINITY;
        *d_out = 0.0;
        return;
    }
    *m_out = m;
    *d_out = d1 * exp(m1 - m) + d2 * exp(m2 - m);
}

typedef struct {
    double x;
    int64_t j;
} keyed;

/* Order for the selection: larger logit first; equal logits, lower index first. */
static int by_logit_then_index(const void *pa, const void *pb) {
    const keyed *a = (const keyed *)pa, *b = (const keyed *)pb;
    if (a->x > b->x) return -1;
    if (a->x < b->x) return 1;
    return (a->j > b->j) - (a->j < b->j);
}

/* Top-K probabilities of each row, sorted by the order above.  Returns 0, or
 * -1 when K is outside [1, cols] or memory runs out. */
int oracle_topk_f64(const double *x, double *vals, int32_t *idx,
                    int64_t rows, int64_t cols, int32_t K) {
    if (K < 1 || (int64_t)K > cols) return -1;
    int failed = 0;
    #pragma omp parallel for schedule(static) reduction(|:failed)
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * cols;
        keyed *order = (keyed *)malloc((size_t)cols * sizeof(keyed));
        if (!order) {
            failed = 1;
            continue;
        }
        for (int64_t j = 0; j < cols; ++j) {
            order[j].x = xr[j];
            order[j].j = j;
        }
        qsort(order, (size_t)cols, sizeof(keyed), by_logit_then_index);
        double m, d;
        row_stats(xr, cols, &m, &d);
        for (int32_t k = 0; k < K; ++k) {
            vals[r * K + k] = exp(order[k].x - m) / d;
            idx[r * K + k] = (int32_t)order[k].j;
        }
        free(order);
    }
    return failed ? -1 : 0;
}

/* Attention forward by its definition, one query row at a time:
 *   s_j = scale * (q_i . k_j)          for the keys j the query sees,
 *   m   = max_j s_j,  d = sum_j e^(s_j - m),
 *   o_i = sum_j (e^(s_j - m) / d) v_j,  L_i = m + ln d.
 * Without the mask a query sees every key; with it, query i sees keys j <= i
 * (equal query and key lengths).  This is softmax(scale Q K^T) V of the
 * "Online normalizer calculation for softmax" notes, FlashAttention section
 * (the attention definition and the (m, d, o) recurrence that reaches it),
 * and the output O and logsumexp L of the "6.2 FlashAttention V2" forward
 * algorithm (section 6.1), whose tiled recurrence telescopes to the same
 * values in exact arithmetic; the definition is therefore the oracle.
 * Layout: q, k, v, o are [bh][n][dh] row-major, lse is [bh][n]. */
static void attend_row(const double *qi, const double *kb, const double *vb, int64_t i, int64_t n,
                       int64_t dh, double scale, int causal, double *s, double *oi,
                       double *lse_out) {
    const int64_t seen = causal ? i + 1 : n;
    double m = -INFINITY;  /* the maximum of the scores seen */
    for (int64_t j = 0; j < seen; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < dh; ++c) acc += qi[c] * kb[j * dh + c];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double d = 0.0;
    for (int64_t j = 0; j < seen; ++j) d += exp(s[j] - m);
    for (int64_t c = 0; c < dh; ++c) oi[c] = 0.0;
    for (int64_t j = 0; j < seen; ++j) {
        const double p = exp(s[j] - m) / d;
        for (int64_t c = 0; c < dh; ++c) oi[c] += p * vb[j * dh + c];
    }
    *lse_out = m + log(d);
}

void oracle_attention_f64(const double *q, const double *k, const double *v, double *o,
                          double *lse, int64_t bh, int64_t n, int64_t dh, double scale,
                          int causal) {
    #pragma omp parallel
    {
        double *s = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
        #pragma omp for schedule(static)
        for (int64_t r = 0; r < bh * n; ++r) {
            const int64_t b = r / n, i = r % n;
            attend_row(q + r * dh, k + b * n * dh, v + b * n * dh, i, n, dh, scale, causal, s,
                       o + r * dh, lse + r);
        }
        free(s);
    }
}

/* The same rows for a list of (slice, query) pairs only: row p of the output
 * is query row[p] of slice slice[p]; q holds just those query rows
 * ([npairs][dh]), k and v the full [bh][n][dh] tensors. */
void oracle_attention_rows_f64(const double *q, const double *k, const double *v,
                               const int64_t *slice, const int64_t *row, int64_t npairs,
                               int64_t n, int64_t dh, double scale, int causal, double *o,
                               double *lse) {
    #pragma omp parallel
    {
        double *s = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
        #pragma omp for schedule(dynamic)
        for (int64_t p = 0; p < npairs; ++p)
            attend_row(q + p * dh, k + slice[p] * n * dh, v + slice[p] * n * dh, row[p], n, dh,
                       scale, causal, s, o + p * dh, lse + p);
        free(s);
    }
}
